"""The varlen prefill oracle against its pins, and planted mistakes in it
against the same pins (each must fail at least one)."""

import inspect
import types

import pytest

import oracle.kda_prefill_oracle as pf
import oracle_pins_prefill


@pytest.mark.parametrize("pin", oracle_pins_prefill.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(pf)


MUTATIONS = [
    ("state rounded after every token",
     "            S, o, _ = decode_step_math(S, q_hat[t], k_hat[t], v[t0 + t], d[t], beta[t], scale)\n",
     "            S, o, _ = decode_step_math(S, q_hat[t], k_hat[t], v[t0 + t], d[t], beta[t], scale)\n"
     "            S = round_to_bf16(S)\n"),
    ("final state not rounded", "new_state[idx[i]] = np.swapaxes(round_to_bf16(S), -1, -2)",
     "new_state[idx[i]] = np.swapaxes(S, -1, -2)"),
    ("state not transposed", "S = np.swapaxes(state[idx[i]], -1, -2)  # [H, K, V], math orientation",
     "S = state[idx[i]]"),
    ("last token dropped", "for t in range(t1 - t0):", "for t in range(t1 - t0 - 1):"),
    ("q and k swapped", "prologue(q[t0:t1], k[t0:t1],", "prologue(k[t0:t1], q[t0:t1],"),
    ("values of the wrong row", "v[t0 + t], d[t]", "v[t0 + t - 1], d[t]"),
    ("bounds allow one row past the end", "if t0 < 0 or t1 < t0 or t1 > L:", "if t0 < 0 or t1 < t0 or t1 > L + 1:"),
    ("negative start allowed", "if t0 < 0 or t1 < t0 or t1 > L:", "if t1 < t0 or t1 > L:"),
    ("inactive rows not written", "        written[t0:t1] = True\n", "        written[t0:t1] = active[i]\n"),
    ("index N active", "idx, active = _active_mask(state_indices, N)",
     "idx, active = _active_mask(state_indices, N + 1)"),
    ("outputs off by 2^-6", "out[t0 + t] = round_to_bf16(o)", "out[t0 + t] = round_to_bf16(o * (1 + 2.0 ** -6))"),
]


def _mutant(old, new):
    src = inspect.getsource(pf)
    assert src.count(old) == 1, f"mutation anchor must occur once: {old!r}"
    src = src.replace("from .kda_oracle import", "from oracle.kda_oracle import")
    mod = types.ModuleType("kda_prefill_oracle_mutant")
    exec(compile(src.replace(old, new), "kda_prefill_oracle_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(name, old, new):
    mod = _mutant(old, new)
    for pin in oracle_pins_prefill.ALL_PINS:
        try:
            pin(mod)
        except Exception:
            return
    pytest.fail(f"no pin caught the planted mistake: {name}")
