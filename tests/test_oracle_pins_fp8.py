"""The fp8 state-pool oracle against its pins, and planted mistakes in it
against the same pins (each must fail at least one)."""

import inspect
import types

import pytest

import oracle.kda_fp8_oracle as fp8
import oracle_pins_fp8


@pytest.mark.parametrize("pin", oracle_pins_fp8.ALL_PINS, ids=lambda f: f.__name__)
def test_pin(pin):
    pin(fp8)


MUTATIONS = [
    ("exponent bias 8", "_E4M3_BIAS = 7", "_E4M3_BIAS = 8"),
    ("subnormal quantum 2^-10", "_E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9", "_E4M3_SUBNORMAL_QUANTUM = 2.0 ** -10"),
    ("decode sign dropped", "val = np.where(s == 1, -mag, mag)", "val = mag"),
    ("encode ties away", "r = np.ldexp(np.rint(np.ldexp(ax, -qexp)), qexp)",
     "r = np.ldexp(np.floor(0.5 + np.ldexp(ax, -qexp)), qexp)"),
    ("encode truncates", "r = np.ldexp(np.rint(np.ldexp(ax, -qexp)), qexp)",
     "r = np.ldexp(np.floor(np.ldexp(ax, -qexp)), qexp)"),
    ("encode no saturation", "r = np.minimum(r, E4M3_MAX)", "r = np.minimum(r, 480.0)"),
    ("normal range from 2^-7", "_E4M3_MIN_NORMAL_EXP = -6", "_E4M3_MIN_NORMAL_EXP = -7"),
    ("row threshold 1.5", "e = np.where(M <= 1.75, E - 8, E - 7)", "e = np.where(M <= 1.5, E - 8, E - 7)"),
    ("row exponent one high", "e = np.where(M <= 1.75, E - 8, E - 7)", "e = np.where(M <= 1.75, E - 7, E - 6)"),
    ("scale applied the wrong way", "return e4m3_encode(np.ldexp(s, -e[..., None])), e",
     "return e4m3_encode(np.ldexp(s, e[..., None])), e"),
    ("row max over the wrong axis", "e = row_exponent(np.max(np.abs(s), axis=-1))",
     "e = row_exponent(np.max(np.abs(s), axis=-1) * 0.5)"),
    ("state not transposed", "S = np.swapaxes(dequantize(codes[slots], scales[slots]), -1, -2)",
     "S = dequantize(codes[slots], scales[slots])"),
    ("scales not applied", "return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]",
     "return e4m3_decode(codes)"),
    ("index N active", "idx, active = _active_mask(state_indices, N)",
     "idx, active = _active_mask(state_indices, N + 1)"),
    ("ring fold continues unrounded", "return np.swapaxes(dequantize(c, new_scales[n]), -1, -2)", "return S"),
    ("ring fold rounds to bf16", "return np.swapaxes(dequantize(c, new_scales[n]), -1, -2)",
     "return round_to_bf16(S)"),
    ("ring fold rows over the values", "rows = np.swapaxes(S, -1, -2)  # value rows over their keys",
     "rows = S"),
    ("ring fold skips fp32", "c, e = requantize_rows(round_to_fp32(rows))", "c, e = requantize_rows(rows)"),
]


def _mutant(old, new):
    src = inspect.getsource(fp8)
    assert src.count(old) == 1, f"mutation anchor must occur once: {old!r}"
    src = src.replace("from .kda_oracle import", "from oracle.kda_oracle import")
    mod = types.ModuleType("kda_fp8_oracle_mutant")
    exec(compile(src.replace(old, new), "kda_fp8_oracle_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(name, old, new):
    mod = _mutant(old, new)
    for pin in oracle_pins_fp8.ALL_PINS:
        try:
            pin(mod)
        except Exception:
            return
    pytest.fail(f"no pin caught the planted mistake: {name}")
