"""Planted mistakes in the oracle must each fail at least one pin.

Each mutation is a one-place text edit of the oracle's source (a dropped term,
a wrong sign, axis or index, a skipped rounding). The edited source is loaded
as a separate module on the CPU and run through the whole pin suite.
"""

import inspect
import types

import pytest

import oracle
import oracle_pins

MUTATIONS = [
    ("cache_base ignored on writes", "P = (cb + base + t) % W", "P = (base + t) % W"),
    ("cache_base ignored on reads", "live = [(cb + j) % W for j in range(h)]", "live = [j for j in range(h)]"),
    ("cache_base subtracted", "live = [(cb + j) % W for j in range(h)]", "live = [(j - cb) % W for j in range(h)]"),
    ("cache_base not validated", "if cb < 0 or cb >= W:", "if cb < 0 or cb > W:"),
    ("l2 eps dropped", "keepdims=True) + L2_EPS)", "keepdims=True))"),
    ("l2 without sqrt", "return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)",
     "return x / (np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)"),
    ("gate without exp(A_log)", "a = np.exp(np.asarray(A_log, dtype=np.float64))[:, None]",
     "a = np.asarray(A_log, dtype=np.float64)[:, None]"),
    ("gate dt_bias sign", "(g_raw + np.asarray(dt_bias", "(g_raw - np.asarray(dt_bias"),
    ("gate sigmoid sign", "return lower_bound * _sigmoid(z)", "return lower_bound * _sigmoid(-z)"),
    ("decay is exp(-g)", "return q_hat, k_hat, g, np.exp(g),", "return q_hat, k_hat, g, np.exp(-g),"),
    ("beta not sigmoided", "return _sigmoid(np.asarray(beta_logit, dtype=np.float64))",
     "return np.asarray(beta_logit, dtype=np.float64)"),
    ("u from undecayed state", 'np.einsum("...kv,...k->...v", S1, k_hat))',
     'np.einsum("...kv,...k->...v", S, k_hat))'),
    ("u sign", "(v - np.einsum(\"...kv", "(v + np.einsum(\"...kv"),
    ("outer product transposed", "S_new = S1 + k_hat[..., :, None] * u[..., None, :]",
     "S_new = S1 + u[..., :, None] * k_hat[..., None, :]"),
    ("output from decayed old state", 'o = scale * np.einsum("...kv,...k->...v", S_new, q_hat)',
     'o = scale * np.einsum("...kv,...k->...v", S1, q_hat)'),
    ("output with k_hat", 'o = scale * np.einsum("...kv,...k->...v", S_new, q_hat)',
     'o = scale * np.einsum("...kv,...k->...v", S_new, k_hat)'),
    ("scale dropped", 'o = scale * np.einsum("...kv,...k->...v", S_new, q_hat)',
     'o = np.einsum("...kv,...k->...v", S_new, q_hat)'),
    ("decay on the value axis", "S1 = d[..., :, None] * S", "S1 = d[..., None, :] * S"),
    ("state not transposed", "S = np.swapaxes(state[slots], -1, -2)", "S = state[slots]"),
    ("index N active", "(idx >= 0) & (idx < N)", "(idx >= 0) & (idx <= N)"),
    ("index -1 active", "(idx >= 0) & (idx < N)", "(idx >= -1) & (idx < N)"),
    ("bf16 through fp32", "    x = np.asarray(x, dtype=np.float64)\n    out = x.copy()",
     "    x = np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)\n    out = x.copy()"),
    ("bf16 ties away", "np.rint(np.ldexp(xs, -qexp))", "np.floor(0.5 + np.ldexp(xs, -qexp))"),
    ("bf16 mantissa width", "_BF16_SIG_BITS = 8", "_BF16_SIG_BITS = 9"),
    ("replay without G difference", "S = np.exp(Gj - G_prev)[..., :, None] * S",
     "S = np.exp(Gj)[..., :, None] * S"),
    ("closed form weight sign", "np.exp(Gl[..., None, :] - G)", "np.exp(G - Gl[..., None, :])"),
    ("fold only above flush_min", "if h >= flush_min:", "if h > flush_min:"),
    ("G kept in fp64", "G_P = round_to_fp32(G_prev + g[t])", "G_P = G_prev + g[t]"),
    ("ring key not rounded", "k_t = round_to_bf16(k_hat[t])", "k_t = k_hat[t]"),
    ("ring u not rounded", "u_t = round_to_bf16(u)", "u_t = u"),
    ("ring position off by one", "P = (cb + base + t) % W", "P = (cb + base + t + 1) % W"),
    ("G restarts without fold", "G_prev = g_cache[n, :, live[-1]] if h > 0",
     "G_prev = 0.0 * g_cache[n, :, 0] if h > 0"),
    ("hist_len kept on fold", 'new["hist_len"][n] = 0', 'new["hist_len"][n] = h'),
    ("bad hist_len accepted", "if h < 0 or h > W:", "if h < 0 or h > W + 1:"),
    ("ring decay from g, not G", "D = np.exp(G_P - G_prev)", "D = np.exp(g[t])"),
    ("precomputed beta sigmoided again", "beta = np.asarray(beta_logit, dtype=np.float64)\n",
     "beta = beta_from_logit(beta_logit)\n"),
    ("precomputed g used as the decay", "g = np.asarray(g_raw, dtype=np.float64)\n",
     "g = np.log(np.asarray(g_raw, dtype=np.float64) + 6.0)\n"),
    ("ring u from undecayed state", '(v[b, t] - np.einsum("hkv,hk->hv", S1, k_t))',
     '(v[b, t] - np.einsum("hkv,hk->hv", S, k_t))'),
]


def _mutant(old, new):
    src = inspect.getsource(oracle.kda_oracle)
    assert src.count(old) == 1, f"mutation anchor must occur once: {old!r}"
    mod = types.ModuleType("kda_oracle_mutant")
    exec(compile(src.replace(old, new), "kda_oracle_mutant.py", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_mutant_is_caught(name, old, new):
    mod = _mutant(old, new)
    for pin in oracle_pins.ALL_PINS:
        try:
            pin(mod)
        except Exception:
            return
    pytest.fail(f"no pin caught the planted mistake: {name}")
