"""Pins for the fp8 (E4M3) state-pool oracle: checks against the format's
definition, exhaustive search, invariants of the step and the bf16 oracle.

Each ``pin_*`` function takes the fp8 oracle module and raises AssertionError
when it disagrees. The same functions run against the real module
(test_oracle_pins_fp8.py) and against copies with planted mistakes, which
must each fail at least one pin.

Source of the format: the OCP 8-bit floating point specification (E4M3:
bias 7, 3 mantissa bits, no infinities, S.1111.111 NaN, largest finite 448).
Source of the step: "feat(kda): add packed-input CuTe decode kernel"
(PR #4417), section "Nsight Compute" (a narrower state as the remaining
headroom); the format and the per-row power-of-two scale are this library's
reading.
"""

import numpy as np

import oracle
from oracle_pins import bf16_values

LB = -5.0


def _positive_table():
    """The 126 positive nonzero finite E4M3 values, from the format's fields
    (written out here, independently of the module)."""
    vals = []
    for code in range(1, 0x7F):
        E, M = code >> 3, code & 7
        vals.append((code, M * 2.0 ** -9 if E == 0 else 2.0 ** (E - 7) * (1 + M / 8)))
    return vals


def _brute_encode(x):
    """Nearest E4M3 code by exhaustive search, ties to the even code (even
    mantissa field), saturating at 448; sign kept."""
    table = [(0, 0.0)] + _positive_table()
    ax = min(abs(x), 448.0)
    best = min(table, key=lambda cv: (abs(cv[1] - ax), cv[0] & 1))
    return best[0] | (0x80 if np.signbit(x) else 0)


def random_pool(rng, N, H, V, K, exp_lo=-14, exp_hi=-8):
    """Codes drawn field by field (sign, exponent field 1..15, mantissa; never
    NaN) and power-of-two row scales."""
    s = rng.integers(0, 2, (N, H, V, K))
    E = np.clip(np.rint(rng.normal(11.0, 2.0, (N, H, V, K))), 1, 15).astype(np.int64)
    M = rng.integers(0, 8, (N, H, V, K))
    M = np.where(E == 15, np.minimum(M, 6), M)
    codes = ((s << 7) | (E << 3) | M).astype(np.uint8)
    scales = np.ldexp(1.0, rng.integers(exp_lo, exp_hi + 1, (N, H, V)))
    return codes, scales


def small_fp8_problem(rng, B=3, H=2, K=4, V=4, N=5):
    codes, scales = random_pool(rng, N, H, V, K)
    return dict(codes=codes, scales=scales, q=bf16_values(rng, (B, H, K)), k=bf16_values(rng, (B, H, K)),
                v=bf16_values(rng, (B, H, V)), g_raw=bf16_values(rng, (B, H, K)),
                beta_logit=bf16_values(rng, (B, H)), A_log=np.log(rng.uniform(1, 16, H)),
                dt_bias=rng.normal(0, 0.5, (H, K)), state_indices=np.array([2, -1, 4])[:B])


# ---------------------------------------------------------------- the format

def pin_e4m3_landmarks(m8):
    cases = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x30: 0.5, 0x38: 1.0,
             0x39: 1.125, 0x3F: 1.875, 0x40: 2.0, 0x78: 256.0, 0x7E: 448.0, 0xB8: -1.0, 0xFE: -448.0}
    got = m8.e4m3_decode(np.array(list(cases), dtype=np.uint8))
    assert np.array_equal(got, np.array(list(cases.values()))), got
    assert np.signbit(m8.e4m3_decode(np.array([0x80], np.uint8))[0])
    assert np.all(np.isnan(m8.e4m3_decode(np.array([0x7F, 0xFF], np.uint8))))


def pin_e4m3_full_table(m8):
    codes = np.arange(1, 0x7F, dtype=np.uint8)
    want = np.array([v for _, v in _positive_table()])
    assert np.array_equal(m8.e4m3_decode(codes), want)
    assert np.array_equal(m8.e4m3_decode(codes | 0x80), -want)
    assert np.all(np.diff(want) > 0)


def pin_e4m3_roundtrip(m8):
    codes = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], dtype=np.uint8)
    assert np.array_equal(m8.e4m3_encode(m8.e4m3_decode(codes)), codes)
    assert m8.e4m3_encode(np.array([np.nan]))[0] == 0x7F


def pin_e4m3_rne_brute_force(m8):
    rng = np.random.default_rng(7)
    xs = np.concatenate([rng.uniform(-500, 500, 400), rng.normal(0, 0.02, 300), rng.normal(0, 2.0 ** -7, 200),
                         np.array([460.0, 479.0, 480.0, 1e6, -1e6, np.inf, -np.inf, 0.0, -0.0])])
    xs = xs.astype(np.float32).astype(np.float64)
    got = m8.e4m3_encode(xs)
    want = np.array([_brute_encode(x) for x in xs], dtype=np.uint8)
    assert np.array_equal(got, want), np.nonzero(got != want)


def pin_e4m3_midpoints(m8):
    table = [(0, 0.0)] + _positive_table()
    for (ca, a), (cb, b) in zip(table[:-1], table[1:]):
        mid = (a + b) / 2
        even = ca if ca % 2 == 0 else cb
        assert m8.e4m3_encode(np.array([mid]))[0] == even, (a, b)
        assert m8.e4m3_encode(np.array([np.nextafter(mid, a)]))[0] == ca
        assert m8.e4m3_encode(np.array([np.nextafter(mid, b)]))[0] == cb


def pin_row_exponent(m8):
    rng = np.random.default_rng(8)
    m = np.concatenate([np.ldexp(rng.uniform(1, 2, 500), rng.integers(-120, 120, 500)),
                        np.array([448.0, 449.0, 224.0, 1.0, 1.75, 1.7500001, 2.0 ** -126])])
    m = m.astype(np.float32).astype(np.float64)
    e = m8.row_exponent(m)
    assert np.all(np.ldexp(m, -e) <= 448.0) and np.all(np.ldexp(m, -(e - 1)) > 448.0)
    assert list(m8.row_exponent(np.array([0.0, 448.0, 449.0, 224.0]))) == [0, 0, 1, -1]
    assert m8.row_exponent(np.array([2.0 ** -130]))[0] == -134


def pin_requantize_bounds(m8):
    rng = np.random.default_rng(9)
    s = (rng.normal(0, 0.02, (64, 128)) * np.ldexp(1.0, rng.integers(-20, 20, (64, 1)))).astype(np.float32)
    s = s.astype(np.float64)
    codes, e = m8.requantize_rows(s)
    deq = m8.e4m3_decode(codes) * np.ldexp(1.0, e)[:, None]
    # the largest element lands in (224, 448] * 2^e; every element within half a quantum
    top = np.max(np.abs(m8.e4m3_decode(codes)), axis=1)
    assert np.all(top >= 224.0) and np.all(top <= 448.0)
    ax = np.abs(s)
    qexp = np.maximum(np.floor(np.log2(np.maximum(ax, 1e-300))) - 3, e[:, None] - 9)
    assert np.all(np.abs(deq - s) <= np.ldexp(0.5, qexp.astype(np.int64)) * (1 + 1e-12))


# ---------------------------------------------------------------- the step

def pin_fp8_step_is_bf16_step_on_dequantized_state(m8):
    """The dequantized pool is exactly bf16, so the output and the unrounded new
    state equal the (separately pinned) bf16 oracle's on that state."""
    rng = np.random.default_rng(10)
    P = small_fp8_problem(rng, K=128, V=128, H=2, N=5)
    new_c, new_s, out, info = m8.kda_decode_fp8(P["codes"], P["scales"], P["state_indices"], P["q"], P["k"],
                                               P["v"], P["g_raw"], P["beta_logit"], P["A_log"], P["dt_bias"], LB)
    deq = m8.dequantize(P["codes"], P["scales"])
    assert np.array_equal(oracle.round_to_bf16(deq), deq)
    st, out_ref = oracle.kda_decode(deq, P["state_indices"], P["q"], P["k"], P["v"], P["g_raw"],
                                    P["beta_logit"], P["A_log"], P["dt_bias"], LB)
    assert np.array_equal(out, out_ref)
    assert np.array_equal(oracle.round_to_bf16(info["S_new"]), st[info["slots"]])


def pin_fp8_identity_keeps_tight_rows(m8):
    """Decay 1 and beta 0 leave the state as it was: rows whose largest code
    is in (224, 448] keep codes and scale; others keep their values."""
    rng = np.random.default_rng(11)
    N, H, V, K, B = 4, 2, 8, 16, 2
    codes, scales = random_pool(rng, N, H, V, K)
    codes[..., 0] = np.where(rng.integers(0, 2, (N, H, V)) == 1, 0x7E, 0x77)  # 448 or 240: tight rows
    idx = np.array([1, 3])
    zeros_k = np.zeros((B, H, K))
    new_c, new_s, out, _ = m8.kda_decode_fp8(codes, scales, idx, bf16_values(rng, (B, H, K)),
                                             bf16_values(rng, (B, H, K)), bf16_values(rng, (B, H, V)),
                                             zeros_k, np.zeros((B, H)), None, None, LB, 1.0, oracle.GATE_PRECOMPUTED)
    assert np.array_equal(new_c, codes) and np.array_equal(new_s, scales)
    # every element below 2.0 (exponent field <= 7), the largest 2.0: each row is
    # rescaled by 2^7 on the way back, exactly
    sgn = rng.integers(0, 2, (N, H, V, K))
    loose = ((sgn << 7) | (rng.integers(0, 8, (N, H, V, K)) << 3) | rng.integers(0, 8, (N, H, V, K)))
    loose = loose.astype(np.uint8)
    loose[..., 0] = 0x40
    new_c, new_s, _, _ = m8.kda_decode_fp8(loose, scales, idx, bf16_values(rng, (B, H, K)),
                                           bf16_values(rng, (B, H, K)), bf16_values(rng, (B, H, V)),
                                           zeros_k, np.zeros((B, H)), None, None, LB, 1.0, oracle.GATE_PRECOMPUTED)
    assert np.array_equal(m8.dequantize(new_c, new_s), m8.dequantize(loose, scales))
    assert not np.array_equal(new_s[idx], scales[idx])


def pin_fp8_inactive_slots(m8):
    rng = np.random.default_rng(12)
    P = small_fp8_problem(rng)
    idx = np.array([-1, 5, 7])
    new_c, new_s, out, _ = m8.kda_decode_fp8(P["codes"], P["scales"], idx, P["q"], P["k"], P["v"], P["g_raw"],
                                             P["beta_logit"], P["A_log"], P["dt_bias"], LB)
    assert np.array_equal(new_c, P["codes"]) and np.array_equal(new_s, P["scales"]) and not np.any(out)
    new_c, new_s, out, info = m8.kda_decode_fp8(P["codes"], P["scales"], P["state_indices"], P["q"], P["k"],
                                                P["v"], P["g_raw"], P["beta_logit"], P["A_log"], P["dt_bias"], LB)
    untouched = [n for n in range(P["codes"].shape[0]) if n not in set(info["slots"].tolist())]
    assert np.array_equal(new_c[untouched], P["codes"][untouched])
    assert not np.any(out[1])  # row 1 has index -1
    assert np.all(np.isin(np.log2(new_s), np.arange(-200, 200)))  # powers of two


# ---------------------------------------------------------------- the ring's checkpoint

def small_ring_fp8_problem(rng, hist, flush_min, T=3, W=8, H=2, K=8, V=8, N=5, zero_history=False):
    """A ring call on an fp8 pool: slot n's history length hist[n]; rows 0..B-1 on slots 1..B."""
    B = len(hist)
    codes, scales = random_pool(rng, N, H, V, K)
    kc = rng.normal(0, 1, (N, H, W, K))
    kc = oracle.round_to_bf16(kc / np.linalg.norm(kc, axis=-1, keepdims=True))
    uc = oracle.round_to_bf16(rng.normal(0, 0.5, (N, H, W, V)))
    gc = oracle.round_to_fp32(np.cumsum(-rng.uniform(0, 0.5, (N, H, W, K)), axis=2))
    if zero_history:
        uc[:] = 0.0
        gc[:] = 0.0
    hl = np.zeros(N, dtype=np.int64)
    hl[1:B + 1] = hist
    return dict(codes=codes, scales=scales, state_indices=np.arange(1, B + 1), q=bf16_values(rng, (B, T, H, K)),
                k=bf16_values(rng, (B, T, H, K)), v=bf16_values(rng, (B, T, H, V)),
                g_raw=bf16_values(rng, (B, T, H, K)), beta_logit=bf16_values(rng, (B, T, H)),
                A_log=np.log(rng.uniform(1, 16, H)), dt_bias=rng.normal(0, 0.5, (H, K)), k_cache=kc, u_cache=uc,
                g_cache=gc, hist_len=hl, flush_min=flush_min)


def _ring_fp8(m8, P, **kw):
    return m8.kda_verify_ring_fp8(P["codes"], P["scales"], P["state_indices"], P["q"], P["k"], P["v"], P["g_raw"],
                                  P["beta_logit"], P["A_log"], P["dt_bias"], P["k_cache"], P["u_cache"],
                                  P["g_cache"], P["hist_len"], P["flush_min"], lower_bound=LB, **kw)


def _ring_bf16(P, state, hist_len=None):
    return oracle.kda_verify_ring(state, P["state_indices"], P["q"], P["k"], P["v"], P["g_raw"], P["beta_logit"],
                                  P["A_log"], P["dt_bias"], P["k_cache"], P["u_cache"], P["g_cache"],
                                  P["hist_len"] if hist_len is None else hist_len, P["flush_min"], lower_bound=LB)


def pin_fp8_ring_without_fold_is_bf16_ring_on_dequantized_pool(m8):
    """No slot reaches flush_min: the (separately pinned) bf16 ring on the
    pool's exact values, codes and scales untouched."""
    rng = np.random.default_rng(13)
    P = small_ring_fp8_problem(rng, hist=[0, 3, 5], flush_min=6)
    got = _ring_fp8(m8, P)
    ref = _ring_bf16(P, m8.dequantize(P["codes"], P["scales"]))
    assert np.array_equal(got["codes"], P["codes"]) and np.array_equal(got["scales"], P["scales"])
    assert not got["folded"]
    for name in ("out", "k_cache", "u_cache", "g_cache", "hist_len"):
        assert np.array_equal(got[name], ref[name], equal_nan=True), name


def pin_fp8_ring_fold_requantizes_the_closed_form_state(m8):
    """A folding slot's codes and scales are the row requantization (fp32
    values, rows over the keys) of the closed-form replay of its history onto
    the dequantized checkpoint, and the tokens continue from their exact
    values: the same call as a bf16 ring call from that checkpoint with no
    history."""
    rng = np.random.default_rng(14)
    P = small_ring_fp8_problem(rng, hist=[6, 2, 7], flush_min=6)
    got = _ring_fp8(m8, P)
    deq = m8.dequantize(P["codes"], P["scales"])
    assert sorted(got["folded"]) == [1, 3]
    for n in (1, 3):
        h = int(P["hist_len"][n])
        S = oracle.ring_fold_closed_form(np.swapaxes(deq[n], -1, -2), P["k_cache"][n][:, :h],
                                         P["u_cache"][n][:, :h], P["g_cache"][n][:, :h])
        rows = np.swapaxes(S, -1, -2)  # [H, V, K]
        c, e = m8.requantize_rows(oracle.round_to_fp32(rows))
        assert np.array_equal(got["codes"][n], c) and np.array_equal(got["scales"][n], np.ldexp(1.0, e))
        top = np.max(np.abs(m8.e4m3_decode(got["codes"][n])), axis=-1)
        assert np.all(top > 224.0) and np.all(top <= 448.0)
    assert np.array_equal(got["codes"][2], P["codes"][2]), "a slot that does not fold keeps its checkpoint"
    hist0 = np.where(P["hist_len"] >= P["flush_min"], 0, P["hist_len"])
    ref = _ring_bf16(P, m8.dequantize(got["codes"], got["scales"]), hist_len=hist0)
    for name in ("out", "k_cache", "u_cache", "g_cache"):
        assert np.array_equal(got[name], ref[name], equal_nan=True), name
    assert list(got["hist_len"][1:4]) == [0, 2, 0]


def pin_fp8_ring_lossless_fold_changes_nothing(m8):
    """A history of zero updates with no decay folds to the checkpoint itself,
    which the pool holds exactly: the outputs are those of the same call
    without the fold, value for value."""
    rng = np.random.default_rng(15)
    P = small_ring_fp8_problem(rng, hist=[5, 7], flush_min=5, W=12, zero_history=True)
    a = _ring_fp8(m8, P)
    P_nofold = dict(P, flush_min=8)
    b = _ring_fp8(m8, P_nofold)
    assert sorted(a["folded"]) == [1, 2] and not b["folded"]
    assert np.array_equal(a["out"], b["out"])
    assert np.array_equal(m8.dequantize(a["codes"], a["scales"]), m8.dequantize(P["codes"], P["scales"]))


def pin_fp8_ring_fold_decides_in_fp32(m8):
    """The fold's requantization is decided on the fp32 value: a folded value
    2^-10 (1 + 2^-4 + 2^-34) is 2^-10 (1 + 2^-4) in fp32, the midpoint of two
    codes at the row's scale 2^-10 (its largest value 448 * 2^-10), which
    rounds to the even code 1.0; the fp64 value would round up to 1.125."""
    rng = np.random.default_rng(16)
    P = small_ring_fp8_problem(rng, hist=[2], flush_min=2, T=1, W=4, H=1, K=8, V=8, N=2)
    P["codes"][1] = 0
    P["codes"][1, :, :, 0] = 0x38  # 1.0
    P["codes"][1, :, :, 1] = 0x7E  # 448
    P["scales"][1] = 2.0 ** -10
    P["k_cache"][1] = 0.0
    P["k_cache"][1, :, :, 0] = 1.0  # both history keys are e_0
    P["u_cache"][1, :, 0] = 2.0 ** -14
    P["u_cache"][1, :, 1] = 2.0 ** -44
    P["g_cache"][1] = 0.0
    got = _ring_fp8(m8, P)
    assert np.all(got["scales"][1] == 2.0 ** -10)
    assert np.all(got["codes"][1, :, :, 0] == 0x38) and np.all(got["codes"][1, :, :, 1] == 0x7E)


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
