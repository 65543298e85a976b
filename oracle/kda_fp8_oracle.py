"""fp8 (E4M3) state pool for the T=1 decode and the ring verify's
checkpoint: the oracle of this library's numeric contract for it.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg use this module. It shares no code with the CUDA library.

Source and reading
------------------
"feat(kda): add packed-input CuTe decode kernel" (PR #4417), section "Nsight
Compute": at B=512 the bf16 decode runs at the observed machine ceiling for
its access pattern, so the remaining headroom is fewer bytes, for example an
fp8 state. The pages fix no format. This library's reading, which both sides
implement:

* Codes: the OCP 8-bit floating-point format E4M3 - 1 sign bit, 4 exponent
  bits (bias 7), 3 mantissa bits; exponent field 0 holds the subnormals
  M * 2^-9; S.1111.111 is NaN; no infinities; the largest finite magnitude is
  448 (S.1111.110).
* One scale per state row (slot, head, value index v): a power of two 2^e,
  stored as an fp32 value, so that the row's key k holds code_k * 2^e exactly.
* The step: the row's exact values go through the bf16 decode's arithmetic
  (decode_step_math, fp64 here); the output is taken from the unrounded new
  state and rounded to bf16, as in the bf16 decode.
* Requantization of every active row, decided in fp32 (the precision the
  kernel computes the new state in): s' = fp32(new state);
  m = max_k |s'_k|; e = the smallest integer with m * 2^-e <= 448 (e = 0 for
  an all-zero row; a row whose m is below 2^-126 takes e = -134); codes =
  E4M3 round-to-nearest-even of s' * 2^-e (saturating at 448, which the
  choice of e never reaches).
"""

import numpy as np

from .kda_oracle import (_active_mask, decode_step_math, kda_verify_ring, prologue, round_to_bf16, round_to_fp32,
                         GATE_RAW)

E4M3_MAX = 448.0
E4M3_NAN = 0x7F
_E4M3_BIAS = 7
_E4M3_MIN_NORMAL_EXP = -6  # 2^-6 = 0.0001.000
_E4M3_SUBNORMAL_QUANTUM = 2.0 ** -9
_TINY_ROW_EXP = -134  # e for rows whose max is below the fp32 normal range


def e4m3_decode(codes):
    """E4M3 codes (uint8) -> fp64 values by the format's definition.

    sign s = bit 7, exponent field E = bits 6..3, mantissa field M = bits 2..0:
    E = 0: (-1)^s * M * 2^-9; E = 15 and M = 7: NaN; else
    (-1)^s * 2^(E - 7) * (1 + M / 8).
    """
    c = np.asarray(codes, dtype=np.uint8).astype(np.int64)
    s = (c >> 7) & 1
    E = (c >> 3) & 15
    M = c & 7
    mag = np.where(E == 0, M * _E4M3_SUBNORMAL_QUANTUM, np.ldexp(1.0 + M / 8.0, E - _E4M3_BIAS))
    val = np.where(s == 1, -mag, mag)
    return np.where((E == 15) & (M == 7), np.nan, val)


def e4m3_encode(x):
    """fp64 values -> E4M3 codes, round to nearest with ties to even,
    saturating at +-448; NaN -> 0x7F. Signed zeros keep their sign.

    The quantum of a value in the binade [2^E, 2^(E+1)) is 2^(E-3) for
    E >= -6, and 2^-9 below (the subnormals): the value is an integer multiple
    of the quantum, whose parity is the parity of M, so rounding the multiple
    to the nearest even integer is the format's round-to-nearest-even.
    """
    x = np.asarray(x, dtype=np.float64)
    ax = np.abs(x)
    with np.errstate(divide="ignore", invalid="ignore"):
        _, fe = np.frexp(ax)  # ax = f * 2^fe, 0.5 <= f < 1
    E = fe - 1
    qexp = np.where(E >= _E4M3_MIN_NORMAL_EXP, E - 3, -9)
    r = np.ldexp(np.rint(np.ldexp(ax, -qexp)), qexp)
    r = np.minimum(r, E4M3_MAX)
    r = np.where(np.isnan(r), 0.0, r)  # NaN is coded below
    # r is now a representable magnitude: split it back into fields
    with np.errstate(divide="ignore", invalid="ignore"):
        _, re = np.frexp(r)
    rE = re - 1
    normal = rE >= _E4M3_MIN_NORMAL_EXP
    Ef = np.where(normal, rE + _E4M3_BIAS, 0)
    Mf = np.where(normal, np.rint(np.ldexp(r, -rE) * 8.0) - 8.0, np.rint(r / _E4M3_SUBNORMAL_QUANTUM))
    Mf = np.where(r == 0.0, 0.0, Mf)
    Ef = np.where(r == 0.0, 0, Ef)
    code = (Ef.astype(np.int64) << 3) | Mf.astype(np.int64)
    code = np.where(np.signbit(x), code | 0x80, code)
    code = np.where(np.isnan(x), E4M3_NAN, code)
    return code.astype(np.uint8)


def row_exponent(m):
    """The requantization exponent of rows whose largest magnitude is m (fp32
    values, >= 0): the smallest integer e with m * 2^-e <= 448.

    With m = M * 2^E, 1 <= M < 2, and 448 = 1.75 * 2^8: e = E - 8 when
    M <= 1.75, else E - 7. e = 0 for m = 0 and -134 for 0 < m < 2^-126.
    """
    m = np.asarray(m, dtype=np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        f, fe = np.frexp(m)  # m = f * 2^fe, 0.5 <= f < 1
    E = fe - 1
    M = 2.0 * f
    e = np.where(M <= 1.75, E - 8, E - 7)
    e = np.where(m < 2.0 ** -126, _TINY_ROW_EXP, e)
    return np.where(m == 0.0, 0, e).astype(np.int64)


def requantize_rows(s):
    """fp32-valued rows [..., K] -> (codes [..., K] uint8, e [...] int)."""
    s = np.asarray(s, dtype=np.float64)
    e = row_exponent(np.max(np.abs(s), axis=-1))
    return e4m3_encode(np.ldexp(s, -e[..., None])), e


def dequantize(codes, scales):
    """Row values code * scale, exactly (scales are powers of two)."""
    return e4m3_decode(codes) * np.asarray(scales, dtype=np.float64)[..., None]


def kda_decode_fp8(codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                   lower_bound=-5.0, scale=1.0, gate_mode=GATE_RAW):
    """T=1 decode on an fp8 state pool (the reading in the module docstring).

    codes: [N, H, V, K] uint8 (memory layout, K contiguous); scales: [N, H, V]
    powers of two. Other inputs as in kda_decode.

    Returns (new_codes, new_scales, out, info): copies of codes and scales
    with every active slot requantized, out [B, H, V] the bf16-rounded output
    (0 for rows whose index is outside [0, N)), and info = {"rows": active
    batch rows, "slots": their slots, "S_new": the unrounded new state [nA, H,
    V, K] in fp64, "S_new_fp32": the same rounded to fp32}.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.float64)
    N, H, V, _ = codes.shape
    B = np.asarray(q).shape[0]
    idx, active = _active_mask(state_indices, N)
    new_codes, new_scales = codes.copy(), scales.copy()
    out = np.zeros((B, H, V), dtype=np.float64)
    info = {"rows": np.zeros(0, np.int64), "slots": np.zeros(0, np.int64)}
    if not np.any(active):
        return new_codes, new_scales, out, info
    rows = np.nonzero(active)[0]
    slots = idx[rows]
    q_hat, k_hat, _, d, beta = prologue(
        np.asarray(q, np.float64)[rows], np.asarray(k, np.float64)[rows],
        np.asarray(g_raw, np.float64)[rows], np.asarray(beta_logit, np.float64)[rows],
        A_log, dt_bias, lower_bound, gate_mode)
    S = np.swapaxes(dequantize(codes[slots], scales[slots]), -1, -2)  # [nA, H, K, V]
    S_new, o, _ = decode_step_math(S, q_hat, k_hat, np.asarray(v, np.float64)[rows], d, beta, scale)
    rows_new = np.swapaxes(S_new, -1, -2)  # [nA, H, V, K]
    s32 = round_to_fp32(rows_new)
    c, e = requantize_rows(s32)
    new_codes[slots] = c
    new_scales[slots] = np.ldexp(1.0, e)
    out[rows] = round_to_bf16(o)
    info = {"rows": rows, "slots": slots, "S_new": rows_new, "S_new_fp32": s32}
    return new_codes, new_scales, out, info


def kda_verify_ring_fp8(codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                        k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush=True,
                        lower_bound=-5.0, scale=1.0, gate_mode=GATE_RAW, cache_base=None):
    """Ring-cache verify on an fp8 checkpoint pool: kda_verify_ring ("feat(kda):
    ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)", sections "What it
    does" and "Caching") with the pool of this module's reading as its
    checkpoint.

    The checkpoint is the pool's exact values. A fold requantizes the replayed
    state (unrounded) row by row as kda_decode_fp8 requantizes a new state -
    fp32 first, then each value row over its keys - writes codes and scales,
    and the new tokens continue from their exact values. The ring entries stay
    as kda_verify_ring writes them (bf16 k~ and u~, fp32 G).

    Returns kda_verify_ring's dict with "codes" and "scales" in place of
    "state", and "folded": {slot: the unrounded folded state [H, V, K]}.
    """
    codes = np.asarray(codes, dtype=np.uint8)
    scales = np.asarray(scales, dtype=np.float64)
    new_codes, new_scales = codes.copy(), scales.copy()
    folded = {}

    def requantize_fold(n, S):  # S: [H, K, V]
        rows = np.swapaxes(S, -1, -2)  # value rows over their keys
        c, e = requantize_rows(round_to_fp32(rows))
        new_codes[n], new_scales[n] = c, np.ldexp(1.0, e)
        folded[int(n)] = rows
        return np.swapaxes(dequantize(c, new_scales[n]), -1, -2)

    res = kda_verify_ring(dequantize(codes, scales), state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                          k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush, lower_bound, scale,
                          gate_mode, cache_base, fold_round=requantize_fold)
    del res["state"]
    res.update(codes=new_codes, scales=new_scales, folded=folded)
    return res
