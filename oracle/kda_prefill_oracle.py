"""Plain fp64 CPU oracle for the varlen KDA prefill.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg use this module. It shares no code with the CUDA library.

Source: "feat(kda): add CuTe DSL recurrent prefill backend" (FlashInfer PR
#4605): recurrent prefill over packed sequences given by cu_seqlens (offsets
that start at zero and never decrease), each sequence starting from a
caller-owned state in an indexed pool and leaving its final state there
(Description and review sections). The page prints no arithmetic of its own;
the step is the decode step of kda_oracle (the PR #4417 decode page), and this
oracle takes the plainest reading of a prefill:

    for each sequence, S = its bf16 slot (exact in fp64);
    for each of its tokens in order: S, o = one decode step in fp64, with no
        rounding of S between tokens; out row = bf16(o);
    the slot = bf16(S) once, after the last token.

Sequences with an index outside [0, N) write zero outputs and leave the pool
as it is; sequences whose bounds are out of order or outside [0, L) are
skipped and reported (PREFILL_ERR_SEQLENS); rows no sequence covers are not
written. Rounding to bf16 is direct from fp64 (round to nearest even).
"""

import numpy as np

from .kda_oracle import _active_mask, decode_step_math, prologue, round_to_bf16, GATE_RAW

# Bit reported for a sequence whose bounds are out of order or outside [0, L].
PREFILL_ERR_SEQLENS = 8


def kda_prefill(state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                lower_bound=-5.0, scale=1.0, gate_mode=GATE_RAW):
    """Varlen prefill.

    state: [N, H, V, K] fp64 holding bf16 values (memory layout); state_indices:
    [S]; cu_seqlens: [S + 1]; q, k, g_raw: [L, H, K]; v: [L, H, V];
    beta_logit: [L, H]; A_log: [H]; dt_bias: [H, K].

    Returns (new_state, out, written, err): out [L, H, V] (bf16 values; zero
    where nothing was written), written [L] bool (rows some valid sequence
    covers), err (PREFILL_ERR_SEQLENS or 0).
    """
    state = np.asarray(state, dtype=np.float64)
    q, k, v = (np.asarray(x, np.float64) for x in (q, k, v))
    g_raw, beta_logit = np.asarray(g_raw, np.float64), np.asarray(beta_logit, np.float64)
    N = state.shape[0]
    L, H = q.shape[0], q.shape[1]
    V = state.shape[2]
    cu = np.asarray(cu_seqlens, dtype=np.int64)
    idx, active = _active_mask(state_indices, N)
    new_state = state.copy()
    out = np.zeros((L, H, V), dtype=np.float64)
    written = np.zeros(L, dtype=bool)
    err = 0
    for i in range(len(idx)):
        t0, t1 = int(cu[i]), int(cu[i + 1])
        if t0 < 0 or t1 < t0 or t1 > L:
            err |= PREFILL_ERR_SEQLENS
            continue
        written[t0:t1] = True
        if t0 == t1 or not active[i]:
            continue  # out rows stay zero; the pool is untouched
        q_hat, k_hat, _, d, beta = prologue(q[t0:t1], k[t0:t1], g_raw[t0:t1], beta_logit[t0:t1],
                                            A_log, dt_bias, lower_bound, gate_mode)
        S = np.swapaxes(state[idx[i]], -1, -2)  # [H, K, V], math orientation
        for t in range(t1 - t0):
            S, o, _ = decode_step_math(S, q_hat[t], k_hat[t], v[t0 + t], d[t], beta[t], scale)
            out[t0 + t] = round_to_bf16(o)
        new_state[idx[i]] = np.swapaxes(round_to_bf16(S), -1, -2)
    return new_state, out, written, err
