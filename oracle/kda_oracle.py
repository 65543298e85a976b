"""Plain fp64 CPU oracle for the KDA gated delta-rule serving step.

TEST INFRASTRUCTURE: only tests/, __graft_entry__.smoke() and bench.py's CPU
baseline leg use this module. It shares no code with the CUDA library.

What it computes, and where the pages state it
----------------------------------------------
Sources are two FlashInfer pull-request pages:

* "feat(kda): add packed-input CuTe decode kernel" (PR #4417), cited below as
  [decode]: the T=1 step on a bf16 state pool [N, 12, 128, 128] updated in
  place through state_indices; slots outside the pool give zero output and are
  left untouched (opening paragraph); the raw-gate convention
  (use_gate_in_kernel=True, lower_bound=-5, beta_is_logit=True, in-kernel q/k
  L2 norm, decay and sigmoid in fp32) and strided q/k/v/g views (section
  "T=1 fast path inside recurrent_kda"); the fused output o = (d*h).q + u*(k.q)
  (section "Kernel design").
* "feat(kda): ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)"
  (PR #4864), cited as [ring]: the T-token speculative verify that appends
  (k_hat, u, G) to a ring instead of writing the state back, replays with
  weights w_j = exp(G_P - G_j), and folds into the checkpoint once
  hist_len >= flush_min (sections "What it does", "API", "Caching").

Per (row, head), with S in R^{K x V} (math orientation):

    q_hat = q / sqrt(sum q^2 + eps),  k_hat likewise              (L2 norm)
    g_c   = lower_bound * sigmoid(exp(A_log[h]) * (g_raw_c + dt_bias[h, c]))
    d_c   = exp(g_c)                                   (per key channel)
    beta  = sigmoid(beta_logit)
    S     <- diag(d) S
    u     =  beta * (v - S^T k_hat)
    S     <- S + k_hat u^T
    o     =  scale * S^T q_hat

The state pool is stored [N][H][V][K] (one V row of K contiguous keys), so the
oracle transposes each slot to S = buf^T before applying the formulas above.

Rounding: all arithmetic is fp64. Values the method stores are rounded where
they are stored: the new state and the output to bf16 (round to nearest even,
directly from fp64), the ring's k_hat and u to bf16, and the ring's cumulative
log-decay G to fp32. The output is computed from the unrounded new state.
"""

import numpy as np

# Epsilon inside the L2 norm: x_hat = x / sqrt(sum x^2 + L2_EPS). The pages
# name an in-kernel q/k L2 norm without its epsilon; 1e-6 is the value this
# library documents for both sides.
L2_EPS = 1e-6

# Bit set in the ring call's error word when a slot's hist_len lies outside
# [0, W]. The slot is then treated as inactive.
RING_ERR_HIST_LEN = 1
RING_ERR_CACHE_BASE = 4

# bf16: 8 significant bits (7 stored), exponent range of fp32.
_BF16_SIG_BITS = 8
_BF16_MIN_QUANTUM_EXP = -133  # spacing of bf16 subnormals, 2^-126 * 2^-7
_BF16_OVERFLOW = 2.0 ** 128  # anything that rounds to this magnitude is inf


def round_to_bf16(x):
    """Round fp64 values to the nearest bf16 value (ties to even), as fp64.

    Done directly from fp64, never through fp32, so no double rounding. The
    quantum of a value in [2^(e-1), 2^e) is 2^(e-8); below the normal range
    it is the subnormal spacing 2^-133. Results of magnitude 2^128 or more
    overflow to +-inf. NaN, inf and signed zeros pass through.
    """
    x = np.asarray(x, dtype=np.float64)
    out = x.copy()
    mask = np.isfinite(x) & (x != 0.0)
    if np.any(mask):
        xs = x[mask]
        _, e = np.frexp(xs)  # xs = m * 2^e, 0.5 <= |m| < 1
        qexp = np.maximum(e - _BF16_SIG_BITS, _BF16_MIN_QUANTUM_EXP)
        # scaling by a power of two is exact; np.rint rounds half to even
        r = np.ldexp(np.rint(np.ldexp(xs, -qexp)), qexp)
        r = np.where(np.abs(r) >= _BF16_OVERFLOW, np.copysign(np.inf, xs), r)
        out[mask] = r
    return out


def round_to_fp32(x):
    """Round fp64 values to the nearest fp32 value (numpy's RNE cast), as fp64."""
    with np.errstate(over="ignore"):
        return np.asarray(x, dtype=np.float64).astype(np.float32).astype(np.float64)


def l2_normalize(x):
    """x / sqrt(sum(x^2) + L2_EPS) over the last axis ([decode] fast path:
    "in-kernel QK L2 norm")."""
    x = np.asarray(x, dtype=np.float64)
    return x / np.sqrt(np.sum(x * x, axis=-1, keepdims=True) + L2_EPS)


def _sigmoid(z):
    with np.errstate(over="ignore"):
        return 1.0 / (1.0 + np.exp(-z))


def gate_log_decay(g_raw, A_log, dt_bias, lower_bound):
    """Per-key-channel log-decay g = lower_bound * sigmoid(exp(A_log) * (g_raw + dt_bias)).

    [ring] API lists the inputs (A_log, g, dt_bias, lower_bound=-5.0); [decode]
    names the raw-gate convention use_gate_in_kernel=True with lower_bound=-5
    where the kernel computes the decay and sigmoid. g_raw: [..., H, K];
    A_log: [H]; dt_bias: [H, K]. Returns g in (lower_bound, 0].
    """
    g_raw = np.asarray(g_raw, dtype=np.float64)
    a = np.exp(np.asarray(A_log, dtype=np.float64))[:, None]
    z = a * (g_raw + np.asarray(dt_bias, dtype=np.float64))
    return lower_bound * _sigmoid(z)


def beta_from_logit(beta_logit):
    """beta = sigmoid(beta_logit) ([decode]: beta_is_logit=True)."""
    return _sigmoid(np.asarray(beta_logit, dtype=np.float64))


GATE_RAW = 0
GATE_PRECOMPUTED = 1


def prologue(q, k, g_raw, beta_logit, A_log, dt_bias, lower_bound, gate_mode=GATE_RAW):
    """The per-(row, head) quantities the state update needs.

    gate_mode GATE_RAW: g from the raw gate (gate_log_decay), beta =
    sigmoid(beta_logit). GATE_PRECOMPUTED ([decode] section "T=1 fast path
    inside recurrent_kda": the API-default form with log-space g and
    pre-sigmoided beta, decay exp(g)): g_raw already holds g and beta_logit
    holds beta; A_log, dt_bias and lower_bound are not used.
    Returns (q_hat, k_hat, g, d, beta) with d = exp(g).
    """
    q_hat = l2_normalize(q)
    k_hat = l2_normalize(k)
    if gate_mode == GATE_PRECOMPUTED:
        g = np.asarray(g_raw, dtype=np.float64)
        beta = np.asarray(beta_logit, dtype=np.float64)
    else:
        g = gate_log_decay(g_raw, A_log, dt_bias, lower_bound)
        beta = beta_from_logit(beta_logit)
    return q_hat, k_hat, g, np.exp(g), beta


def decode_step_math(S, q_hat, k_hat, v, d, beta, scale=1.0):
    """One gated delta-rule step on fp64 states in math orientation [..., K, V].

    Returns (S_new, o, u), none of them rounded:
        S1 = diag(d) S;  u = beta (v - S1^T k_hat);  S_new = S1 + k_hat u^T;
        o = scale * S_new^T q_hat.
    """
    S1 = d[..., :, None] * S
    u = beta[..., None] * (v - np.einsum("...kv,...k->...v", S1, k_hat))
    S_new = S1 + k_hat[..., :, None] * u[..., None, :]
    o = scale * np.einsum("...kv,...k->...v", S_new, q_hat)
    return S_new, o, u


def _active_mask(state_indices, N):
    idx = np.asarray(state_indices, dtype=np.int64)
    return idx, (idx >= 0) & (idx < N)


def kda_decode(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
               lower_bound=-5.0, scale=1.0, gate_mode=GATE_RAW):
    """T=1 decode ([decode] opening paragraph).

    state: [N, H, V, K] fp64 holding bf16 values (memory layout, K contiguous).
    state_indices: [B] ints; q, k, g_raw: [B, H, K]; v: [B, H, V];
    beta_logit: [B, H]; A_log: [H]; dt_bias: [H, K].

    Returns (new_state, out): new_state is a copy of state with every active
    slot replaced by the bf16-rounded updated state; out [B, H, V] is the
    bf16-rounded output, exactly 0 for rows whose index is outside [0, N).
    Duplicate active indices are undefined (the last row wins here).
    """
    state = np.asarray(state, dtype=np.float64)
    N = state.shape[0]
    B = np.asarray(q).shape[0]
    H, V = state.shape[1], state.shape[2]
    idx, active = _active_mask(state_indices, N)
    new_state = state.copy()
    out = np.zeros((B, H, V), dtype=np.float64)
    if not np.any(active):
        return new_state, out
    rows = np.nonzero(active)[0]
    slots = idx[rows]
    q_hat, k_hat, _, d, beta = prologue(
        np.asarray(q, np.float64)[rows], np.asarray(k, np.float64)[rows],
        np.asarray(g_raw, np.float64)[rows], np.asarray(beta_logit, np.float64)[rows],
        A_log, dt_bias, lower_bound, gate_mode)
    S = np.swapaxes(state[slots], -1, -2)  # [nA, H, K, V]
    S_new, o, _ = decode_step_math(S, q_hat, k_hat, np.asarray(v, np.float64)[rows],
                                   d, beta, scale)
    new_state[slots] = np.swapaxes(round_to_bf16(S_new), -1, -2)
    out[rows] = round_to_bf16(o)
    return new_state, out


def kda_verify(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
               lower_bound=-5.0, scale=1.0, gate_mode=GATE_RAW):
    """T-token speculative verify: T single decode steps on the same slots.

    q, k, g_raw: [B, T, H, K]; v: [B, T, H, V]; beta_logit: [B, T, H].
    The state is rounded to bf16 after every token, so this is literally T
    calls of kda_decode. Returns (new_state, out [B, T, H, V]).
    """
    q = np.asarray(q, np.float64)
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    V = np.asarray(state).shape[2]
    out = np.zeros((B, T, H, V), dtype=np.float64)
    for t in range(T):
        state, out[:, t] = kda_decode(state, state_indices, q[:, t], np.asarray(k)[:, t],
                                      np.asarray(v)[:, t], np.asarray(g_raw)[:, t],
                                      np.asarray(beta_logit)[:, t], A_log, dt_bias,
                                      lower_bound, scale, gate_mode)
    return state, out


def ring_replay(S0, k_hist, u_hist, G_hist):
    """Stepwise replay of a ring history onto a checkpoint ([ring] "Caching").

    S0: [..., K, V]; k_hist: [..., h, K]; u_hist: [..., h, V]; G_hist: [..., h, K]
    cumulative log-decay with G_{-1} = 0. Entry j applies
        S <- diag(exp(G_j - G_{j-1})) S + k_j u_j^T.
    """
    S = np.array(S0, dtype=np.float64)
    G_prev = np.zeros(S.shape[:-1], dtype=np.float64)
    for j in range(np.asarray(k_hist).shape[-2]):
        Gj = np.asarray(G_hist, np.float64)[..., j, :]
        S = np.exp(Gj - G_prev)[..., :, None] * S \
            + np.asarray(k_hist, np.float64)[..., j, :, None] * np.asarray(u_hist, np.float64)[..., j, None, :]
        G_prev = Gj
    return S


def ring_fold_closed_form(S0, k_hist, u_hist, G_hist):
    """The state a ring of h entries stands for, in closed form ([ring]
    "Caching": replay weights w_j = exp(G_P - G_j)):

        S_h = diag(exp(G_{h-1})) S0 + sum_j (exp(G_{h-1} - G_j) * k_j) u_j^T
    """
    S0 = np.asarray(S0, dtype=np.float64)
    h = np.asarray(k_hist).shape[-2]
    if h == 0:
        return S0.copy()
    G = np.asarray(G_hist, np.float64)
    Gl = G[..., h - 1, :]
    S = np.exp(Gl)[..., :, None] * S0
    wk = np.exp(Gl[..., None, :] - G) * np.asarray(k_hist, np.float64)  # [..., h, K]
    return S + np.einsum("...jk,...jv->...kv", wk, np.asarray(u_hist, np.float64))


def kda_verify_ring(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                    k_cache, u_cache, g_cache, hist_len, flush_min,
                    restart_hist_on_flush=True, lower_bound=-5.0, scale=1.0, gate_mode=GATE_RAW,
                    cache_base=None, fold_round=None):
    """Ring-cache verify with replay and fold ([ring] "What it does", "API", "Caching").

    state (checkpoint): [N, H, V, K]; k_cache: [N, H, W, K] bf16 k_hat;
    u_cache: [N, H, W, V] bf16 u; g_cache: [N, H, W, K] fp32 cumulative
    log-decay; hist_len: [N] live entries per slot; cache_base: [N] ring start
    per slot (None: 0). Token inputs as kda_verify.

    Ring position P of slot n is the stored entry (cache_base[n] + P) mod W: the
    ring page names a cache_base argument and says nothing more about it, and
    a per-slot start of a circular ring is the plainest reading. cache_base is
    read, never written.

    Per active row (slot n, history length h):
      * h outside [0, W]: the slot is inactive and RING_ERR_HIST_LEN is set;
        cache_base outside [0, W): likewise with RING_ERR_CACHE_BASE.
      * the current state is the checkpoint replayed through the h entries;
      * if h >= flush_min it is folded first: the checkpoint becomes its bf16
        rounding, the new tokens start at ring position 0 with G restarting
        from 0, and hist_len[n] is set to 0 when restart_hist_on_flush;
        otherwise the new tokens go to positions h .. h+T-1 and G continues
        from G_{h-1};
      * token t at position P: G_P = fp32(G_{P-1} + g_t), decay
        exp(G_P - G_{P-1}); k~ = bf16(k_hat_t); u = beta (v - (D S)^T k~);
        u~ = bf16(u); S <- D S + k~ u~^T; o_t = scale * S^T q_hat_t; (k~, u~,
        G_P) are written at position P.
    The kernel leaves hist_len alone unless it folds: the caller adds the
    number of accepted draft tokens afterwards.

    fold_round(n, S) -> S', for an fp8 checkpoint pool (kda_verify_ring_fp8):
    the checkpoint a fold of slot n makes of the replayed state S [H, K, V]
    in place of its bf16 rounding.

    Returns a dict with state, k_cache, u_cache, g_cache, hist_len, out
    [B, T, H, V] and error_word, plus the diagnostic state_fp64 [B, H, K, V]:
    the unrounded state each active row ends at (NaN for inactive rows), which
    replaying the written ring from the checkpoint reproduces.
    """
    state = np.asarray(state, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    u_cache = np.asarray(u_cache, dtype=np.float64)
    g_cache = np.asarray(g_cache, dtype=np.float64)
    hist_len = np.asarray(hist_len, dtype=np.int64)
    cache_base = (np.zeros(k_cache.shape[0], dtype=np.int64) if cache_base is None
                  else np.asarray(cache_base, dtype=np.int64))
    q = np.asarray(q, np.float64)
    k = np.asarray(k, np.float64)
    v = np.asarray(v, np.float64)
    g_raw = np.asarray(g_raw, np.float64)
    beta_logit = np.asarray(beta_logit, np.float64)
    N, H, W = k_cache.shape[0], k_cache.shape[1], k_cache.shape[2]
    B, T = q.shape[0], q.shape[1]
    V = state.shape[2]
    if not (1 <= T <= W):
        raise ValueError("need 1 <= T <= W")
    if flush_min < 1 or (flush_min - 1) + T > W:
        raise ValueError("need flush_min >= 1 and (flush_min - 1) + T <= W")

    new = dict(state=state.copy(), k_cache=k_cache.copy(), u_cache=u_cache.copy(),
               g_cache=g_cache.copy(), hist_len=hist_len.copy(),
               out=np.zeros((B, T, H, V), dtype=np.float64), error_word=0,
               state_fp64=np.full((B, H, state.shape[3], V), np.nan))
    idx, active = _active_mask(state_indices, N)
    for b in np.nonzero(active)[0]:
        n = idx[b]
        h = int(hist_len[n])
        if h < 0 or h > W:
            new["error_word"] |= RING_ERR_HIST_LEN
            continue
        cb = int(cache_base[n])
        if cb < 0 or cb >= W:
            new["error_word"] |= RING_ERR_CACHE_BASE
            continue
        live = [(cb + j) % W for j in range(h)]  # stored entries of positions 0 .. h-1
        q_hat, k_hat, g, _, beta = prologue(q[b], k[b], g_raw[b], beta_logit[b],
                                            A_log, dt_bias, lower_bound, gate_mode)
        S0 = np.swapaxes(state[n], -1, -2)  # [H, K, V]
        S = ring_replay(S0, k_cache[n][:, live], u_cache[n][:, live], g_cache[n][:, live])
        if h >= flush_min:
            S = round_to_bf16(S) if fold_round is None else fold_round(n, S)
            new["state"][n] = np.swapaxes(S, -1, -2)
            if restart_hist_on_flush:
                new["hist_len"][n] = 0
            base = 0
            G_prev = np.zeros((H, S.shape[-2]), dtype=np.float64)
        else:
            base = h
            G_prev = g_cache[n, :, live[-1]] if h > 0 else np.zeros((H, S.shape[-2]))
        for t in range(T):
            P = (cb + base + t) % W  # stored entry of ring position base + t
            G_P = round_to_fp32(G_prev + g[t])
            D = np.exp(G_P - G_prev)
            k_t = round_to_bf16(k_hat[t])
            S1 = D[:, :, None] * S
            u = beta[t][:, None] * (v[b, t] - np.einsum("hkv,hk->hv", S1, k_t))
            u_t = round_to_bf16(u)
            S = S1 + k_t[:, :, None] * u_t[:, None, :]
            new["out"][b, t] = round_to_bf16(scale * np.einsum("hkv,hk->hv", S, q_hat[t]))
            new["k_cache"][n, :, P] = k_t
            new["u_cache"][n, :, P] = u_t
            new["g_cache"][n, :, P] = G_P
            G_prev = G_P
        new["state_fp64"][b] = S
    return new
