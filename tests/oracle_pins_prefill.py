"""Pins for the varlen prefill oracle (oracle/kda_prefill_oracle.py).

Each ``pin_*`` takes the prefill oracle module and raises AssertionError when
it disagrees with something other than itself: a brute-force restatement of
the recurrence in scalar Python at K = V = 4, closed forms (decay only,
orthonormal writes), and the bookkeeping rules of the reading (inactive and
empty sequences, bad bounds). test_oracle_pins_prefill.py runs them against
the oracle and against copies with planted mistakes.

Source: "feat(kda): add CuTe DSL recurrent prefill backend" (PR #4605) for
packed sequences by cu_seqlens and the in-place indexed state; the step is the
one of "feat(kda): add packed-input CuTe decode kernel" (PR #4417).
"""

import math

import numpy as np

LB = -5.0
EPS = 1e-6


def bf16_values(rng, shape, std=1.0):
    """Random values that are exactly bf16 (fp32 with the low 16 bits cleared)."""
    x = (rng.standard_normal(shape) * std).astype(np.float32)
    return (x.view(np.uint32) & np.uint32(0xFFFF0000)).view(np.float32).astype(np.float64)


def is_bf16(x):
    """True where x is exactly a bf16 value (checked on the fp32 bit pattern)."""
    x = np.asarray(x, np.float64)
    f = x.astype(np.float32)
    return (f.astype(np.float64) == x) & ((f.view(np.uint32) & np.uint32(0xFFFF)) == 0)


def half_ulp(x):
    """Half a bf16 ulp at |x| (8 significant bits)."""
    m = np.maximum(np.abs(np.asarray(x, np.float64)), 2.0 ** -126)
    return np.ldexp(0.5, np.floor(np.log2(m)).astype(np.int64) - 7)


def problem(rng, lengths, H=2, K=4, V=4, N=6):
    L = int(sum(lengths))
    return dict(
        state=bf16_values(rng, (N, H, V, K), 0.3),
        q=bf16_values(rng, (L, H, K)), k=bf16_values(rng, (L, H, K)), v=bf16_values(rng, (L, H, V)),
        g_raw=bf16_values(rng, (L, H, K)), beta_logit=bf16_values(rng, (L, H)),
        A_log=np.log(rng.uniform(1.0, 16.0, H)).astype(np.float32).astype(np.float64),
        dt_bias=(rng.standard_normal((H, K)) * 0.5).astype(np.float32).astype(np.float64),
        cu=np.concatenate([[0], np.cumsum(lengths)]).astype(np.int64),
    )


def brute_sequence(S0_mem, q, k, v, g_in, b_in, A_log, dt_bias, gate_mode=0, scale=1.0):
    """The recurrence in scalar Python for one sequence, one head at a time.
    S0_mem [H, V, K] (memory layout); token inputs [T, H, ...]. Returns the
    unrounded outputs [T][H][V] and final state [H][V][K] (memory layout)."""
    H, V, K = S0_mem.shape
    T = len(q)
    outs = [[[0.0] * V for _ in range(H)] for _ in range(T)]
    final = []
    for h in range(H):
        S = [[float(S0_mem[h][vv][c]) for vv in range(V)] for c in range(K)]  # S[c][v]
        for t in range(T):
            qn = math.sqrt(sum(float(x) ** 2 for x in q[t][h]) + EPS)
            kn = math.sqrt(sum(float(x) ** 2 for x in k[t][h]) + EPS)
            qh = [float(x) / qn for x in q[t][h]]
            kh = [float(x) / kn for x in k[t][h]]
            if gate_mode == 0:
                a = math.exp(float(A_log[h]))
                g = [LB / (1.0 + math.exp(-a * (float(g_in[t][h][c]) + float(dt_bias[h][c])))) for c in range(K)]
                beta = 1.0 / (1.0 + math.exp(-float(b_in[t][h])))
            else:
                g = [float(g_in[t][h][c]) for c in range(K)]
                beta = float(b_in[t][h])
            for c in range(K):
                dc = math.exp(g[c])
                for vv in range(V):
                    S[c][vv] *= dc
            for vv in range(V):
                x = sum(S[c][vv] * kh[c] for c in range(K))
                u = beta * (float(v[t][h][vv]) - x)
                for c in range(K):
                    S[c][vv] += kh[c] * u
            for vv in range(V):
                outs[t][h][vv] = scale * sum(S[c][vv] * qh[c] for c in range(K))
        final.append([[S[c][vv] for c in range(K)] for vv in range(V)])
    return np.array(outs), np.array(final)


def _run(m, p, idx, cu=None, gate_mode=0, scale=1.0):
    return m.kda_prefill(p["state"], idx, p["cu"] if cu is None else cu, p["q"], p["k"], p["v"], p["g_raw"],
                         p["beta_logit"], p["A_log"], p["dt_bias"], lower_bound=LB, scale=scale,
                         gate_mode=gate_mode)


def _assert_rounds(got, exact, what):
    """got must be a bf16 value within half an ulp (plus fp64 noise) of exact."""
    got, exact = np.asarray(got, np.float64), np.asarray(exact, np.float64)
    assert np.all(is_bf16(got)), f"{what}: not all values are bf16"
    err = np.abs(got - exact) - half_ulp(exact) - 1e-12 * (1.0 + np.abs(exact))
    assert np.all(err <= 0.0), f"{what}: off the bf16 rounding of the exact value by {float(err.max()):.3g}"


# ---------------------------------------------------------------- pins

def pin_brute_force_sequences(m):
    """Three sequences (lengths 5, 1, 7) against the scalar recurrence, raw gate."""
    rng = np.random.default_rng(11)
    lengths = [5, 1, 7]
    p = problem(rng, lengths)
    idx = np.array([4, 0, 2])
    new, out, written, err = _run(m, p, idx)
    assert err == 0 and np.all(written)
    for i, n in enumerate(idx):
        t0, t1 = p["cu"][i], p["cu"][i + 1]
        o_ref, s_ref = brute_sequence(p["state"][n], p["q"][t0:t1], p["k"][t0:t1], p["v"][t0:t1],
                                      p["g_raw"][t0:t1], p["beta_logit"][t0:t1], p["A_log"], p["dt_bias"])
        _assert_rounds(out[t0:t1], o_ref, f"outputs of sequence {i}")
        _assert_rounds(new[n], s_ref, f"final state of sequence {i}")
    untouched = [s for s in range(p["state"].shape[0]) if s not in set(idx.tolist())]
    assert np.array_equal(new[untouched], p["state"][untouched])


def pin_brute_force_precomputed_gate_scaled(m):
    """The pre-computed gate convention (log-space g in [-5, 0), beta in [0, 1)) and an output scale."""
    rng = np.random.default_rng(12)
    p = problem(rng, [9])
    p["g_raw"] = -5.0 * rng.uniform(0.0, 1.0, p["g_raw"].shape)
    p["beta_logit"] = rng.uniform(0.0, 1.0, p["beta_logit"].shape)
    idx = np.array([3])
    new, out, _, _ = _run(m, p, idx, gate_mode=1, scale=0.75)
    o_ref, s_ref = brute_sequence(p["state"][3], p["q"], p["k"], p["v"], p["g_raw"], p["beta_logit"],
                                  p["A_log"], p["dt_bias"], gate_mode=1, scale=0.75)
    _assert_rounds(out, o_ref, "outputs")
    _assert_rounds(new[3], s_ref, "final state")


def pin_decay_only_closed_form(m):
    """beta = 0: no writes, S_T = diag(exp(sum_t g_t)) S_0 over the key channels,
    and o_t = S_t^T q_hat_t."""
    rng = np.random.default_rng(13)
    T, H, K, V = 6, 2, 4, 4
    p = problem(rng, [T], H=H, K=K, V=V)
    p["g_raw"] = -rng.uniform(0.0, 0.5, (T, H, K))
    p["beta_logit"] = np.zeros((T, H))
    new, out, _, _ = _run(m, p, np.array([1]), gate_mode=1)
    S0 = p["state"][1]  # [H, V, K]
    G = np.cumsum(p["g_raw"], axis=0)  # [T, H, K]
    qh = p["q"] / np.sqrt(np.sum(p["q"] ** 2, axis=-1, keepdims=True) + EPS)
    for t in range(T):
        St = S0 * np.exp(G[t])[:, None, :]  # decay along K (the last memory axis)
        _assert_rounds(out[t], np.sum(St * qh[t][:, None, :], axis=-1), f"output of token {t}")
    _assert_rounds(new[1], S0 * np.exp(G[-1])[:, None, :], "final state")


def pin_orthonormal_writes(m):
    """beta = 1, no decay, keys on distinct axes, zero initial state: each
    token writes its value onto its key axis exactly, so S_T = sum_t k_t v_t^T
    and a query along the first key reads v_0 back at every token."""
    K = V = 4
    T, H = 3, 1
    state = np.zeros((2, H, V, K))
    k = np.zeros((T, H, K))
    for t in range(T):
        k[t, 0, t] = 1024.0  # k_hat = e_t up to (1 + 1e-6 / 2^20)^(-1/2)
    q = np.zeros((T, H, K))
    q[:, 0, 0] = 3.0
    rng = np.random.default_rng(14)
    v = bf16_values(rng, (T, H, V))
    p = dict(state=state, q=q, k=k, v=v, g_raw=np.zeros((T, H, K)), beta_logit=np.ones((T, H)),
             A_log=np.zeros(H), dt_bias=np.zeros((H, K)), cu=np.array([0, T]))
    new, out, _, _ = _run(m, p, np.array([1]), gate_mode=1)
    for t in range(T):
        _assert_rounds(out[t, 0], v[0, 0], f"output of token {t}")
    S = np.zeros((V, K))
    for t in range(T):
        S[:, t] = v[t, 0]
    _assert_rounds(new[1, 0], S, "final state")
    assert np.array_equal(new[0], state[0])


def pin_varlen_bookkeeping(m):
    """Inactive sequences (index -1 and N) write zero rows and leave the pool;
    an empty sequence writes nothing; active ones match the brute force on
    their own rows."""
    rng = np.random.default_rng(15)
    lengths = [2, 3, 0, 4, 1]
    p = problem(rng, lengths, N=5)
    idx = np.array([3, -1, 1, 5, 0])  # 5 == N: inactive
    new, out, written, err = _run(m, p, idx)
    assert err == 0
    assert np.all(written)  # the empty sequence covers no row; every other row is covered
    cu = p["cu"]
    for i in (1, 3):
        assert np.all(out[cu[i]:cu[i + 1]] == 0.0), f"inactive sequence {i} must write zeros"
    for i in (0, 4):
        n = idx[i]
        t0, t1 = cu[i], cu[i + 1]
        o_ref, s_ref = brute_sequence(p["state"][n], p["q"][t0:t1], p["k"][t0:t1], p["v"][t0:t1],
                                      p["g_raw"][t0:t1], p["beta_logit"][t0:t1], p["A_log"], p["dt_bias"])
        _assert_rounds(out[t0:t1], o_ref, f"outputs of sequence {i}")
        _assert_rounds(new[n], s_ref, f"final state of sequence {i}")
    for n in (1, 2, 4):  # slot 1 belongs to the empty sequence; 2 and 4 to none
        assert np.array_equal(new[n], p["state"][n]), f"slot {n} must be untouched"


def pin_bad_bounds(m):
    """A sequence whose bounds are out of order or past the last row is
    skipped and reported; its rows are not written, the others are."""
    rng = np.random.default_rng(16)
    p = problem(rng, [3, 3], N=4)
    L = 6
    for cu in ([0, 3, 2], [0, 3, L + 1], [-1, 3, 6]):
        cu = np.array(cu)
        new, out, written, err = _run(m, p, np.array([0, 1]), cu=cu)
        assert err == 8, f"cu_seqlens {cu.tolist()} must be reported"
        bad = 1 if cu[0] >= 0 else 0
        good = 1 - bad
        lo, hi = cu[good], cu[good + 1]
        assert np.all(written[lo:hi]) and not np.any(written[[r for r in range(L) if not lo <= r < hi]])
        assert np.array_equal(new[bad], p["state"][bad]), "a skipped sequence leaves its slot"
        assert not np.array_equal(new[good], p["state"][good])


def pin_single_tokens_are_decode_steps(m):
    """Sequences of one token each are one decode step per slot: the result of
    the same step written out as vectors here (fp64, bf16-rounded outputs and
    state)."""
    rng = np.random.default_rng(17)
    p = problem(rng, [1, 1, 1], N=4)
    idx = np.array([2, 0, 3])
    new, out, _, _ = _run(m, p, idx)
    for i, n in enumerate(idx):
        S = p["state"][n].transpose(0, 2, 1)  # [H, K, V]
        qh = p["q"][i] / np.sqrt(np.sum(p["q"][i] ** 2, -1, keepdims=True) + EPS)
        kh = p["k"][i] / np.sqrt(np.sum(p["k"][i] ** 2, -1, keepdims=True) + EPS)
        g = LB / (1.0 + np.exp(-np.exp(p["A_log"])[:, None] * (p["g_raw"][i] + p["dt_bias"])))
        beta = 1.0 / (1.0 + np.exp(-p["beta_logit"][i]))
        S1 = np.exp(g)[:, :, None] * S
        u = beta[:, None] * (p["v"][i] - np.einsum("hkv,hk->hv", S1, kh))
        S2 = S1 + kh[:, :, None] * u[:, None, :]
        _assert_rounds(out[i], np.einsum("hkv,hk->hv", S2, qh), f"output of row {i}")
        _assert_rounds(new[n], S2.transpose(0, 2, 1), f"state of slot {n}")


ALL_PINS = [pin_brute_force_sequences, pin_brute_force_precomputed_gate_scaled, pin_decay_only_closed_form,
            pin_orthonormal_writes, pin_varlen_bookkeeping, pin_bad_bounds, pin_single_tokens_are_decode_steps]
