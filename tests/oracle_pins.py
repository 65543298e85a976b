"""Pins for the CPU oracle: checks against things other than the oracle itself.

Each ``pin_*`` function takes the oracle module and raises AssertionError when
the oracle disagrees with a closed form, an invariant of the method, a
library rounding routine or a brute-force computation at K=V=4. The same
functions run against the real oracle (test_oracle_pins.py) and against
copies with planted mistakes (test_oracle_mutants.py), which must each fail
at least one pin.

Sources: "feat(kda): add packed-input CuTe decode kernel" (PR #4417) for the
T=1 step, the raw-gate convention and the inactive-slot rule;
"feat(kda): ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)"
(PR #4864) for the ring cache, replay weights exp(G_P - G_j) and the fold.
"""

import math
from fractions import Fraction

import numpy as np
import torch

LB = -5.0


# ---------------------------------------------------------------- helpers

def bf16_values(rng, shape, std=1.0):
    """Random values that are exactly bf16 (fp32 with the low 16 bits cleared)."""
    x = (rng.standard_normal(shape) * std).astype(np.float32)
    bits = x.view(np.uint32) & np.uint32(0xFFFF0000)
    return bits.view(np.float32).astype(np.float64)


def small_problem(rng, B=3, H=2, K=4, V=4, N=5, T=None):
    tok = () if T is None else (T,)
    return dict(
        state=bf16_values(rng, (N, H, V, K), 0.3),
        q=bf16_values(rng, (B,) + tok + (H, K)),
        k=bf16_values(rng, (B,) + tok + (H, K)),
        v=bf16_values(rng, (B,) + tok + (H, V)),
        g_raw=bf16_values(rng, (B,) + tok + (H, K)),
        beta_logit=bf16_values(rng, (B,) + tok + (H,)),
        A_log=np.log(rng.uniform(1.0, 16.0, H)).astype(np.float32).astype(np.float64),
        dt_bias=(rng.standard_normal((H, K)) * 0.5).astype(np.float32).astype(np.float64),
    )


def _decode(m, p, idx, **kw):
    return m.kda_decode(p["state"], idx, p["q"], p["k"], p["v"], p["g_raw"], p["beta_logit"],
                        p["A_log"], p["dt_bias"], lower_bound=LB, **kw)


def _unrounded_step(m, S_mem, q, k, v, g_raw, beta_logit, A_log, dt_bias, scale=1.0):
    """Oracle's unrounded step for one row (all heads); S_mem [H, V, K]."""
    q_hat, k_hat, g, d, beta = m.prologue(q, k, g_raw, beta_logit, A_log, dt_bias, LB)
    S = np.swapaxes(S_mem, -1, -2)
    S_new, o, u = m.decode_step_math(S, q_hat, k_hat, v, d, beta, scale)
    return dict(S=S, S_new=S_new, o=o, u=u, q_hat=q_hat, k_hat=k_hat, d=d, beta=beta, g=g)


def brute_step(S_mem, q, k, v, g_raw, beta_logit, A_log_h, dt_bias_h, lb=LB, scale=1.0):
    """Pure-Python step for one (row, head) with explicit index loops.

    S_mem[v][k] is the stored state (one V row of K keys), so the math state
    is S[k][v] = S_mem[v][k]. Returns (S_new[k][v], o[v]).
    """
    K, V = len(q), len(v)
    nq = math.sqrt(sum(x * x for x in q) + 1e-6)
    nk = math.sqrt(sum(x * x for x in k) + 1e-6)
    qh = [x / nq for x in q]
    kh = [x / nk for x in k]
    a = math.exp(A_log_h)
    d = []
    for c in range(K):
        z = a * (g_raw[c] + dt_bias_h[c])
        sig = 1.0 / (1.0 + math.exp(-z)) if z > -700 else 0.0
        d.append(math.exp(lb * sig))
    beta = 1.0 / (1.0 + math.exp(-beta_logit))
    S = [[S_mem[vv][kk] * d[kk] for vv in range(V)] for kk in range(K)]
    u = []
    for vv in range(V):
        acc = 0.0
        for kk in range(K):
            acc += S[kk][vv] * kh[kk]
        u.append(beta * (v[vv] - acc))
    S_new = [[S[kk][vv] + kh[kk] * u[vv] for vv in range(V)] for kk in range(K)]
    o = []
    for vv in range(V):
        acc = 0.0
        for kk in range(K):
            acc += S_new[kk][vv] * qh[kk]
        o.append(scale * acc)
    return S_new, o


def torch_bf16(x):
    """Library reference: torch's fp32 -> bf16 round-to-nearest-even."""
    return torch.from_numpy(np.asarray(x, np.float32)).to(torch.bfloat16).double().numpy()


# ---------------------------------------------------------------- rounding

def pin_bf16_matches_torch_on_fp32_values(m):
    rng = np.random.default_rng(1)
    x = np.concatenate([
        rng.standard_normal(20000).astype(np.float32),
        (rng.standard_normal(5000) * 1e-30).astype(np.float32),
        (rng.standard_normal(5000) * 1e-39).astype(np.float32),  # fp32 subnormals
        (rng.standard_normal(5000) * 1e37).astype(np.float32),
        np.array([3.3895e38, 3.39e38, -3.3999e38, 1.0, -2.0, 0.0], np.float32),
    ])
    got = m.round_to_bf16(x.astype(np.float64))
    ref = torch_bf16(x)
    same = (got == ref) | (np.isnan(got) & np.isnan(ref))
    assert same.all(), f"{(~same).sum()} mismatches vs torch, first at {x[~same][:4]}"


def pin_bf16_direct_rounding_and_ties(m):
    r = m.round_to_bf16
    # direct fp64 -> bf16: just above the 1 + 2^-8 tie rounds up (through fp32 it would tie to 1)
    assert r(np.array([1.0 + 2.0 ** -8 + 2.0 ** -40]))[0] == 1.0 + 2.0 ** -7
    assert r(np.array([1.0 + 2.0 ** -8]))[0] == 1.0  # tie to even (down)
    assert r(np.array([1.0 + 3 * 2.0 ** -8]))[0] == 1.0 + 2.0 ** -6  # tie to even (up)
    assert r(np.array([-(1.0 + 3 * 2.0 ** -8)]))[0] == -(1.0 + 2.0 ** -6)
    assert r(np.array([1.5 * 2.0 ** -133]))[0] == 2.0 ** -132  # subnormal tie, up to even
    assert r(np.array([2.0 ** -134]))[0] == 0.0  # subnormal tie, down to even zero
    assert r(np.array([2.0 ** -134 + 2.0 ** -160]))[0] == 2.0 ** -133
    big = (2.0 - 2.0 ** -8) * 2.0 ** 127  # midpoint between bf16 max and 2^128
    assert np.isinf(r(np.array([big]))[0])
    assert r(np.array([big * (1 - 2.0 ** -30)]))[0] == (2.0 - 2.0 ** -7) * 2.0 ** 127
    sp = r(np.array([np.nan, np.inf, -np.inf, 0.0, -0.0]))
    assert np.isnan(sp[0]) and sp[1] == np.inf and sp[2] == -np.inf
    assert sp[3] == 0.0 and not np.signbit(sp[3]) and np.signbit(sp[4])


def pin_fp32_rounding_matches_torch(m):
    rng = np.random.default_rng(2)
    x = rng.standard_normal(10000) * np.exp(rng.uniform(-60, 60, 10000))
    ref = torch.from_numpy(x).float().double().numpy()
    assert (m.round_to_fp32(x) == ref).all()


# ---------------------------------------------------------------- prologue

def pin_gate_closed_forms(m):
    A0 = np.array([0.0])  # exp(A_log) = 1
    dt0 = np.zeros((1, 3))
    # sigmoid(log 3) = 3/4 -> g = -3.75 ; sigmoid(0) = 1/2 -> g = -2.5
    g = m.gate_log_decay(np.array([[math.log(3.0), 0.0, -math.log(3.0)]]), A0, dt0, LB)
    assert np.allclose(g, [[-3.75, -2.5, -1.25]], rtol=0, atol=1e-14), g
    # g_raw = -dt_bias gives exactly lower_bound * 1/2 for any A_log
    rng = np.random.default_rng(3)
    dtb = rng.standard_normal((2, 8))
    g = m.gate_log_decay(-dtb, np.array([0.7, 2.3]), dtb, LB)
    assert (g == -2.5).all()
    # exp(A_log) scales the pre-activation: A_log = log 2 on x equals A_log = 0 on 2x
    x = rng.standard_normal((1, 8))
    g1 = m.gate_log_decay(x, np.array([math.log(2.0)]), np.zeros((1, 8)), LB)
    g2 = m.gate_log_decay(2 * x, np.array([0.0]), np.zeros((1, 8)), LB)
    assert np.allclose(g1, g2, rtol=1e-14, atol=1e-15)
    # dt_bias is added per (head, channel) before the scale
    dtb = rng.standard_normal((1, 8))
    g3 = m.gate_log_decay(x - dtb, np.array([math.log(2.0)]), dtb, LB)
    assert np.allclose(g1, g3, rtol=1e-12, atol=1e-13)
    # sigmoid(z) + sigmoid(-z) = 1 -> g(z) + g(-z) = lower_bound; monotone decreasing in g_raw
    z = np.linspace(-8, 8, 33)[None, :]
    gp = m.gate_log_decay(z, np.array([0.0]), np.zeros((1, 33)), LB)
    gm = m.gate_log_decay(-z, np.array([0.0]), np.zeros((1, 33)), LB)
    assert np.allclose(gp + gm, LB, atol=1e-13)
    assert (np.diff(gp[0]) < 0).all() and (gp > LB).all() and (gp < 0).all()
    # limits: g_raw -> -inf gives g = 0 (decay 1); +inf gives lower_bound
    lim = m.gate_log_decay(np.array([[-np.inf, np.inf]]), np.array([0.5]), np.zeros((1, 2)), LB)
    assert lim[0, 0] == 0.0 and lim[0, 1] == LB


def pin_beta_closed_forms(m):
    b = m.beta_from_logit(np.array([0.0, math.log(3.0), -math.log(3.0), -np.inf, np.inf]))
    assert np.allclose(b[:3], [0.5, 0.75, 0.25], rtol=0, atol=1e-15)
    assert b[3] == 0.0 and b[4] == 1.0


def pin_l2_norm(m):
    x = m.l2_normalize(np.array([[3.0, 4.0], [0.0, 0.0]]))
    assert np.allclose(x[0], np.array([3.0, 4.0]) / math.sqrt(25.0 + 1e-6), rtol=1e-15, atol=0)
    assert (x[1] == 0).all()
    rng = np.random.default_rng(4)
    y = rng.standard_normal((5, 128))
    n = np.linalg.norm(m.l2_normalize(y), axis=-1)
    assert np.allclose(n, 1.0, rtol=0, atol=1e-8)
    assert np.allclose(m.l2_normalize(3.0 * y), m.l2_normalize(y), rtol=1e-8, atol=0)


# ---------------------------------------------------------------- decode step

def pin_identity_step(m):
    """beta = 0 and g = 0 (decay 1) leave the state bitwise unchanged; o = S^T q_hat."""
    rng = np.random.default_rng(5)
    p = small_problem(rng, B=3, H=2, K=8, V=8, N=5)
    p["beta_logit"][:] = -np.inf
    p["g_raw"][:] = -np.inf
    idx = np.array([4, 0, 2])
    new, out = _decode(m, p, idx)
    assert np.array_equal(new, p["state"])
    q_hat = m.l2_normalize(p["q"])
    ref = np.einsum("bhvk,bhk->bhv", p["state"][idx], q_hat)
    assert np.array_equal(out, m.round_to_bf16(ref))


def pin_delta_rule_exactness(m):
    """decay 1, beta 1: the updated state maps k_hat exactly onto v."""
    rng = np.random.default_rng(6)
    p = small_problem(rng, B=1, H=3, K=16, V=12, N=1)
    r = _unrounded_step(m, p["state"][0], p["q"][0], p["k"][0], p["v"][0],
                        np.full((3, 16), -np.inf), np.full(3, np.inf), p["A_log"], p["dt_bias"])
    back = np.einsum("hkv,hk->hv", r["S_new"], r["k_hat"])
    nk2 = np.sum(r["k_hat"] ** 2, axis=-1, keepdims=True)  # 1 - O(1e-8) because of eps
    # S_new^T k = S^T k + k.k (v - S^T k) = v exactly when |k| = 1
    expect = p["v"][0] * nk2 + np.einsum("hkv,hk->hv", r["S"], r["k_hat"]) * (1 - nk2)
    assert np.allclose(back, expect, rtol=1e-12, atol=1e-12)
    assert np.allclose(back, p["v"][0], rtol=0, atol=1e-6)


def pin_zero_state_closed_form(m):
    """S = 0: S_new = beta k_hat v^T and o = scale beta v (k_hat . q_hat); q = k gives beta v."""
    rng = np.random.default_rng(7)
    p = small_problem(rng, B=2, H=2, K=8, V=6, N=3)
    p["state"][:] = 0.0
    p["q"][1] = p["k"][1]
    idx = np.array([0, 2])
    r = _unrounded_step(m, p["state"][0], p["q"][0], p["k"][0], p["v"][0],
                        p["g_raw"][0], p["beta_logit"][0], p["A_log"], p["dt_bias"], scale=0.5)
    outer = r["beta"][:, None, None] * r["k_hat"][:, :, None] * p["v"][0][:, None, :]
    assert np.allclose(r["S_new"], outer, rtol=1e-14, atol=1e-16)
    kq = np.sum(r["k_hat"] * r["q_hat"], axis=-1)
    assert np.allclose(r["o"], 0.5 * r["beta"][:, None] * p["v"][0] * kq[:, None], rtol=1e-13, atol=1e-15)
    new, out = _decode(m, p, idx)
    beta1 = m.beta_from_logit(p["beta_logit"][1])
    assert np.allclose(out[1], beta1[:, None] * p["v"][1], rtol=2 ** -8, atol=1e-7)


def pin_householder_form(m):
    """S_new = (I - beta k k^T) D S + beta k v^T, an independent arrangement of the update."""
    rng = np.random.default_rng(8)
    p = small_problem(rng, B=1, H=2, K=8, V=5, N=1)
    r = _unrounded_step(m, p["state"][0], p["q"][0], p["k"][0], p["v"][0],
                        p["g_raw"][0], p["beta_logit"][0], p["A_log"], p["dt_bias"])
    for h in range(2):
        kk = r["k_hat"][h]
        P = np.eye(8) - r["beta"][h] * np.outer(kk, kk)
        ref = P @ (np.diag(r["d"][h]) @ r["S"][h]) + r["beta"][h] * np.outer(kk, p["v"][0][h])
        assert np.allclose(r["S_new"][h], ref, rtol=1e-12, atol=1e-14)


def pin_fused_output(m):
    """o = (D S)^T q_hat + u (k_hat . q_hat) equals S_new^T q_hat ("Kernel design")."""
    rng = np.random.default_rng(9)
    p = small_problem(rng, B=1, H=2, K=16, V=16, N=1)
    r = _unrounded_step(m, p["state"][0], p["q"][0], p["k"][0], p["v"][0],
                        p["g_raw"][0], p["beta_logit"][0], p["A_log"], p["dt_bias"], scale=1.0)
    DS = r["d"][:, :, None] * r["S"]
    kq = np.sum(r["k_hat"] * r["q_hat"], axis=-1)
    fused = np.einsum("hkv,hk->hv", DS, r["q_hat"]) + r["u"] * kq[:, None]
    assert np.allclose(r["o"], fused, rtol=1e-12, atol=1e-14)


def pin_brute_force_k4(m):
    """Full step (prologue + update + output + rounding) at K = V = 4 against explicit loops."""
    rng = np.random.default_rng(10)
    p = small_problem(rng, B=3, H=2, K=4, V=4, N=4)
    idx = np.array([3, 1, 0])
    new, out = _decode(m, p, idx, scale=0.75)
    for b in range(3):
        for h in range(2):
            S_new, o = brute_step(p["state"][idx[b], h].tolist(), p["q"][b, h].tolist(),
                                  p["k"][b, h].tolist(), p["v"][b, h].tolist(),
                                  p["g_raw"][b, h].tolist(), float(p["beta_logit"][b, h]),
                                  float(p["A_log"][h]), p["dt_bias"][h].tolist(), scale=0.75)
            S_mem = np.array(S_new).T  # back to [V][K]
            # the oracle rounds once from fp64; allow the two fp64 paths to straddle a bf16 midpoint
            assert np.allclose(new[idx[b], h], S_mem, rtol=2.0 ** -8, atol=0)
            assert np.allclose(out[b, h], np.array(o), rtol=2.0 ** -8, atol=1e-30)
            r = _unrounded_step(m, p["state"][idx[b]], p["q"][b], p["k"][b], p["v"][b],
                                p["g_raw"][b], p["beta_logit"][b], p["A_log"], p["dt_bias"], 0.75)
            assert np.allclose(r["S_new"][h], np.array(S_new), rtol=1e-12, atol=1e-14)
            assert np.allclose(r["o"][h], np.array(o), rtol=1e-12, atol=1e-14)


def pin_exact_rational_core(m):
    """The update with rational inputs, evaluated exactly with Fractions."""
    K = V = 4
    S = [[Fraction(i * V + j - 7, 8) for j in range(V)] for i in range(K)]  # S[k][v]
    kh = [Fraction(1, 2), Fraction(-1, 4), Fraction(3, 8), Fraction(1, 8)]
    qh = [Fraction(-1, 8), Fraction(1, 2), Fraction(1, 4), Fraction(-3, 4)]
    v = [Fraction(3, 2), Fraction(-1, 2), Fraction(5, 4), Fraction(0)]
    d = [Fraction(1), Fraction(1, 2), Fraction(3, 4), Fraction(1, 16)]
    beta = Fraction(3, 4)
    S1 = [[d[i] * S[i][j] for j in range(V)] for i in range(K)]
    u = [beta * (v[j] - sum(S1[i][j] * kh[i] for i in range(K))) for j in range(V)]
    Sn = [[S1[i][j] + kh[i] * u[j] for j in range(V)] for i in range(K)]
    o = [Fraction(1, 2) * sum(Sn[i][j] * qh[i] for i in range(K)) for j in range(V)]
    f = lambda a: np.array(a, dtype=np.float64)  # noqa: E731
    S_new, o_m, u_m = m.decode_step_math(f([[float(x) for x in r] for r in S]), f([float(x) for x in qh]),
                                         f([float(x) for x in kh]), f([float(x) for x in v]),
                                         f([float(x) for x in d]), np.float64(0.75), 0.5)
    assert np.array_equal(S_new, f([[float(x) for x in r] for r in Sn]))
    assert np.array_equal(o_m, f([float(x) for x in o]))
    assert np.array_equal(u_m, f([float(x) for x in u]))


def pin_memory_layout_and_channel_decay(m):
    """State memory is [N][H][V][K]: buf[n, h, v, k] = S[k][v]; the decay scales key channel k."""
    K, V, H = 8, 6, 1
    state = np.zeros((2, H, V, K))
    v0, k0 = 4, 2
    state[1, 0, v0, k0] = 1.0
    g_raw = np.full((1, H, K), -np.inf)
    g_raw[0, 0, k0] = 0.0  # only channel k0 decays: d = exp(-5 sigmoid(dt_bias))
    dt = np.zeros((H, K))
    q = np.zeros((1, H, K))
    q[0, 0, k0] = 1.0
    new, out = m.kda_decode(state, np.array([1]), q, np.ones((1, H, K)), np.zeros((1, H, V)),
                            g_raw, np.full((1, H), -np.inf), np.zeros(H), dt, lower_bound=LB)
    d = math.exp(LB * 0.5)
    exp_state = np.zeros_like(state)
    exp_state[1, 0, v0, k0] = m.round_to_bf16(np.array([d]))[0]
    assert np.array_equal(new, exp_state)
    exp_out = np.zeros((1, H, V))
    exp_out[0, 0, v0] = m.round_to_bf16(np.array([d / math.sqrt(1 + 1e-6)]))[0]
    assert np.array_equal(out, exp_out)


def pin_inactive_slots(m):
    """Indices outside [0, N): zero output, pool untouched; N = 0 makes every row inactive."""
    rng = np.random.default_rng(11)
    p = small_problem(rng, B=5, H=2, K=8, V=8, N=4)
    idx = np.array([-1, 4, 2, 2 ** 31 - 1, -(2 ** 31)])
    new, out = _decode(m, p, idx)
    assert (out[[0, 1, 3, 4]] == 0).all()
    untouched = [0, 1, 3]
    assert np.array_equal(new[untouched], p["state"][untouched])
    assert not np.array_equal(new[2], p["state"][2])
    assert np.abs(out[2]).sum() > 0
    p0 = dict(p)
    p0["state"] = np.zeros((0, 2, 8, 8))
    new0, out0 = _decode(m, p0, np.array([0, 1, -1, 3, 2]))
    assert new0.shape == (0, 2, 8, 8) and (out0 == 0).all()


def pin_verify_is_stepwise(m):
    """T verify tokens equal T single decode steps."""
    rng = np.random.default_rng(12)
    p = small_problem(rng, B=3, H=2, K=8, V=8, N=6, T=4)
    idx = np.array([5, -1, 1])
    new, out = m.kda_verify(p["state"], idx, p["q"], p["k"], p["v"], p["g_raw"], p["beta_logit"],
                            p["A_log"], p["dt_bias"], lower_bound=LB)
    st = p["state"]
    for t in range(4):
        st, o = m.kda_decode(st, idx, p["q"][:, t], p["k"][:, t], p["v"][:, t], p["g_raw"][:, t],
                             p["beta_logit"][:, t], p["A_log"], p["dt_bias"], lower_bound=LB)
        assert np.array_equal(out[:, t], o)
    assert np.array_equal(new, st)
    assert (out[1] == 0).all()


def pin_precomputed_gate_convention(m):
    """Log-space g and beta given directly: decay exp(g) per key channel, beta as
    given; fed the raw form's own g and beta it reproduces the raw form exactly."""
    rng = np.random.default_rng(19)
    p = small_problem(rng, B=3, H=2, K=8, V=8, N=4)
    idx = np.array([3, -1, 1])
    raw_state, raw_out = _decode(m, p, idx)
    g = m.gate_log_decay(p["g_raw"], p["A_log"], p["dt_bias"], LB)
    beta = m.beta_from_logit(p["beta_logit"])
    pre_state, pre_out = m.kda_decode(p["state"], idx, p["q"], p["k"], p["v"], g, beta, None, None,
                                      gate_mode=m.GATE_PRECOMPUTED)
    assert np.array_equal(pre_state, raw_state) and np.array_equal(pre_out, raw_out)
    # closed form: S = 0 row, g = log(1/2) everywhere, beta = 1/4
    q_hat, k_hat, gg, d, bb = m.prologue(p["q"][0], p["k"][0], np.full((2, 8), math.log(0.5)),
                                         np.full(2, 0.25), None, None, LB, m.GATE_PRECOMPUTED)
    assert np.allclose(d, 0.5, rtol=1e-15) and (bb == 0.25).all()
    assert np.array_equal(gg, np.full((2, 8), math.log(0.5)))


# ---------------------------------------------------------------- ring

def ring_problem(rng, B=3, H=2, K=8, V=8, N=5, T=3, W=12, hist=None):
    p = small_problem(rng, B=B, H=H, K=K, V=V, N=N, T=T)
    kc = m_free_unit_keys(rng, (N, H, W, K))
    uc = bf16_values(rng, (N, H, W, V), 0.5)
    steps = -rng.uniform(0.0, 5.0, (N, H, W, K)).astype(np.float32)
    gc = np.cumsum(steps, axis=2, dtype=np.float32).astype(np.float64)
    if hist is None:
        hist = rng.integers(0, W // 2, N)
    hist = np.asarray(hist, dtype=np.int64)
    for n in range(N):  # positions past the live history hold NaN sentinels
        kc[n, :, hist[n]:] = np.nan
        uc[n, :, hist[n]:] = np.nan
        gc[n, :, hist[n]:] = np.nan
    p.update(k_cache=kc, u_cache=uc, g_cache=gc, hist_len=hist)
    return p


def m_free_unit_keys(rng, shape):
    x = rng.standard_normal(shape)
    x /= np.linalg.norm(x, axis=-1, keepdims=True)
    bits = x.astype(np.float32).view(np.uint32) & np.uint32(0xFFFF0000)
    return bits.view(np.float32).astype(np.float64)


def _ring(m, p, idx, flush_min, restart=True, scale=1.0, cache_base=None):
    return m.kda_verify_ring(p["state"], idx, p["q"], p["k"], p["v"], p["g_raw"], p["beta_logit"],
                             p["A_log"], p["dt_bias"], p["k_cache"], p["u_cache"], p["g_cache"],
                             p["hist_len"], flush_min, restart_hist_on_flush=restart,
                             lower_bound=LB, scale=scale, cache_base=cache_base)


def pin_ring_replay_closed_form(m):
    """Stepwise replay with exp(G_j - G_{j-1}) equals the closed form with weights exp(G_P - G_j)."""
    rng = np.random.default_rng(13)
    p = ring_problem(rng, N=1, W=16, hist=[16])
    S0 = np.swapaxes(p["state"][0], -1, -2)
    for h in (0, 1, 5, 16):
        a = m.ring_replay(S0, p["k_cache"][0, :, :h], p["u_cache"][0, :, :h], p["g_cache"][0, :, :h])
        b = m.ring_fold_closed_form(S0, p["k_cache"][0, :, :h], p["u_cache"][0, :, :h],
                                    p["g_cache"][0, :, :h])
        assert np.allclose(a, b, rtol=1e-10, atol=1e-12), h
    # one entry by hand: diag(exp(G_0)) S0 + k_0 u_0^T
    one = m.ring_replay(S0, p["k_cache"][0, :, :1], p["u_cache"][0, :, :1], p["g_cache"][0, :, :1])
    ref = np.exp(p["g_cache"][0, :, 0])[:, :, None] * S0 \
        + p["k_cache"][0, :, 0, :, None] * p["u_cache"][0, :, 0, None, :]
    assert np.allclose(one, ref, rtol=1e-14, atol=1e-16)


def pin_ring_outputs_replay(m):
    """Every o_t equals S_P^T q_hat_t, S_P being the checkpoint replayed through the written ring."""
    rng = np.random.default_rng(14)
    p = ring_problem(rng, B=2, N=3, T=4, W=12, hist=[0, 2, 5])
    idx = np.array([2, 0])
    r = _ring(m, p, idx, flush_min=9, scale=1.5)
    for b, n in enumerate(idx):
        h0 = int(p["hist_len"][n])
        S0 = np.swapaxes(r["state"][n], -1, -2)
        q_hat = m.l2_normalize(p["q"][b])
        for t in range(4):
            P = h0 + t
            S = m.ring_fold_closed_form(S0, r["k_cache"][n, :, :P + 1], r["u_cache"][n, :, :P + 1],
                                        r["g_cache"][n, :, :P + 1])
            o = 1.5 * np.einsum("hkv,hk->hv", S, q_hat[t])
            assert np.allclose(r["out"][b, t], o, rtol=2.0 ** -8, atol=1e-6)
        # the history before h0 and the sentinels after h0 + T are untouched
        assert np.array_equal(r["k_cache"][n, :, :h0], p["k_cache"][n, :, :h0])
        assert np.isnan(r["k_cache"][n, :, h0 + 4:]).all()
        assert np.isnan(r["g_cache"][n, :, h0 + 4:]).all()
        assert np.array_equal(r["state"][n], p["state"][n])  # no fold
        assert r["hist_len"][n] == p["hist_len"][n]
    # stored entries are k_hat in bf16, u in bf16 and G in fp32
    n = 0
    ks = r["k_cache"][n, :, :4]
    assert np.array_equal(ks, m.round_to_bf16(m.l2_normalize(p["k"][1])).transpose(1, 0, 2))
    assert np.array_equal(r["u_cache"][n, :, :4], m.round_to_bf16(r["u_cache"][n, :, :4]))
    G = r["g_cache"][n, :, :4]
    assert np.array_equal(G, m.round_to_fp32(G))
    g = m.gate_log_decay(p["g_raw"][1], p["A_log"], p["dt_bias"], LB)  # [T, H, K]
    assert np.array_equal(G[:, 0], m.round_to_fp32(g[0]))
    assert np.allclose(np.diff(G, axis=1), np.swapaxes(g[1:], 0, 1), rtol=0, atol=1e-4)


def pin_ring_chained_calls(m):
    """One call with T tokens equals T calls with one token each (hist_len advanced in between)."""
    rng = np.random.default_rng(15)
    p = ring_problem(rng, B=2, N=3, T=4, W=12, hist=[2, 0, 1])
    idx = np.array([0, 2])
    whole = _ring(m, p, idx, flush_min=9)
    st = dict(p)
    outs = []
    for t in range(4):
        pt = dict(st)
        for key in ("q", "k", "v", "g_raw", "beta_logit"):
            pt[key] = p[key][:, t:t + 1]
        r = _ring(m, pt, idx, flush_min=9)
        outs.append(r["out"][:, 0])
        st.update(state=r["state"], k_cache=r["k_cache"], u_cache=r["u_cache"], g_cache=r["g_cache"])
        hl = r["hist_len"].copy()
        hl[idx] += 1
        st["hist_len"] = hl
    for key in ("state", "k_cache", "u_cache", "g_cache"):
        assert np.array_equal(whole[key], st[key], equal_nan=True), key
    assert np.array_equal(whole["out"], np.stack(outs, axis=1))
    # the last single-token call replays the ring written by the earlier ones
    assert np.array_equal(whole["state_fp64"], r["state_fp64"])
    # and replaying the whole written ring from the checkpoint lands on the same state
    for b, n in enumerate(idx):
        P = int(p["hist_len"][n]) + 4
        S0 = np.swapaxes(whole["state"][n], -1, -2)
        S = m.ring_replay(S0, whole["k_cache"][n, :, :P], whole["u_cache"][n, :, :P],
                          whole["g_cache"][n, :, :P])
        assert np.array_equal(S, whole["state_fp64"][b])


def pin_ring_fold(m):
    """hist_len >= flush_min folds first: checkpoint = bf16(replay); new tokens from position 0."""
    rng = np.random.default_rng(16)
    W, T, fm = 16, 4, 9
    p = ring_problem(rng, B=3, N=4, T=T, W=W, hist=[9, 12, 8, 16])
    idx = np.array([0, 2, 3])
    r = _ring(m, p, idx, flush_min=fm)
    for n, folds in ((0, True), (2, False), (3, True)):
        h = int(p["hist_len"][n])
        S0 = np.swapaxes(p["state"][n], -1, -2)
        if folds:
            Sh = m.ring_fold_closed_form(S0, p["k_cache"][n, :, :h], p["u_cache"][n, :, :h],
                                         p["g_cache"][n, :, :h])
            got = np.swapaxes(r["state"][n], -1, -2)
            assert np.allclose(got, m.round_to_bf16(Sh), rtol=2.0 ** -7, atol=1e-30)
            assert r["hist_len"][n] == 0
            assert np.isfinite(r["g_cache"][n, :, :T]).all()
            # positions T..h-1 keep the consumed history, untouched
            assert np.array_equal(r["k_cache"][n, :, T:h], p["k_cache"][n, :, T:h])
        else:
            assert np.array_equal(r["state"][n], p["state"][n])
            assert r["hist_len"][n] == h
            assert np.isfinite(r["g_cache"][n, :, h:h + T]).all()
    b = 1  # slot 2 is not folding: G continues from G_{h-1}
    g = m.gate_log_decay(p["g_raw"][b], p["A_log"], p["dt_bias"], LB)
    assert np.array_equal(r["g_cache"][2, :, 8], m.round_to_fp32(p["g_cache"][2, :, 7] + g[0]))
    b = 0  # slot 0 folded: G restarts at 0
    g = m.gate_log_decay(p["g_raw"][b], p["A_log"], p["dt_bias"], LB)
    assert np.array_equal(r["g_cache"][0, :, 0], m.round_to_fp32(g[0]))
    # without restart the fold still commits the checkpoint but leaves hist_len to the caller
    r2 = _ring(m, p, idx, flush_min=fm, restart=False)
    assert r2["hist_len"][0] == 9 and np.array_equal(r2["state"], r["state"])


def pin_ring_inactive_and_bad_hist(m):
    """Out-of-range slots and hist_len outside [0, W] touch nothing; the latter sets the error bit."""
    rng = np.random.default_rng(17)
    p = ring_problem(rng, B=4, N=4, T=2, W=8, hist=[3, -1, 9, 2])
    idx = np.array([1, 2, 7, -3])
    r = _ring(m, p, idx, flush_min=5)
    assert (r["out"] == 0).all()
    for key in ("state", "k_cache", "u_cache", "g_cache", "hist_len"):
        assert np.array_equal(r[key], np.asarray(p[key], dtype=r[key].dtype), equal_nan=True), key
    assert r["error_word"] == m.RING_ERR_HIST_LEN
    r = _ring(m, p, np.array([0, 3, -1, 4]), flush_min=5)
    assert r["error_word"] == 0


def pin_ring_single_token_is_decode_with_stored_values(m):
    """Empty history, one token: the step is the decode step fed the stored k~ and the G-derived decay."""
    rng = np.random.default_rng(18)
    p = ring_problem(rng, B=1, N=1, T=1, W=4, hist=[0])
    r = _ring(m, p, np.array([0]), flush_min=2)
    q_hat, k_hat, g, d, beta = m.prologue(p["q"][0, 0], p["k"][0, 0], p["g_raw"][0, 0],
                                          p["beta_logit"][0, 0], p["A_log"], p["dt_bias"], LB)
    kt = m.round_to_bf16(k_hat)
    G0 = m.round_to_fp32(g)
    S = np.swapaxes(p["state"][0], -1, -2)
    S1 = np.exp(G0)[:, :, None] * S
    u = m.round_to_bf16(beta[:, None] * (p["v"][0, 0] - np.einsum("hkv,hk->hv", S1, kt)))
    Sn = S1 + kt[:, :, None] * u[:, None, :]
    o = m.round_to_bf16(np.einsum("hkv,hk->hv", Sn, q_hat))
    assert np.array_equal(r["out"][0, 0], o)
    assert np.array_equal(r["u_cache"][0, :, 0], u)
    assert np.array_equal(r["g_cache"][0, :, 0], G0)


def pin_ring_cache_base_is_a_rotation(m):
    """A ring stored from entry cache_base on (circularly) computes what the same ring stored from
    entry 0 computes: same outputs, checkpoint and hist_len, and the written ring rotated alike.
    Slots fold and not, and some live histories and appended tokens wrap past the last entry."""
    rng = np.random.default_rng(19)
    W, T, fm = 8, 3, 5
    p = ring_problem(rng, B=4, N=5, T=T, W=W, hist=[2, 6, 4, 0, 5])
    idx = np.array([0, 1, 2, 4])
    cb = np.array([7, 5, 3, 1, 6])
    r0 = _ring(m, p, idx, flush_min=fm)
    q = dict(p)
    for key in ("k_cache", "u_cache", "g_cache"):
        q[key] = np.stack([np.roll(p[key][n], cb[n], axis=1) for n in range(5)])
    r1 = _ring(m, q, idx, flush_min=fm, cache_base=cb)
    for key in ("out", "state", "hist_len"):
        assert np.array_equal(r1[key], r0[key]), key
    for key in ("k_cache", "u_cache", "g_cache"):
        back = np.stack([np.roll(r1[key][n], -cb[n], axis=1) for n in range(5)])
        assert np.array_equal(back, r0[key], equal_nan=True), key
    assert r1["error_word"] == 0
    # the wrap is exercised: slot 1 (cb 5, six live entries) stores positions 0..2 at entries 5..7
    # and positions 3..5 at entries 0..2
    assert np.array_equal(r1["k_cache"][1][:, 0], p["k_cache"][1][:, 3])


def pin_ring_bad_cache_base(m):
    """cache_base outside [0, W) skips the slot (zero output, nothing touched) and sets its error bit."""
    rng = np.random.default_rng(20)
    p = ring_problem(rng, B=2, N=3, T=2, W=8, hist=[3, 2, 1])
    r = _ring(m, p, np.array([0, 1]), flush_min=5, cache_base=np.array([8, -1, 0]))
    assert (r["out"] == 0).all()
    for key in ("state", "k_cache", "u_cache", "g_cache", "hist_len"):
        assert np.array_equal(r[key], np.asarray(p[key], dtype=r[key].dtype), equal_nan=True), key
    assert r["error_word"] == m.RING_ERR_CACHE_BASE
    r = _ring(m, p, np.array([2, -1]), flush_min=5, cache_base=np.array([8, -1, 7]))
    assert r["error_word"] == 0


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
