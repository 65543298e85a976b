"""Shared test helpers: run the oracle and the CUDA library on the same workload,
and the tolerances the comparisons use.

Tolerances:
  * outputs: |o - o_ref| <= 2e-2 + 2e-2 |o_ref| element-wise;
  * state, one step from a given bf16 state: |s - s_ref| <= 2 bf16 ulps, the
    ulp taken at max(|s_ref|, 2^-12 M) where M is the largest |s_ref| of that
    (slot, head). The floor comes from the fp32 arithmetic of the kernels: the
    gate's exp/sigmoid chain carries a relative error of up to about 2^-20
    into the decay, so an element whose new value cancels to far below the
    size of the terms it was summed from (|d s| and |k u|, both of order M)
    carries an absolute error of order 2^-20 M. Measured at 2^-12 M, 2 ulps
    are 2^-18 M, four times that.
  * state after several rounded steps (verify, chained decodes, the ring's u~
    after earlier tokens): the same per-element bound, token by token, with
    the oracle "teacher-forced": each token's oracle step starts from the
    GPU's own bf16 state (or ring entries) before that token, which the GPU
    wrote and the oracle only reads as its input. That keeps every comparison
    a single step, whatever the number of tokens.
  * drift diagnostics only (two free-running chains, GPU and oracle, each
    from the same inputs): 2 bf16 ulps at the head's scale M. Where the two
    chains round one element to neighbouring bf16 values, the 1-ulp
    difference is carried into the next steps in absolute terms (the step
    map S -> (I - beta k k^T) diag(d) S is non-expansive) while the element
    itself may shrink; this bound holds for the chains, not per element.
  * prefill state (carried in fp32 across L tokens, rounded to bf16 once;
    there is no intermediate bf16 state to force the oracle with): 2 bf16
    ulps at max(|s_ref|, F_L M), F_L = min(1, max(2^-12, L 2^-11)). Per token
    the fp32 step adds an absolute error of at most about 2^-19 M to an
    element (the 128-term dot products' rounding, at most ~2^-17.5 M, times
    |k_i| <= 1/2 in the update, plus the decay's ~2^-20 M), and the step map
    is non-expansive, so after L tokens the fp32 state is within L 2^-19 M of
    the exact one. The final rounding takes one ulp of the element; the
    other ulp, at least 2^-8 F_L M = L 2^-19 M, covers the carried error.
"""

import numpy as np
import torch

import oracle

OUT_ATOL = 2e-2
OUT_RTOL = 2e-2
STATE_ULPS = 2.0
STATE_FLOOR = 2.0 ** -12
DRIFT_ULPS = 2.0


def prefill_floor(L):
    """F_L of the prefill state bound (module docstring); a one-token sequence
    is one decode step and keeps the single-step floor."""
    return STATE_FLOOR if L <= 1 else min(1.0, max(STATE_FLOOR, L * 2.0 ** -11))


def f64(t):
    """bf16 / fp32 / int tensor -> numpy (fp64 for floating types; exact); None passes."""
    if t is None:
        return None
    t = t.detach().cpu()
    if t.dtype in (torch.bfloat16, torch.float16, torch.float32, torch.float64):
        return t.double().numpy()
    return t.numpy()


def bf16_ulp(mag):
    mag = np.maximum(np.asarray(mag, dtype=np.float64), 2.0 ** -126)
    return np.ldexp(1.0, np.floor(np.log2(mag)).astype(np.int64) - 7)


def output_excess(got, ref):
    """max over elements of |got - ref| / (atol + rtol |ref|); <= 1 passes."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / (OUT_ATOL + OUT_RTOL * np.abs(ref))))


def assert_output_close(got, ref, what="output"):
    e = output_excess(got, ref)
    assert e <= 1.0, f"{what}: error reaches {e:.3f} x the tolerance 2e-2 + 2e-2|ref|"


def state_ulps(got, ref, floor=STATE_FLOOR):
    """Per-element error in bf16 ulps, the ulp taken at max(|ref|, floor * M),
    M the largest |ref| over the last two axes; got/ref [..., V, K]."""
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    if got.size == 0:
        return np.zeros(got.shape)
    M = np.max(np.abs(ref), axis=(-1, -2), keepdims=True)
    mag = np.maximum(np.abs(ref), floor * M)
    return np.abs(got - ref) / bf16_ulp(mag)


def assert_state_close(got, ref, what="state", max_ulps=STATE_ULPS, floor=STATE_FLOOR):
    """One step from a given bf16 state (per element, module docstring)."""
    u = state_ulps(got, ref, floor)
    worst = float(u.max()) if u.size else 0.0
    assert worst <= max_ulps, f"{what}: error reaches {worst:.2f} bf16 ulps (limit {max_ulps}, floor {floor:g} M)"


def assert_drift_close(got, ref, what="state drift", max_ulps=DRIFT_ULPS):
    """Drift diagnostic of two free-running chains: bf16 ulps of the head scale."""
    u = state_ulps(got, ref, 1.0)
    worst = float(u.max()) if u.size else 0.0
    assert worst <= max_ulps, f"{what}: chains {worst:.2f} bf16 ulps of the head scale apart (limit {max_ulps})"


def assert_prefill_state_close(got, ref, L, what="prefill state"):
    """The final state of an L-token prefill (fp32 across tokens, one rounding)."""
    assert_state_close(got, ref, what, floor=prefill_floor(L))


# ------------------------------------------------------------------ runners

def oracle_decode(w, scale=1.0, lower_bound=-5.0):
    return oracle.kda_decode(f64(w.state), f64(w.state_indices), f64(w.q), f64(w.k), f64(w.v),
                             f64(w.g_raw), f64(w.beta_logit), f64(w.A_log), f64(w.dt_bias),
                             lower_bound=lower_bound, scale=scale, gate_mode=w.gate_mode)


def oracle_verify(w, scale=1.0, lower_bound=-5.0):
    return oracle.kda_verify(f64(w.state), f64(w.state_indices), f64(w.q), f64(w.k), f64(w.v),
                             f64(w.g_raw), f64(w.beta_logit), f64(w.A_log), f64(w.dt_bias),
                             lower_bound=lower_bound, scale=scale, gate_mode=w.gate_mode)


def oracle_ring(w, restart=True, scale=1.0, lower_bound=-5.0):
    r = w.ring
    return oracle.kda_verify_ring(f64(w.state), f64(w.state_indices), f64(w.q), f64(w.k), f64(w.v),
                                  f64(w.g_raw), f64(w.beta_logit), f64(w.A_log), f64(w.dt_bias),
                                  f64(r["k_cache"]), f64(r["u_cache"]), f64(r["g_cache"]),
                                  f64(r["hist_len"]), r["flush_min"], restart_hist_on_flush=restart,
                                  lower_bound=lower_bound, scale=scale, gate_mode=w.gate_mode,
                                  cache_base=None if r.get("cache_base") is None else f64(r["cache_base"]))


def gpu_decode(wd, **kw):
    from linear_attention_ssm_step_gb300 import kda
    kw.setdefault("gate_mode", wd.gate_mode)
    return kda.kda_decode(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                          wd.A_log, wd.dt_bias, **kw)


def gpu_verify(wd, **kw):
    from linear_attention_ssm_step_gb300 import kda
    kw.setdefault("gate_mode", wd.gate_mode)
    return kda.kda_verify(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                          wd.A_log, wd.dt_bias, **kw)


def gpu_ring(wd, restart=True, **kw):
    from linear_attention_ssm_step_gb300 import kda
    r = wd.ring
    kw.setdefault("gate_mode", wd.gate_mode)
    if r.get("cache_base") is not None:
        kw.setdefault("cache_base", r["cache_base"])
    return kda.kda_verify_ring(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                               wd.A_log, wd.dt_bias, r["k_cache"], r["u_cache"], r["g_cache"],
                               r["hist_len"], r["flush_min"], restart_hist_on_flush=restart, **kw)


# ------------------------------------------------------------------ teacher forcing

def token_slice(w, t0, t1):
    """Tokens t0 .. t1-1 of a T-token workload, as a (t1 - t0)-token workload on the same pool."""
    from dataclasses import replace
    sl = lambda x: None if x is None else x[:, t0:t1]  # noqa: E731
    return replace(w, T=t1 - t0, g_raw=w.g_raw[:, t0:t1], beta_logit=w.beta_logit[:, t0:t1],
                   qkv=sl(w.qkv), q_sep=sl(w.q_sep), k_sep=sl(w.k_sep), v_sep=sl(w.v_sep))


def decode_token(w, t):
    """Token t of a T-token workload, as a decode (T = None) workload on the same pool."""
    from dataclasses import replace
    pick = lambda x: None if x is None else x[:, t]  # noqa: E731
    return replace(w, T=None, g_raw=w.g_raw[:, t], beta_logit=w.beta_logit[:, t],
                   qkv=pick(w.qkv), q_sep=pick(w.q_sep), k_sep=pick(w.k_sep), v_sep=pick(w.v_sep))


def identity_tokens(w, t_from):
    """A copy of w whose tokens t >= t_from are identity steps: decay 1 and beta 0
    (raw gate: g_raw = beta_logit = -inf; pre-computed: g = beta = 0), which
    leave the state bitwise unchanged."""
    c = w.clone()
    fill = float("-inf") if c.gate_mode == oracle.GATE_RAW else 0.0
    c.g_raw[:, t_from:] = fill
    c.beta_logit[:, t_from:] = fill
    return c


def with_state(w, state_slots):
    """w (rows already selected, all active) on a compact pool holding state_slots [R, H, V, K]."""
    from dataclasses import replace
    R = state_slots.shape[0]
    return replace(w, state=torch.from_numpy(np.ascontiguousarray(state_slots)).to(torch.bfloat16),
                   state_indices=torch.arange(R, dtype=torch.int32))


def verify_teacher_forced(w, dev, rows=None, **kw):
    """Run kda_verify on w (kw go to the call) and check it token by token.

    The GPU's state after each prefix of t tokens comes from a verify of the
    first t tokens on a fresh copy of the pool in the configuration of the full
    call (the state after t tokens does not depend on later tokens); the
    one-token prefix is a two-token call whose second token is an identity
    step, so that the tensor-core configuration (T > 1 only) runs it too. Each
    prefix call's outputs must equal the full call's, bit for bit. Token t is
    then held against one oracle step from the GPU's state after t tokens:
    its output at the output tolerance, the state after it per element at the
    single-step bound. rows: the batch rows given to the oracle (all by
    default); inactive ones must give zero output. Returns (wd, out, cfg)."""
    from linear_attention_ssm_step_gb300 import kda
    T = w.T
    cfg = kw.pop("config_override", -1)
    if cfg < 0:
        cfg = kda.kda_select_config(w.B, T)
    wd = w.to(dev)
    out = gpu_verify(wd, config_override=cfg, **kw)
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    idx = w.state_indices.numpy().astype(np.int64)
    act = (idx[rows] >= 0) & (idx[rows] < w.N)
    got_out = f64(out)[rows]
    assert (got_out[~act] == 0).all(), "inactive rows must give exactly zero"
    arows = rows[act]
    slots = torch.as_tensor(idx[arows])
    states = [f64(w.state)[slots.numpy()]]
    for t in range(1, T):
        pre = identity_tokens(token_slice(w, 0, 2), 1) if t == 1 else token_slice(w, 0, t)
        pd = pre.to(dev)
        out_t = gpu_verify(pd, config_override=cfg, **kw)
        assert torch.equal(out_t[:, :t].view(torch.int16), out[:, :t].view(torch.int16)), \
            f"the {t}-token prefix call computes other outputs than the full call"
        states.append(f64(pd.state[slots.to(dev)]))
        del pd
    states.append(f64(wd.state[slots.to(dev)]))
    sub = w.select_rows(arows)
    for t in range(T):
        ref_state, ref_out = oracle_decode(with_state(decode_token(sub, t), states[t]), **_scale_kw(kw))
        assert_output_close(got_out[act][:, t], ref_out, f"token {t} output")
        assert_state_close(states[t + 1], ref_state, f"state after token {t}")
    return wd, out, cfg


def _scale_kw(kw):
    return {k: kw[k] for k in ("scale", "lower_bound") if k in kw}


def ring_teacher_forced(w, wd, out, rows=None):
    """Token-by-token check of a finished kda_verify_ring call of w (wd: the
    GPU tensors after it, out: its outputs).

    Token t of a valid row is held against a one-token oracle ring call made
    from what the GPU wrote: its checkpoint after the call (the folded one
    where the row folded, else the untouched original) and its ring, with the
    live history ending just before token t's position (the original history,
    or none after a fold, then the GPU's own entries for tokens < t), and no
    fold. Checked: the output of token t, and its u~ (per element, the
    single-step bound over the entry's 128 values), k~ (1 ulp) and G at its
    position. rows: the batch rows to check (all by default)."""
    r = w.ring
    T, W, fm = w.T, r["W"], r["flush_min"]
    rows = np.arange(w.B) if rows is None else np.asarray(rows)
    idx = w.state_indices.numpy().astype(np.int64)
    hist0 = r["hist_len"].numpy().astype(np.int64)
    cb0 = (np.zeros(w.N, dtype=np.int64) if r.get("cache_base") is None
           else r["cache_base"].numpy().astype(np.int64))
    ok = (idx[rows] >= 0) & (idx[rows] < w.N)
    ok[ok] = ((hist0[idx[rows[ok]]] >= 0) & (hist0[idx[rows[ok]]] <= W)
              & (cb0[idx[rows[ok]]] >= 0) & (cb0[idx[rows[ok]]] < W))
    vrows = rows[ok]
    if vrows.size == 0:
        return
    slots = idx[vrows]
    base = np.where(hist0[slots] >= fm, 0, hist0[slots])
    sl_dev = torch.as_tensor(slots).to(wd.state.device)
    st = f64(wd.state[sl_dev])
    kc, uc, gc = (f64(wd.ring[name][sl_dev]) for name in ("k_cache", "u_cache", "g_cache"))
    cb = cb0[slots]
    got_out = f64(out)[vrows]
    sub = w.select_rows(vrows)
    R = len(vrows)
    for t in range(T):
        tok = token_slice(sub, t, t + 1)
        ref = oracle.kda_verify_ring(st, np.arange(R), f64(tok.q), f64(tok.k), f64(tok.v), f64(tok.g_raw),
                                     f64(tok.beta_logit), f64(w.A_log), f64(w.dt_bias), kc, uc, gc,
                                     base + t, W, restart_hist_on_flush=False, gate_mode=w.gate_mode,
                                     cache_base=cb)
        assert ref["error_word"] == 0
        assert_output_close(got_out[:, t], ref["out"][:, 0], f"ring token {t} output")
        for i in range(R):
            P = int((cb[i] + base[i] + t) % W)
            u_got, u_ref = uc[i][:, P], ref["u_cache"][i][:, P]  # [H, 128]
            # k~ = bf16(k_hat) with k_hat computed in fp32 on the GPU: a key
            # within fp32 rounding of a bf16 midpoint may land on the other
            # neighbour (checked below: 1 ulp). u~ then follows from that key:
            # the part sum_k |dk~_k| |(D S)[k, v]| (beta <= 1) of its error is
            # explained, D S the oracle's decayed state before the update.
            dk = np.abs(kc[i][:, P] - ref["k_cache"][i][:, P])  # [H, K]
            if dk.any():
                DS = ref["state_fp64"][i] - ref["k_cache"][i][:, P][:, :, None] * u_ref[:, None, :]
                explained = np.einsum("hk,hkv->hv", dk, np.abs(DS))
                diff = u_got - u_ref
                u_got = u_ref + np.sign(diff) * np.maximum(np.abs(diff) - explained, 0.0)
            assert_state_close(u_got[:, None, :], u_ref[:, None, :], f"ring token {t} u~ (row {vrows[i]})")
            assert float(state_ulps(kc[i][:, P][:, None, :], ref["k_cache"][i][:, P][:, None, :]).max()) <= 1.0
            G, Gr = gc[i][:, P], ref["g_cache"][i][:, P]
            assert np.all(np.abs(G - Gr) <= 1e-5 * (1.0 + np.abs(Gr))), f"ring token {t} G"
