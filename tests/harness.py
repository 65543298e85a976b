"""Shared test helpers: run the oracle and the CUDA library on the same workload,
and the tolerances the comparisons use.

Tolerances:
  * outputs: |o - o_ref| <= 2e-2 + 2e-2 |o_ref| element-wise;
  * state after one step: |s - s_ref| <= 2 bf16 ulps, the ulp taken at
    max(|s_ref|, 2^-12 M) where M is the largest |s_ref| of that (slot, head).
    The floor comes from the fp32 arithmetic of the kernels: the gate's
    exp/sigmoid chain carries a relative error of up to about 2^-20 into the
    decay, so an element whose new value cancels to far below the size of the
    terms it was summed from (|d s| and |k u|, both of order M) carries an
    absolute error of order 2^-20 M. Measured at 2^-12 M, 2 ulps are 2^-18 M,
    four times that.
  * state after t > 1 rounded steps (verify, chained decodes): 2 bf16 ulps at
    the head's scale M. Each step rounds the state to bf16; where the GPU and
    the oracle round one element to neighbouring bf16 values (a 1-ulp
    difference at that element's size, at most ulp(M)), the difference is
    carried into the next steps in absolute terms: the step map
    S -> (I - beta k k^T) diag(d) S is non-expansive, so it does not grow, but
    the element itself may shrink, which makes the same difference many ulps
    of its new, smaller value. The GPU and the oracle each run their own chain
    (no oracle input ever comes from the GPU), so this is the bound that holds.
    Single steps are held to the per-element bound above, and the GPU verify
    equals the GPU's chained decodes bit for bit.
"""

import numpy as np
import torch

import oracle

OUT_ATOL = 2e-2
OUT_RTOL = 2e-2
STATE_ULPS = 2.0
STATE_FLOOR = 2.0 ** -12


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


def assert_state_close(got, ref, what="state", steps=1, max_ulps=STATE_ULPS):
    """The state tolerance of the module docstring for one step (steps = 1) or
    for `steps` > 1 rounded steps."""
    u = state_ulps(got, ref, STATE_FLOOR if steps == 1 else 1.0)
    worst = float(u.max()) if u.size else 0.0
    assert worst <= max_ulps, f"{what}: error reaches {worst:.2f} bf16 ulps (limit {max_ulps}, {steps} step(s))"


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
