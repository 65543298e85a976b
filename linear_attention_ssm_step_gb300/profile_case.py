"""Run one library call on a standard synthetic workload a few times, for
profilers (Nsight Compute) that need a short, clean stream of launches.

  python -m linear_attention_ssm_step_gb300.profile_case decode 512
  python -m linear_attention_ssm_step_gb300.profile_case verify 512 --T 8
  python -m linear_attention_ssm_step_gb300.profile_case ring 512 --T 8 --fold 0.5
  python -m linear_attention_ssm_step_gb300.profile_case ring_fp8 512 --T 8 --fold 0.5
  python -m linear_attention_ssm_step_gb300.profile_case decode_fp8 512
  python -m linear_attention_ssm_step_gb300.profile_case prefill 8 --len 2048

For prefill, B is the number of sequences, each of --len tokens.

Each call is launched --reps times (default 3) on the same inputs, with a
device synchronize after each; nothing is timed here. For the ring, hist_len
is restored before every launch (a fold resets it), so that every launch
folds the same rows.
"""

import argparse

import torch

from . import kda, workloads


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("call", choices=["decode", "verify", "ring", "ring_fp8", "decode_fp8", "prefill"])
    ap.add_argument("B", type=int)
    ap.add_argument("--T", type=int, default=8)
    ap.add_argument("--fold", type=float, default=0.0)
    ap.add_argument("--reps", type=int, default=3)
    ap.add_argument("--config", type=int, default=-1)
    ap.add_argument("--len", type=int, default=16, help="prefill: tokens per sequence")
    ap.add_argument("--H", type=int, default=12, help="prefill: heads")
    a = ap.parse_args()
    dev = torch.device("cuda:0")
    kda.load_library()
    if a.call == "decode":
        w = workloads.decode_inputs(a.B, a.B + 128, seed=2, layout="fused", inactive_frac=0.05).to(dev)
        fn = lambda: kda.kda_decode(w.state, w.state_indices, w.q, w.k, w.v, w.g_raw, w.beta_logit,  # noqa: E731
                                    w.A_log, w.dt_bias, config_override=a.config)
    elif a.call == "decode_fp8":
        w = workloads.decode_inputs(a.B, a.B + 128, seed=2, layout="fused", inactive_frac=0.05).to(dev)
        codes, scales = (t.to(dev) for t in workloads.fp8_pool(a.B + 128, seed=5))
        fn = lambda: kda.kda_decode_fp8(codes, scales, w.state_indices, w.q, w.k, w.v, w.g_raw,  # noqa: E731
                                        w.beta_logit, w.A_log, w.dt_bias, config_override=a.config)
    elif a.call == "prefill":
        w = workloads.prefill_inputs([a.len] * a.B, a.B + 8, seed=90 + a.B, layout="fused", H=a.H).to(dev)
        ws = kda.prefill_workspace(a.len * a.B, a.B, a.H, dev)  # the two-stage configurations' workspace
        fn = lambda: kda.kda_prefill(w.state, w.state_indices, w.cu_seqlens, w.q, w.k, w.v, w.g_raw,  # noqa: E731
                                     w.beta_logit, w.A_log, w.dt_bias, config_override=a.config, workspace=ws)
    elif a.call == "verify":
        w = workloads.decode_inputs(a.B, a.B + 64, seed=3, T=a.T).to(dev)
        fn = lambda: kda.kda_verify(w.state, w.state_indices, w.q, w.k, w.v, w.g_raw, w.beta_logit,  # noqa: E731
                                    w.A_log, w.dt_bias, config_override=a.config)
    elif a.call == "ring":
        w = workloads.ring_inputs(a.B, a.B + 64, T=a.T, W=32, flush_min=9, fold_frac=a.fold, seed=4).to(dev)
        r = w.ring
        fn = lambda: kda.kda_verify_ring(w.state, w.state_indices, w.q, w.k, w.v, w.g_raw,  # noqa: E731
                                         w.beta_logit, w.A_log, w.dt_bias, r["k_cache"], r["u_cache"],
                                         r["g_cache"], r["hist_len"], r["flush_min"], config_override=a.config)
    else:  # ring_fp8: the ring on an fp8 checkpoint pool
        w = workloads.ring_inputs(a.B, a.B + 64, T=a.T, W=32, flush_min=9, fold_frac=a.fold, seed=4)
        codes, scales = (t.to(dev) for t in workloads.fp8_pool(a.B + 64, seed=5))
        w.state = None  # the bf16 pool is not used
        w = w.to(dev)
        r = w.ring
        fn = lambda: kda.kda_verify_ring_fp8(codes, scales, w.state_indices, w.q, w.k, w.v, w.g_raw,  # noqa: E731
                                             w.beta_logit, w.A_log, w.dt_bias, r["k_cache"], r["u_cache"],
                                             r["g_cache"], r["hist_len"], r["flush_min"],
                                             config_override=a.config)
    hist0 = w.ring["hist_len"].clone() if a.call in ("ring", "ring_fp8") else None
    for _ in range(a.reps):
        if hist0 is not None:
            w.ring["hist_len"].copy_(hist0)
        fn()
        torch.cuda.synchronize()
    print(f"{a.call} B={a.B} ran {a.reps} times")


if __name__ == "__main__":
    main()
