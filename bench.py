#!/usr/bin/env python3
"""Benchmark of the KDA serving step (libkda_gb300.so) on GB300.

Headline step: one kda_decode call (T = 1) over a 512-row serving batch:
H = 12, K = V = 128, bf16 state pool of 640 slots, q/k/v strided views of a
fused [512, 4672] bf16 projection buffer, about 5% of the rows inactive.
value = algorithmic state GB/s (bytes the method must move / kernel time),
measured with CUDA events on the launching stream around each call, the call
replayed from a CUDA graph (so host-side argument marshalling stays out of the
device timing), with L2 emptied between calls (a 2 x L2 write, then a 2 x L2
read of another buffer, so that no dirty lines are left). The same line
carries:
  e2e          the same metric through the public binding as a serving loop
               runs it: every step's inputs copied in from pinned host memory
               and its output copied back, all inside one timed region,
               pipelined over two buffer sets (the pool stays resident);
  roofline     the decode kernel's achieved GB/s against the measured HBM peak;
  warm         the headline call in a steady decode loop (16 chained calls in
               one graph, no flush), per call, with its fraction of the peak;
  t8           the metric's T = 8 half at B = 512: verify and ring (W = 32,
               0/50/100% folding), us, GB/s and fraction of the peak;
  cpu_baseline the fp64 CPU oracle on a bounded sample of the same workload,
               on one core and on all host cores;
  sweep        T=1 decode at B = 1..2048, L2-cold per call and warm in 16-step
               loops (also on an fp8 pool, with T = 8 verify on the fp8 pool
               at B = 1, 32, 512, and with the pre-computed gate
               convention at B = 8, 512), T=8 verify and T=8 ring verify at
               B = 1, 32, 512 (0/50/100% of rows folding; the ring also on an
               fp8 checkpoint pool at B = 512), L2-cold, and the
               varlen prefill at 1 x 4096, 8 x 2048, 64 x 256 and 512 x 16
               tokens (H = 12) and two shapes of the prefill page (H = 16,
               1 x 16384; H = 4, lengths 1..15) with a caller's workspace
               and the library's choice of configuration (two stages from
               512 tokens per sequence), each with its median and
               10th/90th percentiles, and (state GB/s points) the fraction
               of the measured HBM peak.
               streaming_reference: a plain PyTorch in-place multiply over the
               headline state's bytes, the same flush (context for the roofline).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl reference] [--no-sweep]

For N > 1, launch one process per GPU with torch.distributed.run; each rank
processes its own batch and pool (no data exchange), the timed region is
bracketed by barriers and the time taken is the maximum over ranks.
--impl reference times the CPU oracle (the only other implementation of this
path) on the same workload, a bounded sample of rows per step.
"""

import argparse
from dataclasses import replace
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

# the CPU oracle runs single-threaded; its reported core count relies on this
for _v in ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS"):
    os.environ.setdefault(_v, "1")

import numpy as np  # noqa: E402
import torch  # noqa: E402

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_attention_ssm_step_gb300 import kda, traffic, workloads  # noqa: E402

METRIC = "KDA decode µs/step and state GB/s (% HBM peak) at B=1..512, T=1 and T=8"
WORKLOAD = ("T=1 KDA decode, B=512, H=12, K=V=128, bf16 state pool [640,12,128,128] ~N(0,0.02^2), "
            "q/k/v strided views of a fused bf16 [512,4672] projection buffer, ~5% of rows inactive")
B_HEAD, N_HEAD, SEED_HEAD = 512, 640, 2
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "kda_decode_b512_ncu.md")
FALLBACK_HBM_GBS = 6800.0


# ------------------------------------------------------------------ helpers

DECODE_SOURCES = ("include/kda.h", "linear_attention_ssm_step_gb300/csrc/kda_device.cuh",
                  "linear_attention_ssm_step_gb300/csrc/kda_launch.h",
                  "linear_attention_ssm_step_gb300/csrc/kda_step.cu")


def kernel_source_hash():
    """Hash of the sources the decode kernel is compiled from; a profile summary
    taken from other sources is stale."""
    h = hashlib.sha256()
    for rel in DECODE_SOURCES:
        h.update(open(os.path.join(ROOT, rel), "rb").read())
    return h.hexdigest()[:16]


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        peaks = json.load(open(path))
        return float(peaks["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic():
    """dram bytes per launch of the decode kernel from the committed ncu summary,
    or None when the summary is missing or was taken from different sources."""
    try:
        text = open(PROFILE_SUMMARY).read()
    except OSError:
        return None
    vals = {}
    for line in text.splitlines():
        if ":" in line and line.strip().startswith(("source_hash", "traffic_bytes_per_launch")):
            k, v = line.strip().strip("`").split(":", 1)
            vals[k.strip()] = v.strip().strip("`")
    if vals.get("source_hash") != kernel_source_hash() or "traffic_bytes_per_launch" not in vals:
        return None
    return float(vals["traffic_bytes_per_launch"])


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device):
        self.proc = None
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits", "-lms", "50"]
        try:
            uuid = str(torch.cuda.get_device_properties(device).uuid)
            cmd += ["-i", uuid if uuid.startswith("GPU-") else "GPU-" + uuid]
        except Exception:
            pass
        self.cmd = cmd

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.2)
        return self

    def __exit__(self, *exc):
        time.sleep(0.1)
        self.lines = []
        if self.proc is not None:
            self.proc.terminate()
            out, _ = self.proc.communicate(timeout=10)
            self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        if not self.lines:
            return None
        sm, smax, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 8:
                continue
            try:
                sm.append(float(f[0]))
                smax.append(float(f[1]))
            except ValueError:
                continue
            for name, val in zip(names, f[4:8]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    if n_gpus != world and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device=None):
    """Largest value of x over all ranks (x itself when there is one rank)."""
    if world == 1:
        return x
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


class L2Flush:
    """Empties L2 between timed calls: writes a buffer of twice its size, then
    reads a second buffer of that size. The write evicts the call's inputs; the
    read evicts the write's dirty lines, so that the timed call neither finds
    its inputs in L2 nor writes back the flush's data inside its own timing."""

    def __init__(self, device):
        l2 = torch.cuda.get_device_properties(device).L2_cache_size
        n = max(2 * l2, 256 << 20) // 4
        self.buf = torch.empty(n, dtype=torch.int32, device=device)
        self.rbuf = torch.ones(n, dtype=torch.float32, device=device)
        self.sink = torch.empty((), dtype=torch.float32, device=device)
        self.nbytes = n * 4

    def __call__(self):
        self.buf.fill_(1)
        torch.sum(self.rbuf, dim=(0,), out=self.sink)  # fp32 in, fp32 out: one reduction kernel, no cast


def graphed(fn):
    """fn captured once in a CUDA graph; returns the replay. The library makes
    no host-side decisions that depend on device data, so a replay repeats the
    call exactly (on whatever the captured buffers hold at replay time)."""
    fn()  # first call outside capture: one-time kernel attribute setup
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g.replay


def time_calls(fn, steps, warmup, before=None, world=1):
    """Per-call device time (ms) of fn() with CUDA events on the current stream;
    before() runs outside the event pair ahead of every call."""
    for _ in range(warmup):
        if before:
            before()
        fn()
    torch.cuda.synchronize()
    barrier(world)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    for s, e in evs:
        if before:
            before()
        s.record()
        fn()
        e.record()
    torch.cuda.synchronize()
    barrier(world)
    return [s.elapsed_time(e) for s, e in evs]


# ------------------------------------------------------------------ the GPU arm

def decode_call(wd, out):
    return lambda: kda.kda_decode(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                                  wd.A_log, wd.dt_bias, out=out)


def n_active(w):
    idx = w.state_indices.to(torch.int64)
    return int(((idx >= 0) & (idx < w.N)).sum())


def headline(dev, steps, warmup, world, rank):
    w = workloads.decode_inputs(B_HEAD, N_HEAD, seed=SEED_HEAD + rank, layout="fused", inactive_frac=0.05)
    wd = w.to(dev)
    out = torch.empty((B_HEAD, 12, 128), dtype=torch.bfloat16, device=dev)
    flush = L2Flush(dev)
    act = n_active(w)
    nbytes = traffic.decode_bytes(act, B_HEAD - act)
    replay = graphed(decode_call(wd, out))
    with ClockSampler(dev) as clk:
        times = time_calls(replay, steps, warmup, before=flush, world=world)
    total_ms = max_over_ranks(sum(times), world, dev)
    # Steady state beside the cold figure: 16 consecutive calls on the same batch
    # (the state chained in place) in one CUDA graph, no flush between them.
    loop = graphed(lambda: [decode_call(wd, out)() for _ in range(16)])
    warm_ms = statistics.median(time_calls(loop, max(10, steps // 4), warmup)) / 16
    return dict(w=w, wd=wd, out=out, times=times, total_ms=total_ms, nbytes=nbytes, clocks=clk.summary(),
                active=act, flush=flush, warm_ms=warm_ms)


def e2e(dev, h, steps, warmup, world):
    """The same call through the binding as a serving loop runs it: every step's
    inputs copied in from pinned host memory and its output copied back, all
    inside the timed region. The loop is pipelined over two sets of device input
    and output buffers: step i+1's inputs copy in (one stream) while step i
    computes (the launching stream) and step i-1's output copies out (a third
    stream); events order each buffer's reuse. The state pool (250 MB) is larger
    than L2, so no flush runs between steps. Returns the max over ranks of the
    timed region (ms) and the bytes copied in and out per step."""
    w, wd = h["w"], h["wd"]
    names = ("qkv", "g_raw", "beta_logit", "state_indices")
    host_in = {name: getattr(w, name).pin_memory() for name in names}
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    sets = [wd, replace(wd, **{name: getattr(wd, name).clone() for name in names})]
    outs = [torch.empty_like(h["out"]) for _ in range(2)]
    host_out = [torch.empty(outs[0].shape, dtype=outs[0].dtype).pin_memory() for _ in range(2)]
    d2h = host_out[0].numel() * host_out[0].element_size()
    calls = [kda.prepare_decode(x.state, x.state_indices, x.q, x.k, x.v, x.g_raw, x.beta_logit, x.A_log,
                                x.dt_bias, out=o) for x, o in zip(sets, outs)]
    main = torch.cuda.current_stream(dev)
    s_in, s_out = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev = lambda: torch.cuda.Event()  # noqa: E731
    copied, computed, read, sent = [ev(), ev()], [ev(), ev()], [ev(), ev()], [ev(), ev()]

    def run(n, start=None):
        for i in range(n + 1):
            b = i % 2
            if i < n:  # inputs of step i into set b, once step i-2 has read them
                with torch.cuda.stream(s_in):
                    if start is not None and i == 0:
                        s_in.wait_event(start)
                    if i >= 2:
                        s_in.wait_event(read[b])
                    for name in names:
                        getattr(sets[b], name).copy_(host_in[name], non_blocking=True)
                    copied[b].record(s_in)
            if i >= 1:  # step i-1: compute, then its output out
                c = (i - 1) % 2
                main.wait_event(copied[c])
                if i >= 3:
                    main.wait_event(sent[c])  # output set c of step i-3 has left
                calls[c]()
                computed[c].record(main)
                read[c].record(main)
                with torch.cuda.stream(s_out):
                    s_out.wait_event(computed[c])
                    host_out[c].copy_(outs[c], non_blocking=True)
                    sent[c].record(s_out)
        for c in range(2):
            main.wait_event(sent[c])

    run(max(warmup, 2))
    torch.cuda.synchronize()
    barrier(world)
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(main)
    run(steps, start=t0)
    t1.record(main)
    torch.cuda.synchronize()
    barrier(world)
    total_ms = max_over_ranks(t0.elapsed_time(t1), world, dev)
    return total_ms, h2d, d2h


def spread(ts):
    """Median, 10th and 90th percentile of per-call times (ms), in µs."""
    q = statistics.quantiles(ts, n=10, method="inclusive")
    return round(statistics.median(ts) * 1e3, 2), round(q[0] * 1e3, 2), round(q[-1] * 1e3, 2)


def sweep(dev, steps=100, warmup=100):
    """Each point: the median (and 10th/90th percentiles) of `steps` timed calls
    after `warmup` untimed ones (100 and 100: the pages' protocol)."""
    flush = L2Flush(dev)
    res = {"t1_decode": []}  # more keys added below
    for B in (1, 8, 16, 32, 64, 128, 256, 512, 1024, 2048):
        w = workloads.decode_inputs(B, B + 128, seed=10 + B, layout="fused")
        wd = w.to(dev)
        out = torch.empty((B, 12, 128), dtype=torch.bfloat16, device=dev)
        fn = decode_call(wd, out)
        us, p10, p90 = spread(time_calls(graphed(fn), steps, warmup, before=flush))
        td = statistics.median(time_calls(fn, steps, warmup, before=flush))
        nb = traffic.decode_bytes(B)
        row = {"B": B, "us": us, "us_p10": p10, "us_p90": p90, "GB/s": round(nb / us / 1e3, 1),
               "us_direct": round(td * 1e3, 2), "config": kda.kda_select_config(B, 1)}
        # WARM L2, marked as such: a decode loop of 16 consecutive steps on the same
        # slots (the state chained in place) captured as one graph, per step. Up to
        # B = 128 the state stays in L2 between steps, as it does when serving; at
        # larger B most of it does not.
        loop = graphed(lambda: [fn() for _ in range(16)])
        tw = statistics.median(time_calls(loop, steps, warmup)) / 16
        row["us_warm_16step_graph"] = round(tw * 1e3, 2)
        res["t1_decode"].append(row)
        del w, wd
    # Context for the small-batch points: the same cold single-call timing of a
    # graph holding one trivial kernel (a one-element fill), the launch and
    # event floor every cold single-call figure above includes.
    tiny = torch.zeros(1, dtype=torch.float32, device=dev)
    t = statistics.median(time_calls(graphed(lambda: tiny.fill_(1.0)), steps, warmup, before=flush))
    res["launch_floor"] = {"what": "one-element fill in a CUDA graph, the same cold single-call timing",
                           "us": round(t * 1e3, 2)}
    # Context for the decode's roofline: a plain streaming kernel (PyTorch's
    # in-place elementwise multiply) over the bytes of the headline's state
    # (486 active rows: read and written once), behind the same flush.
    x = torch.ones(486 * traffic.STATE_BYTES // 2, dtype=torch.bfloat16, device=dev)
    t = statistics.median(time_calls(graphed(lambda: x.mul_(1.0)), steps, warmup, before=flush))
    nb = 2 * x.numel() * 2
    res["streaming_reference"] = {"what": "torch in-place bf16 multiply, read + write once, graph replay",
                                  "bytes": nb, "us": round(t * 1e3, 2), "GB/s": round(nb / t / 1e6, 1)}
    del x
    # T=1 decode on an fp8 (E4M3) pool with per-row power-of-two scales: the
    # same activations, half the state bytes (all rows active, pool B+128)
    res["t1_decode_fp8_state"] = []
    for B in (1, 8, 32, 128, 512):
        w = workloads.decode_inputs(B, B + 128, seed=50 + B, layout="fused")
        codes, scales = workloads.fp8_pool(B + 128, seed=60 + B)
        wd = w.to(dev)
        c_d, s_d = codes.to(dev), scales.to(dev)
        out = torch.empty((B, 12, 128), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_decode_fp8(c_d, s_d, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw,  # noqa: E731
                                        wd.beta_logit, wd.A_log, wd.dt_bias, out=out)
        us, p10, p90 = spread(time_calls(graphed(fn), steps, warmup, before=flush))
        loop = graphed(lambda: [fn() for _ in range(16)])
        tw = statistics.median(time_calls(loop, steps, warmup)) / 16
        nb = traffic.decode_fp8_bytes(B)
        res["t1_decode_fp8_state"].append({"B": B, "us": us, "us_p10": p10, "us_p90": p90,
                                           "GB/s": round(nb / us / 1e3, 1),
                                           "us_warm_16step_graph": round(tw * 1e3, 2)})
        del w, wd, c_d, s_d
    # T=8 verify on the fp8 pool (kda_verify_fp8): T decode steps per call,
    # the row requantized after every token
    res["t8_verify_fp8_state"] = []
    for B in (1, 32, 512):
        w = workloads.decode_inputs(B, B + 128, seed=70 + B, T=8, layout="fused")
        codes, scales = workloads.fp8_pool(B + 128, seed=80 + B)
        wd = w.to(dev)
        c_d, s_d = codes.to(dev), scales.to(dev)
        out = torch.empty((B, 8, 12, 128), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_verify_fp8(c_d, s_d, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw,  # noqa: E731
                                        wd.beta_logit, wd.A_log, wd.dt_bias, out=out)
        us, p10, p90 = spread(time_calls(graphed(fn), steps, warmup, before=flush))
        nb = traffic.verify_fp8_bytes(B, 8)
        res["t8_verify_fp8_state"].append({"B": B, "us": us, "us_p10": p10, "us_p90": p90,
                                           "GB/s": round(nb / us / 1e3, 1)})
        del w, wd, c_d, s_d
    res["t1_decode_precomputed_gate"] = []
    for B in (8, 512):
        w = workloads.decode_inputs(B, B + 128, seed=40 + B, layout="fused", gate_mode=1)
        wd = w.to(dev)
        out = torch.empty((B, 12, 128), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_decode(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw,  # noqa: E731
                                    wd.beta_logit, None, None, out=out, gate_mode=kda.KDA_GATE_PRECOMPUTED)
        t = statistics.median(time_calls(graphed(fn), steps, warmup, before=flush))
        res["t1_decode_precomputed_gate"].append({"B": B, "us": round(t * 1e3, 2),
                                                  "GB/s": round(traffic.decode_bytes(B) / t / 1e6, 1)})
        del w, wd
    res["t8_verify"] = t8_verify_points(dev, (1, 32, 512), steps, warmup, flush)
    # varlen prefill (kda_prefill): S sequences of equal length packed row after
    # row, each filling its own slot; L2 flushed before each call
    # (the last two are shapes of the prefill page's portfolio: H16 with one
    # 16384-token sequence, and H4 with sequences of 1..15 tokens)
    res["prefill"] = []
    for name, lens, Hh in (("1x4096", [4096], 12), ("8x2048", [2048] * 8, 12), ("64x256", [256] * 64, 12),
                           ("512x16", [16] * 512, 12), ("h16_1x16384", [16384], 16),
                           ("h4_seq1_to_15", list(range(1, 16)), 4)):
        S, toks = len(lens), sum(lens)
        w = workloads.prefill_inputs(lens, S + 8, seed=90 + S, layout="fused", H=Hh)
        wd = w.to(dev)
        st0 = wd.state.clone()
        out = torch.empty((toks, Hh, 128), dtype=torch.bfloat16, device=dev)
        ws = kda.prefill_workspace(toks, S, Hh, dev)  # the caller-owned workspace, allocated once
        fn = lambda: kda.kda_prefill(wd.state, wd.state_indices, wd.cu_seqlens, wd.q, wd.k, wd.v,  # noqa: E731
                                     wd.g_raw, wd.beta_logit, wd.A_log, wd.dt_bias, out=out, workspace=ws)

        def reset():
            wd.state.copy_(st0)
            flush()

        n = max(10, steps // 4)
        us, p10, p90 = spread(time_calls(graphed(fn), n, max(3, warmup // 4), before=reset))
        flops = traffic.prefill_flops(toks, Hh)
        res["prefill"].append({"case": name, "H": Hh, "seqs": S, "tokens": toks, "us": us, "us_p10": p10,
                               "us_p90": p90, "Mtokens/s": round(toks / us, 3),
                               "TFLOP/s": round(flops / us / 1e6, 2),
                               "config": kda.kda_select_prefill_ws_config(toks, S, Hh),
                               "workspace_MB": round(ws.numel() / 1e6, 1)})
        del w, wd, st0, out, ws
    res["t8_ring_w32"] = t8_ring_points(dev, [(1, 32), (32, 32), (512, 32)], steps, warmup, flush)
    # the pages' own ring width for T = 8, at the serving batch
    res["t8_ring_w16"] = t8_ring_points(dev, [(512, 16)], steps, warmup, flush)
    # the ring's checkpoint on an fp8 pool, at the serving batch
    res["t8_ring_fp8_w32"] = t8_ring_points(dev, [(512, 32)], steps, warmup, flush, fp8=True)
    add_fractions(res)
    return res


def t8_verify_points(dev, Bs, steps, warmup, flush):
    """T = 8 kda_verify at each B (pool B + 64, all rows active), L2 emptied before every call."""
    pts = []
    for B in Bs:
        w = workloads.decode_inputs(B, B + 64, seed=20 + B, T=8)
        wd = w.to(dev)
        out = torch.empty((B, 8, 12, 128), dtype=torch.bfloat16, device=dev)
        fn = lambda: kda.kda_verify(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw,  # noqa: E731
                                    wd.beta_logit, wd.A_log, wd.dt_bias, out=out)
        us, p10, p90 = spread(time_calls(graphed(fn), steps, warmup, before=flush))
        nb = traffic.verify_bytes(B, 8)
        pts.append({"B": B, "us": us, "us_p10": p10, "us_p90": p90, "GB/s": round(nb / us / 1e3, 1),
                    "config": kda.kda_select_config(B, 8)})
        del w, wd
    return pts


def t8_ring_points(dev, cases, steps, warmup, flush, fp8=False):
    """T = 8 kda_verify_ring (fp8: kda_verify_ring_fp8 on an fp8 checkpoint pool),
    flush_min = 9, for each (B, W) at 0 / 50 / 100 % of rows folding; the pool,
    the ring and hist_len restored and L2 emptied before every call."""
    pts = []
    for B, W in cases:
        for fold in (0.0, 0.5, 1.0):
            w = workloads.ring_inputs(B, B + 64, T=8, W=W, flush_min=9, fold_frac=fold, seed=30 + B)
            wd = w.to(dev)
            saved = {k: v.clone() for k, v in wd.ring.items() if isinstance(v, torch.Tensor)}
            if fp8:
                codes, scales = (x.to(dev) for x in workloads.fp8_pool(B + 64, seed=31 + B))
                pool = [codes, scales]
                wd.state = None  # the bf16 pool is not used
            else:
                pool = [wd.state]
            pool0 = [x.clone() for x in pool]
            out = torch.empty((B, 8, 12, 128), dtype=torch.bfloat16, device=dev)
            r = wd.ring

            def restore():
                for x, x0 in zip(pool, pool0):
                    x.copy_(x0)
                for k, v in saved.items():
                    r[k].copy_(v)
                flush()

            ring_args = (wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log, wd.dt_bias,
                         r["k_cache"], r["u_cache"], r["g_cache"], r["hist_len"], 9)
            if fp8:
                fn = lambda: kda.kda_verify_ring_fp8(codes, scales, *ring_args, out=out)  # noqa: E731
            else:
                fn = lambda: kda.kda_verify_ring(pool[0], *ring_args, out=out)  # noqa: E731
            us, p10, p90 = spread(time_calls(graphed(fn), steps, warmup, before=restore))
            idx = w.state_indices.to(torch.int64)
            hists = [int(w.ring["hist_len"][n]) for n in idx]
            nb = traffic.ring_bytes(hists, 8, 9, state_bytes=traffic.FP8_STATE_BYTES if fp8 else traffic.STATE_BYTES)
            pts.append({"B": B, "W": W, "fold": fold, "us": us, "us_p10": p10, "us_p90": p90,
                        "GB/s": round(nb / us / 1e3, 1)})
            del w, wd, saved, pool, pool0
    return pts


def add_fractions(res):
    """Every sweep point with a state GB/s also gets its fraction of the measured HBM peak."""
    peak, _ = measured_peak()
    for key, pts in res.items():
        if not isinstance(pts, list):
            continue
        for pt in pts:
            if "GB/s" in pt and key != "prefill":
                pt["frac"] = round(pt["GB/s"] / peak, 4)


def t8_summary(dev, sweep_res, steps=100, warmup=100):
    """The metric's T = 8 half at the serving batch: verify and the ring (W = 32) at
    B = 512, 0 / 50 / 100 % folding, with their fractions of the measured HBM peak.
    Taken from the sweep when it ran, else measured here."""
    peak, kind = measured_peak()
    if sweep_res is not None:
        ver = [p for p in sweep_res["t8_verify"] if p["B"] == 512]
        ring = [p for p in sweep_res["t8_ring_w32"] if p["B"] == 512]
    else:
        flush = L2Flush(dev)
        ver = t8_verify_points(dev, (512,), steps, warmup, flush)
        ring = t8_ring_points(dev, [(512, 32)], steps, warmup, flush)
    keep = lambda p: {k: p[k] for k in ("B", "fold", "us", "GB/s") if k in p}  # noqa: E731
    return {"verify": [dict(keep(p), frac=round(p["GB/s"] / peak, 4)) for p in ver],
            "ring_w32": [dict(keep(p), frac=round(p["GB/s"] / peak, 4)) for p in ring],
            "peak": peak, "peak_kind": f"{kind} HBM copy bandwidth",
            "how": "one CUDA-graph replay per call, L2 emptied (and the ring restored) before each, median of 100"}


def _oracle_chunk_worker(path, n_iter, q):
    """One forked worker of the all-cores oracle timing: n_iter oracle decode
    calls on the chunk saved at `path`; puts the elapsed seconds on q."""
    import oracle

    a = np.load(path)
    args = tuple(a[k] for k in ("state", "idx", "q", "k", "v", "g_raw", "beta_logit", "A_log", "dt_bias"))
    oracle.kda_decode(*args)
    t0 = time.perf_counter()
    for _ in range(n_iter):
        oracle.kda_decode(*args)
    q.put(time.perf_counter() - t0)


def oracle_all_cores(path, n_iter):
    """Run in a fresh process that has made no CUDA call (so forking is safe):
    one oracle worker per host core, each on its own copy of the chunk; prints
    the core count and the slowest worker's time as one JSON line."""
    import multiprocessing

    cores = len(os.sched_getaffinity(0))
    ctx = multiprocessing.get_context("fork")
    q = ctx.Queue()
    procs = [ctx.Process(target=_oracle_chunk_worker, args=(path, n_iter, q)) for _ in range(cores)]
    for pr in procs:
        pr.start()
    times = [q.get() for _ in procs]
    for pr in procs:
        pr.join()
    print(json.dumps({"cores": cores, "max_s": max(times), "n_iter": n_iter}), flush=True)


def cpu_baseline_all_cores(sub, rows, per_call, seconds=10.0):
    """The oracle on every host core at once: each core runs the same 16-row call
    (its own copy, a compact pool of those rows' slots) in a separate process."""
    import tempfile

    idx = sub.state_indices.to(torch.int64)
    f = lambda t: t.double().numpy()  # noqa: E731
    chunk = {"state": f(sub.state[idx]), "idx": np.arange(len(rows), dtype=np.int32), "q": f(sub.q),
             "k": f(sub.k), "v": f(sub.v), "g_raw": f(sub.g_raw), "beta_logit": f(sub.beta_logit),
             "A_log": f(sub.A_log), "dt_bias": f(sub.dt_bias)}
    n_iter = max(3, int(seconds / per_call))
    with tempfile.TemporaryDirectory() as d:
        path = os.path.join(d, "chunk.npz")
        np.savez(path, **chunk)
        r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-all-cores", path, str(n_iter)],
                           capture_output=True, text=True, timeout=30 * seconds + 120)
    if r.returncode != 0:
        return {"unavailable": (r.stderr.strip().splitlines() or ["worker failed"])[-1][:200]}
    res = json.loads(r.stdout.strip().splitlines()[-1])
    cores, el = res["cores"], res["max_s"]
    gbs = cores * traffic.decode_bytes(len(rows)) * n_iter / el / 1e9
    return {"value": round(gbs, 6), "unit": "GB/s", "cores": cores, "kind": "oracle",
            "sample": f"{cores} processes, each {n_iter} calls on its own copy of {len(rows)} active rows of the "
                      f"B=512 workload; slowest {el:.1f} s; numpy fp64, one thread each"}


def cpu_baseline(seconds=10.0):
    """The fp64 oracle, as it stands, on 16 active rows of the headline workload
    (one thread), plus the same on every host core."""
    import oracle

    w = workloads.decode_inputs(B_HEAD, N_HEAD, seed=SEED_HEAD, layout="fused", inactive_frac=0.05)
    idx = w.state_indices.to(torch.int64)
    rows = [b for b in range(B_HEAD) if 0 <= int(idx[b]) < N_HEAD][:16]
    sub = w.select_rows(rows)
    f = lambda t: t.double().numpy()  # noqa: E731
    args = (f(sub.state), sub.state_indices.numpy(), f(sub.q), f(sub.k), f(sub.v), f(sub.g_raw),
            f(sub.beta_logit), f(sub.A_log), f(sub.dt_bias))
    oracle.kda_decode(*args)  # first touch of the arrays
    n, t0 = 0, time.perf_counter()
    while True:
        oracle.kda_decode(*args)
        n += 1
        el = time.perf_counter() - t0
        if el >= seconds or n >= 200:
            break
    per_call = el / n
    return {"value": round(traffic.decode_bytes(len(rows)) / per_call / 1e9, 6), "unit": "GB/s", "cores": 1,
            "kind": "oracle",
            "sample": f"{len(rows)} active rows of the B=512 workload per call, {n} calls in {el:.1f} s "
                      f"({per_call * 1e3:.1f} ms per call), numpy fp64, one thread",
            "all_cores": cpu_baseline_all_cores(sub, rows, per_call, seconds)}


def run_gpu(args):
    rank, world, local = dist_setup(args.gpus)
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA device (the library has no CPU path)")
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    import __graft_entry__
    __graft_entry__.build()

    h = headline(dev, args.steps, args.warmup, world, rank)
    e2e_ms, h2d, d2h = e2e(dev, h, args.steps, args.warmup, world)
    if rank != 0:
        return
    ms_per_step = h["total_ms"] / args.steps
    gbs = h["nbytes"] * world * args.steps / (h["total_ms"] / 1e3) / 1e9
    per_launch_gbs = h["nbytes"] / (statistics.mean(h["times"]) / 1e3) / 1e9
    peak, peak_kind = measured_peak()
    line = {
        "metric": METRIC,
        "value": round(gbs, 1),
        "unit": "GB/s",
        "us_per_step": round(ms_per_step * 1e3, 2),
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B_HEAD, "T": 1, "H": 12, "K": 128, "V": 128, "pool": N_HEAD,
                   "active_rows": h["active"], "bytes_per_step": h["nbytes"],
                   "l2": (f"flushed between steps ({h['flush'].nbytes >> 20} MiB write, then a "
                          f"{h['flush'].nbytes >> 20} MiB read of another buffer; outside the timed calls)"),
                   "launch": "each timed call is one CUDA-graph replay of kda_decode",
                   "parallelism": f"{world} GPU(s), one independent batch and pool per GPU, no collective on the data path"},
        "e2e": {"value": round(h["nbytes"] * world * args.steps / (e2e_ms / 1e3) / 1e9, 1), "unit": "GB/s",
                "us_per_step": round(e2e_ms / args.steps * 1e3, 2),
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "how": "prepared kda_decode call; each step's inputs copied in from pinned host memory and its "
                       "output copied back inside one timed region over all steps, pipelined over two buffer "
                       "sets on three streams; no L2 flush (the state pool is larger than L2)"},
        "roofline": {"kernel": "kda_step_kernel<128,bulk,T=1>", "bound": "hbm",
                     "achieved": round(per_launch_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(per_launch_gbs / peak, 4), "peak_kind": f"{peak_kind} HBM copy bandwidth",
                     "traffic": profiled_traffic(), "algorithmic_bytes": h["nbytes"]},
        "warm": {"us_per_step": round(h["warm_ms"] * 1e3, 2),
                 "GB/s": round(h["nbytes"] / h["warm_ms"] / 1e6, 1),
                 "frac": round(h["nbytes"] / h["warm_ms"] / 1e6 / peak, 4),
                 "how": "16 consecutive kda_decode calls on the headline batch, state chained in place, captured "
                        "as one CUDA graph, no L2 flush; median over replays, per call"},
        "gpu_launches": args.steps,
        "clocks": h["clocks"],
        "context_b200_pages": {"B512_direct_us": 63.82, "B512_effective_TBps": 6.43,
                               "note": "B200 numbers from the pages, no inactive rows; context only"},
    }
    sw = None if args.no_sweep else sweep(dev)
    line["t8"] = t8_summary(dev, sw)
    if sw is not None:
        line["sweep"] = sw
    line["cpu_baseline"] = cpu_baseline()
    print(json.dumps(line), flush=True)


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    w = workloads.decode_inputs(B_HEAD, N_HEAD, seed=SEED_HEAD, layout="fused", inactive_frac=0.05)
    idx = w.state_indices.to(torch.int64)
    rows = [b for b in range(B_HEAD) if 0 <= int(idx[b]) < N_HEAD][:8]
    sub = w.select_rows(rows)
    f = lambda t: t.double().numpy()  # noqa: E731
    args_ = (f(sub.state), sub.state_indices.numpy(), f(sub.q), f(sub.k), f(sub.v), f(sub.g_raw),
             f(sub.beta_logit), f(sub.A_log), f(sub.dt_bias))
    for _ in range(args.warmup):
        oracle.kda_decode(*args_)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.kda_decode(*args_)
    el = time.perf_counter() - t0
    nbytes = traffic.decode_bytes(len(rows))
    gbs = nbytes * args.steps / el / 1e9
    sample = f"{len(rows)} active rows of the B=512 workload per step, numpy fp64, one thread"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(gbs, 6), "unit": "GB/s",
        "n_gpus": int(os.environ.get("WORLD_SIZE", "1")), "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(el / args.steps * 1e3, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": WORKLOAD, "B": B_HEAD, "T": 1, "H": 12, "K": 128, "V": 128, "pool": N_HEAD},
        "cpu_baseline": {"value": round(gbs, 6), "unit": "GB/s", "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(gbs, 6), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["gb300", "reference"], default="gb300")
    ap.add_argument("--no-sweep", action="store_true", help="skip the B / T / fold sweep")
    ap.add_argument("--oracle-all-cores", nargs=2, metavar=("CHUNK", "N_ITER"), help=argparse.SUPPRESS)
    args = ap.parse_args()
    if args.oracle_all_cores:
        oracle_all_cores(args.oracle_all_cores[0], int(args.oracle_all_cores[1]))
        return
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
