"""kda_verify_ring_fp8 (the ring verify on an fp8 checkpoint pool) on the GPU, through the C ABI.

The reading: kda_verify_ring's call with the pool's exact values as the
checkpoint; a fold requantizes the replayed state row by row (decided in
fp32, as the fp8 decode requantizes), writes codes and scales, and the new
tokens continue from their exact values. Checked:

* rows that do not fold compute, bit for bit, what kda_verify_ring computes
  on a bf16 pool holding the pool's exact values (every value of these pools
  is a bf16 value), and leave codes and scales untouched;
* against the oracle (kda_verify_ring_fp8) from the same pool: outputs
  (2e-2 + 2e-2 |o_ref|), hist_len, k~ (1 ulp), G, the untouched ring entries,
  the error word, and the folded rows' codes and scales with the fp8 decode's
  bounds around the oracle's unrounded folded state (its slack: 2^-16 of the
  row's largest magnitude for the fold's fp32 sums of up to 64 entries);
* token by token, teacher-forced from the GPU's own checkpoint after the call
  (the requantized one where the row folded) with the ring tests' bounds.
"""

from dataclasses import replace

import numpy as np
import pytest
import torch

import oracle
from harness import assert_output_close, f64, gpu_ring, ring_teacher_forced
from linear_attention_ssm_step_gb300 import kda, workloads
from test_fp8_gpu import check_state
from test_ring_gpu import ring_ulps

pytestmark = pytest.mark.gpu

FOLD_SLACK = 2.0 ** -16


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def make(B, N, T=8, W=32, flush_min=9, fold=0.5, seed=0, **kw):
    w = workloads.ring_inputs(B, N, T=T, W=W, flush_min=flush_min, fold_frac=fold, seed=seed, **kw)
    codes, scales = workloads.fp8_pool(N, H=w.H, seed=seed + 3)
    return w, codes, scales


def ring_fp8(wd, c, s, restart=True, **kw):
    r = wd.ring
    kw.setdefault("gate_mode", wd.gate_mode)
    if r.get("cache_base") is not None:
        kw.setdefault("cache_base", r["cache_base"])
    return kda.kda_verify_ring_fp8(c, s, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log,
                                   wd.dt_bias, r["k_cache"], r["u_cache"], r["g_cache"], r["hist_len"],
                                   r["flush_min"], restart_hist_on_flush=restart, **kw)


def oracle_ring_fp8(w, codes, scales, restart=True):
    r = w.ring
    return oracle.kda_verify_ring_fp8(
        codes.numpy(), f64(scales), f64(w.state_indices), f64(w.q), f64(w.k), f64(w.v), f64(w.g_raw),
        f64(w.beta_logit), f64(w.A_log), f64(w.dt_bias), f64(r["k_cache"]), f64(r["u_cache"]), f64(r["g_cache"]),
        f64(r["hist_len"]), r["flush_min"], restart_hist_on_flush=restart, gate_mode=w.gate_mode,
        cache_base=None if r.get("cache_base") is None else f64(r["cache_base"]))


def _valid_rows(w):
    idx = w.state_indices.numpy().astype(np.int64)
    hist0 = w.ring["hist_len"].numpy().astype(np.int64)
    cb0 = (np.zeros(w.N, dtype=np.int64) if w.ring.get("cache_base") is None
           else w.ring["cache_base"].numpy().astype(np.int64))
    valid = (idx >= 0) & (idx < w.N)
    valid[valid] = ((hist0[idx[valid]] >= 0) & (hist0[idx[valid]] <= w.ring["W"])
                    & (cb0[idx[valid]] >= 0) & (cb0[idx[valid]] < w.ring["W"]))
    return idx, hist0, cb0, valid


def check_ring_fp8(w, codes, scales, dev, rows=None, restart=True):
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = ring_fp8(wd, c_d, s_d, restart=restart, error_word=err)
    torch.cuda.synchronize()
    sub = w if rows is None else w.select_rows(rows)
    ref = oracle_ring_fp8(sub, codes, scales, restart)
    got_out = f64(out) if rows is None else f64(out)[rows]
    got_c, got_s = c_d.cpu().numpy(), s_d.cpu().double().numpy()
    W, fm, T = w.ring["W"], w.ring["flush_min"], w.T

    idx, hist0, cb0, valid = _valid_rows(sub)
    assert (got_out[~valid] == 0).all()
    assert_output_close(got_out, ref["out"])
    slots = idx[valid]
    fslots = slots[hist0[slots] >= fm]
    if fslots.size:
        check_state(got_c[fslots], got_s[fslots], ref["codes"][fslots], ref["scales"][fslots],
                    np.stack([ref["folded"][int(n)] for n in fslots]), slack=FOLD_SLACK)
    # every slot that no row of the whole call folded keeps codes and scales
    idx_all, hist_all, _, valid_all = _valid_rows(w)
    all_folded = idx_all[valid_all][hist_all[idx_all[valid_all]] >= fm]
    keep = np.setdiff1d(np.arange(w.N), all_folded)
    assert np.array_equal(got_c[keep], codes.numpy()[keep]), "codes of a slot that did not fold changed"
    assert np.array_equal(got_s[keep], scales.double().numpy()[keep]), "scales of a slot that did not fold changed"

    assert np.array_equal(f64(wd.ring["hist_len"])[slots], ref["hist_len"][slots])
    kc, uc, gc = f64(wd.ring["k_cache"]), f64(wd.ring["u_cache"]), f64(wd.ring["g_cache"])
    for n in slots:
        base = 0 if hist0[n] >= fm else hist0[n]
        new = [(cb0[n] + base + t) % W for t in range(T)]
        assert float(ring_ulps(kc[n][:, new], ref["k_cache"][n][:, new]).max()) <= 1.0
        G, Gr = gc[n][:, new], ref["g_cache"][n][:, new]
        assert np.all(np.abs(G - Gr) <= 1e-5 * (1.0 + np.abs(Gr))), "G differs"
        untouched = np.ones(W, dtype=bool)
        untouched[new] = False
        for name, got in (("k_cache", kc), ("u_cache", uc), ("g_cache", gc)):
            assert np.array_equal(got[n][:, untouched], f64(w.ring[name])[n][:, untouched], equal_nan=True), name
    assert int(err.item()) == ref["error_word"]
    # u~ and the outputs token by token, from the GPU's own checkpoint after the call
    after = replace(wd, state=torch.from_numpy(oracle.dequantize(got_c, got_s)).to(dev))
    ring_teacher_forced(w, after, out, rows=rows)
    return wd, c_d, s_d, out, ref


@pytest.mark.parametrize("B,fold", [(1, 1.0), (6, 0.5), (32, 0.0), (32, 0.5), (32, 1.0)])
def test_fp8_ring_matches_oracle(dev, B, fold):
    w, codes, scales = make(B, B + 24, fold=fold, seed=700 + B + int(10 * fold),
                            inactive_frac=0.2 if B == 6 else 0.0)
    check_ring_fp8(w, codes, scales, dev)


@pytest.mark.parametrize("fold", [0.0, 0.5])
def test_fp8_ring_rows_without_fold_equal_bf16_ring(dev, fold):
    """The fp8 checkpoint enters the kernel as the bf16 operand the bf16 pool
    would give: rows that do not fold are the bf16 ring's, bit for bit."""
    w, codes, scales = make(24, 40, fold=fold, seed=720 + int(10 * fold))
    deq = oracle.dequantize(codes.numpy(), scales.double().numpy())
    pool = torch.from_numpy(deq).to(torch.bfloat16)
    assert np.array_equal(f64(pool), deq), "the pool's values are bf16 values"
    a = w.to(dev)
    b = replace(w, state=pool).to(dev)
    c, s = codes.to(dev), scales.to(dev)
    oa = ring_fp8(a, c, s)
    ob = gpu_ring(b)
    torch.cuda.synchronize()
    idx, hist0, _, valid = _valid_rows(w)
    plain = valid & (hist0[np.clip(idx, 0, w.N - 1)] < w.ring["flush_min"])
    assert plain.sum() >= 10
    assert torch.equal(oa[torch.as_tensor(plain)].view(torch.int16), ob[torch.as_tensor(plain)].view(torch.int16))
    sl = torch.as_tensor(idx[plain])
    for name in ("k_cache", "u_cache", "g_cache", "hist_len"):
        x, y = a.ring[name].cpu()[sl], b.ring[name].cpu()[sl]
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)), name


def test_fp8_ring_serving_batch_512_sampled(dev):
    """T = 8, W = 32, flush_min = 9, B = 512, half the rows folding: all rows
    run, 16 compared with the oracle."""
    w, codes, scales = make(512, 576, fold=0.5, seed=730)
    rows = np.sort(np.random.default_rng(3).choice(512, 16, replace=False))
    check_ring_fp8(w, codes, scales, dev, rows=rows)


@pytest.mark.parametrize("T,W,flush_min", [(4, 16, 13), (16, 32, 17), (1, 16, 16), (16, 64, 49)])
def test_fp8_ring_other_widths_and_token_counts(dev, T, W, flush_min):
    w, codes, scales = make(6, 16, T=T, W=W, flush_min=flush_min, fold=0.5, seed=740 + T + W)
    check_ring_fp8(w, codes, scales, dev)


@pytest.mark.parametrize("fold", [0.0, 0.5])
def test_fp8_ring_circular_cache_base(dev, fold):
    w, codes, scales = make(12, 20, fold=fold, seed=750 + int(10 * fold), circular=True)
    assert w.ring["cache_base"] is not None
    check_ring_fp8(w, codes, scales, dev)


def test_fp8_ring_precomputed_gate_without_restart(dev):
    w, codes, scales = make(6, 12, fold=1.0, seed=760, gate_mode=1)
    w.A_log = w.dt_bias = None
    wd, _, _, _, _ = check_ring_fp8(w, codes, scales, dev, restart=False)
    idx = w.state_indices.long()
    assert torch.equal(wd.ring["hist_len"].cpu()[idx], w.ring["hist_len"][idx])


@pytest.mark.parametrize("H", [1, 64])
def test_fp8_ring_other_head_counts(dev, H):
    w, codes, scales = make(3, 6, fold=0.5, seed=770 + H, H=H)
    check_ring_fp8(w, codes, scales, dev)


def test_fp8_ring_invalid_history_sets_error_and_touches_nothing(dev):
    w, codes, scales = make(4, 8, fold=0.5, seed=780)
    idx = w.state_indices.long()
    w.ring["hist_len"][idx[0]] = -1
    w.ring["hist_len"][idx[1]] = 33
    wd, c_d, _, out, ref = check_ring_fp8(w, codes, scales, dev)
    assert ref["error_word"] == kda.KDA_ERR_HIST_LEN
    for b in (0, 1):
        n = int(idx[b])
        assert (out[b].float() == 0).all()
        assert torch.equal(c_d[n].cpu(), codes[n])


def test_fp8_ring_graph_replay_is_deterministic(dev):
    w, codes, scales = make(6, 12, fold=0.5, seed=790)
    wd = w.to(dev)
    c, s = codes.to(dev), scales.to(dev)
    snap = {k: v.clone() for k, v in wd.ring.items() if isinstance(v, torch.Tensor)}
    c0, s0 = c.clone(), s.clone()

    def reset():
        c.copy_(c0)
        s.copy_(s0)
        for k, v in snap.items():
            wd.ring[k].copy_(v)

    ring_fp8(wd, c, s)
    torch.cuda.synchronize()
    reset()
    out = torch.empty((6, 8, 12, 128), dtype=torch.bfloat16, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        ring_fp8(wd, c, s, out=out)
    res = []
    for _ in range(2):
        reset()
        graph.replay()
        torch.cuda.synchronize()
        res.append([out.clone(), c.clone(), s.clone()] + [wd.ring[k].clone() for k in snap])
    for x, y in zip(res[0], res[1]):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


def test_fp8_ring_rejects_bad_arguments(dev):
    w, codes, scales = make(2, 3, fold=0.5, seed=795)
    wd = w.to(dev)
    c, s = codes.to(dev), scales.to(dev)
    with pytest.raises(kda.KdaError) as e:
        ring_fp8(wd, c, s, config_override=0)
    assert e.value.status == kda.KDA_EUNSUPPORTED
    flat = torch.empty(codes.numel() + 16, dtype=torch.uint8, device=dev)
    mis = flat[1:1 + codes.numel()].view(codes.shape)
    mis.copy_(c)
    with pytest.raises(kda.KdaError) as e:
        ring_fp8(wd, mis, s)
    assert e.value.status == kda.KDA_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(mis.cpu(), codes), "nothing ran"
