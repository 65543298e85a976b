"""kda_verify_ring on the GPU against the oracle: replay of the live history,
fold into the checkpoint, appended ring entries, hist_len bookkeeping, the
inactive and invalid-history rules, and replay consistency on the GPU.

Every call's new ring entries are checked token by token against one-token
oracle calls made from what the GPU wrote (harness.ring_teacher_forced), so
each u~ is held per element to the single-step bound; the folded checkpoint
is one rounding of the replayed history and held to the same bound."""

import numpy as np
import pytest
import torch

import oracle
from harness import (DRIFT_ULPS, assert_drift_close, assert_output_close, assert_state_close, f64, gpu_ring, oracle_ring,
                     ring_teacher_forced, state_ulps)
from linear_attention_ssm_step_gb300 import kda, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def ring_ulps(got, ref, floor=None):
    """bf16 ulps of ring rows [..., W, D], the floor taken per (slot, head, entry) row."""
    got, ref = np.asarray(got), np.asarray(ref)
    if floor is None:
        return state_ulps(got[..., None, :], ref[..., None, :])
    return state_ulps(got[..., None, :], ref[..., None, :], floor=floor)


def check_ring(w, dev, rows=None, restart=True, **kw):
    wd = w.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gpu_ring(wd, restart=restart, error_word=err, **kw)
    torch.cuda.synchronize()
    sub = w if rows is None else w.select_rows(rows)
    ref = oracle_ring(sub, restart=restart)
    got_out = f64(out) if rows is None else f64(out)[rows]
    idx = sub.state_indices.numpy().astype(np.int64)
    hist0 = w.ring["hist_len"].numpy()
    W = w.ring["W"]
    cb0 = (np.zeros(w.N, dtype=np.int64) if w.ring.get("cache_base") is None
           else w.ring["cache_base"].numpy().astype(np.int64))
    active = (idx >= 0) & (idx < w.N)
    valid = active.copy()
    valid[active] = ((hist0[idx[active]] >= 0) & (hist0[idx[active]] <= W)
                     & (cb0[idx[active]] >= 0) & (cb0[idx[active]] < W))
    assert (got_out[~valid] == 0).all()
    assert_output_close(got_out, ref["out"])
    for n in idx[active & ~valid]:  # skipped for an invalid history: nothing touched
        assert np.array_equal(f64(wd.state)[n], f64(w.state)[n])
        for name in ("k_cache", "u_cache", "g_cache", "hist_len"):
            assert np.array_equal(f64(wd.ring[name])[n], f64(w.ring[name])[n], equal_nan=True), name
    slots = idx[valid]
    T = w.T
    assert_state_close(f64(wd.state)[slots], ref["state"][slots])
    for n in slots:
        folded = hist0[n] >= w.ring["flush_min"]
        if not folded:  # the checkpoint is written only by a fold
            assert np.array_equal(f64(wd.state)[n], f64(w.state)[n])
    assert np.array_equal(f64(wd.ring["hist_len"])[slots], ref["hist_len"][slots])
    kc, uc, gc = f64(wd.ring["k_cache"]), f64(wd.ring["u_cache"]), f64(wd.ring["g_cache"])
    for n in slots:
        base = 0 if hist0[n] >= w.ring["flush_min"] else hist0[n]
        new = [(cb0[n] + base + t) % W for t in range(T)]  # stored entries of the new positions
        assert float(ring_ulps(kc[n][:, new], ref["k_cache"][n][:, new]).max()) <= 1.0
        G, Gr = gc[n][:, new], ref["g_cache"][n][:, new]
        assert np.all(np.abs(G - Gr) <= 1e-5 * (1.0 + np.abs(Gr))), "G differs"
        # everything else in the ring is untouched, NaN sentinels included
        keep = np.ones(W, dtype=bool)
        keep[new] = False
        for name, got in (("k_cache", kc), ("u_cache", uc), ("g_cache", gc)):
            assert np.array_equal(got[n][:, keep], f64(w.ring[name])[n][:, keep], equal_nan=True), name
    assert int(err.item()) == ref["error_word"]
    # u~ (and again the outputs, k~, G) token by token, the oracle started from the GPU's own entries
    ring_teacher_forced(w, wd, out, rows=rows)
    return wd, out, ref


@pytest.mark.parametrize("fold", [0.0, 0.5, 1.0])
@pytest.mark.parametrize("B", [1, 6, 32])
def test_ring_matches_oracle(dev, B, fold):
    w = workloads.ring_inputs(B, B + 64, T=8, W=32, flush_min=9, fold_frac=fold, seed=500 + B,
                              inactive_frac=0.2 if B == 6 else 0.0)
    check_ring(w, dev)


def test_ring_serving_batch_512_sampled(dev):
    """T = 8, W = 32, flush_min = 9, B = 512, half the rows folding: all rows run,
    20 compared with the oracle."""
    w = workloads.ring_inputs(512, 576, T=8, W=32, flush_min=9, fold_frac=0.5, seed=4)
    rows = np.sort(np.random.default_rng(2).choice(512, 20, replace=False))
    check_ring(w, dev, rows=rows)


def test_ring_whole_head_config_is_the_default(dev):
    w = workloads.ring_inputs(5, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=7)
    a, b = w.to(dev), w.to(dev)
    oa = gpu_ring(a, config_override=3)
    ob = gpu_ring(b)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    for name in ("k_cache", "u_cache", "g_cache", "hist_len"):
        x, y = a.ring[name], b.ring[name]
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)), name
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_ring_w16_t4(dev):
    """The other mode of the pages: ring width 16, T = 4, flush_min = 13."""
    w = workloads.ring_inputs(6, 20, T=4, W=16, flush_min=13, fold_frac=0.5, seed=8)
    check_ring(w, dev)


@pytest.mark.parametrize("T,W,flush_min", [(16, 32, 17), (1, 16, 16), (8, 64, 40), (16, 64, 49)])
def test_ring_other_widths_and_token_counts(dev, T, W, flush_min):
    """T = 16 and T = 1 token slots, and a 64-wide ring whose histories run to
    flush_min - 1 + T entries."""
    w = workloads.ring_inputs(6, 16, T=T, W=W, flush_min=flush_min, fold_frac=0.5, seed=40 + T + W)
    check_ring(w, dev)


@pytest.mark.parametrize("fold", [0.0, 0.5, 1.0])
def test_ring_circular_cache_base(dev, fold):
    """Rings stored from a random entry per slot (cache_base), histories and
    appends wrapping past the last entry."""
    w = workloads.ring_inputs(12, 20, T=8, W=32, flush_min=9, fold_frac=fold, seed=60, circular=True)
    assert w.ring["cache_base"] is not None
    check_ring(w, dev)


def test_ring_circular_matches_rotated_plain_ring(dev):
    """A circular ring computes what the same ring stored from entry 0 computes, bit for bit."""
    w = workloads.ring_inputs(6, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=61, circular=True)
    a = w.to(dev)
    b = w.to(dev)
    cb = [int(c) for c in w.ring["cache_base"]]
    for name in ("k_cache", "u_cache", "g_cache"):
        b.ring[name] = torch.stack([torch.roll(b.ring[name][n], -cb[n], dims=1) for n in range(12)]).contiguous()
    b.ring["cache_base"] = None
    oa, ob = gpu_ring(a), gpu_ring(b)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))
    assert torch.equal(a.ring["hist_len"], b.ring["hist_len"])
    for name in ("k_cache", "u_cache", "g_cache"):
        back = torch.stack([torch.roll(a.ring[name][n], -cb[n], dims=1) for n in range(12)])
        x, y = back, b.ring[name]
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)), name


def test_ring_invalid_cache_base_sets_error_and_touches_nothing(dev):
    w = workloads.ring_inputs(4, 8, T=8, W=32, flush_min=9, fold_frac=0.5, seed=62, circular=True)
    idx = w.state_indices.long()
    w.ring["cache_base"][idx[0]] = 32
    w.ring["cache_base"][idx[1]] = -1
    wd, out, ref = check_ring(w, dev)
    assert ref["error_word"] == kda.KDA_ERR_CACHE_BASE
    for b in (0, 1):
        n = int(idx[b])
        assert (out[b].float() == 0).all()


@pytest.mark.parametrize("H", [1, 3, 64])
def test_ring_other_head_counts(dev, H):
    w = workloads.ring_inputs(3, 6, T=8, W=32, flush_min=9, fold_frac=0.5, seed=70 + H, H=H)
    check_ring(w, dev)


def test_ring_large_batch_sampled(dev):
    """B = 2048, half the rows folding: about 54 (row, head) items per persistent CTA; 12 rows
    compared with the oracle, the written ring and hist_len checked on those rows."""
    w = workloads.ring_inputs(2048, 2112, T=8, W=32, flush_min=9, fold_frac=0.5, seed=71)
    rows = np.sort(np.random.default_rng(7).choice(2048, 12, replace=False))
    check_ring(w, dev, rows=rows)


def test_ring_misaligned_pool_uses_plain_copies_with_same_bits(dev):
    w = workloads.ring_inputs(6, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=14, inactive_frac=0.2)
    a, b = w.to(dev), w.to(dev)
    flat = torch.empty(b.state.numel() + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[1:1 + b.state.numel()].view(b.state.shape)  # 2-byte aligned only
    mis.copy_(b.state)
    assert mis.data_ptr() % 16 == 2
    b.state = mis
    oa = gpu_ring(a)
    ob = gpu_ring(b)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))
    for name in ("k_cache", "u_cache", "g_cache", "hist_len"):
        x, y = a.ring[name], b.ring[name]
        assert torch.equal(x.view(torch.int16) if x.dtype == torch.bfloat16 else x.view(torch.int32),
                           y.view(torch.int16) if y.dtype == torch.bfloat16 else y.view(torch.int32)), name


def test_ring_without_restart_keeps_hist_len(dev):
    w = workloads.ring_inputs(4, 10, T=8, W=32, flush_min=9, fold_frac=1.0, seed=9)
    wd, _, _ = check_ring(w, dev, restart=False)
    idx = w.state_indices.long()
    assert torch.equal(wd.ring["hist_len"].cpu()[idx], w.ring["hist_len"][idx])


def test_ring_invalid_history_sets_error_and_touches_nothing(dev):
    w = workloads.ring_inputs(4, 8, T=8, W=32, flush_min=9, seed=10)
    idx = w.state_indices.long()
    w.ring["hist_len"][idx[0]] = -1
    w.ring["hist_len"][idx[1]] = 33
    wd, out, ref = check_ring(w, dev)
    assert ref["error_word"] == kda.KDA_ERR_HIST_LEN
    for b in (0, 1):
        n = int(idx[b])
        assert (out[b].float() == 0).all()
        assert torch.equal(wd.state[n].cpu().view(torch.int16), w.state[n].view(torch.int16))


def test_ring_single_token_calls_chain(dev):
    """Without a fold, T single-token calls (hist_len advanced by the caller
    between them) compute what one T-token call computes: the later calls
    replay what the earlier ones appended. Each single-token call is checked
    against the oracle from the ring the GPU had written before it; k~ and G
    are the same bits as the T-token call's; u~ and the outputs of the two GPU
    chains (which sum the same terms in other orders) stay within the
    tolerance and the drift bound of each other."""
    from dataclasses import replace
    from harness import token_slice
    T = 6
    w = workloads.ring_inputs(5, 12, T=T, W=32, flush_min=20, fold_frac=0.0, seed=11)
    hl = w.ring["hist_len"]
    hl.copy_(torch.minimum(hl, torch.full_like(hl, 10)))  # no slot reaches flush_min within the T calls
    a = w.to(dev)
    out_all = gpu_ring(a)
    c = w.to(dev)
    idx = c.state_indices.long()
    outs = []
    for t in range(T):
        before = replace(token_slice(w, t, t + 1), state=c.state.cpu(),
                         ring={k: (v.cpu() if isinstance(v, torch.Tensor) else v) for k, v in c.ring.items()})
        wt = token_slice(c, t, t + 1)
        outs.append(gpu_ring(wt))
        torch.cuda.synchronize()
        ring_teacher_forced(before, wt, outs[-1])
        c.ring["hist_len"][idx] += 1
    torch.cuda.synchronize()
    assert_output_close(f64(torch.cat(outs, dim=1)), f64(out_all))
    ug, ur = f64(c.ring["u_cache"]), f64(a.ring["u_cache"])
    assert np.array_equal(np.isnan(ug), np.isnan(ur))  # the same positions written, sentinels kept
    assert float(ring_ulps(np.nan_to_num(ug), np.nan_to_num(ur), floor=1.0).max()) <= DRIFT_ULPS
    assert torch.equal(a.ring["k_cache"].view(torch.int16), c.ring["k_cache"].view(torch.int16))
    assert torch.equal(a.ring["g_cache"].view(torch.int32), c.ring["g_cache"].view(torch.int32))


def test_ring_cuda_graph_bitwise(dev):
    w = workloads.ring_inputs(6, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=12)
    wd = w.to(dev)
    snap = {k: v.clone() for k, v in wd.ring.items() if isinstance(v, torch.Tensor)}
    st0 = wd.state.clone()

    def reset():
        wd.state.copy_(st0)
        for k, v in snap.items():
            wd.ring[k].copy_(v)

    gpu_ring(wd)
    torch.cuda.synchronize()
    reset()
    out = torch.empty((6, 8, 12, 128), dtype=torch.bfloat16, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_ring(wd, out=out)
    res = []
    for _ in range(2):
        reset()
        graph.replay()
        torch.cuda.synchronize()
        res.append([out.clone(), wd.state.clone()] + [wd.ring[k].clone() for k in snap])
    for x, y in zip(res[0], res[1]):
        assert torch.equal(x.view(torch.uint8), y.view(torch.uint8))


def test_ring_precomputed_gate_convention(dev):
    w = workloads.ring_inputs(6, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=13, gate_mode=1)
    w.A_log = w.dt_bias = None
    check_ring(w, dev)


def test_ring_serving_loop(dev):
    """Six consecutive T = 8 calls on the same slots, as a speculative-decoding
    loop runs them: between calls the caller advances hist_len by the tokens it
    accepted (8, 5, 8, 3, 8, 8), and a call folds whenever the history has
    reached flush_min = 9. Every call is checked against the oracle started
    from the GPU's own checkpoint, ring and hist_len before it (check_ring:
    outputs, the fold's checkpoint per element, u~ token by token); the oracle
    also runs its own chain from the first call (drift diagnostic: outputs
    within tolerance, hist_len equal, checkpoints within the drift bound)."""
    from dataclasses import replace
    B, N, T, W, FM = 4, 8, 8, 32, 9
    w0 = workloads.ring_inputs(B, N, T=T, W=W, flush_min=FM, fold_frac=0.0, seed=40)
    w0.ring["hist_len"].zero_()
    idx_t = w0.state_indices
    idx = idx_t.numpy().astype(np.int64)
    g_state = w0.state.to(dev)
    g_ring = {k: w0.ring[k].to(dev) for k in ("k_cache", "u_cache", "g_cache", "hist_len")}
    r_state = f64(w0.state)
    r_ring = {k: f64(w0.ring[k]) for k in ("k_cache", "u_cache", "g_cache", "hist_len")}
    folds = 0
    for call, accepted in enumerate((8, 5, 8, 3, 8, 8)):
        w = workloads.decode_inputs(B, N, seed=50 + call, T=T, indices=idx_t)
        folds += int((r_ring["hist_len"][idx] >= FM).any())
        before = replace(w, state=g_state.cpu(), ring=dict({k: v.cpu() for k, v in g_ring.items()}, W=W,
                                                               flush_min=FM, cache_base=None))
        wd = replace(before.to(dev), state=g_state, ring=dict(g_ring, W=W, flush_min=FM, cache_base=None))
        out = gpu_ring(wd)
        torch.cuda.synchronize()
        _check_finished_call(before, wd, out)
        ref = oracle.kda_verify_ring(r_state, idx, f64(w.q), f64(w.k), f64(w.v), f64(w.g_raw), f64(w.beta_logit),
                                     f64(w.A_log), f64(w.dt_bias), r_ring["k_cache"], r_ring["u_cache"],
                                     r_ring["g_cache"], r_ring["hist_len"], FM)
        assert_output_close(f64(out), ref["out"], f"call {call} output against the oracle's chain")
        assert np.array_equal(f64(g_ring["hist_len"]), ref["hist_len"]), f"call {call} hist_len"
        assert_drift_close(f64(g_state)[idx], ref["state"][idx], f"call {call} checkpoint chains")
        r_state = ref["state"]
        r_ring = {k: ref[k] for k in ("k_cache", "u_cache", "g_cache")}
        r_ring["hist_len"] = ref["hist_len"].copy()
        # the caller accepts `accepted` of the T draft tokens
        r_ring["hist_len"][idx] += accepted
        g_ring["hist_len"][idx_t.long().to(dev)] += accepted
    assert folds >= 2


def _check_finished_call(w, wd, out, restart=True):
    """check_ring's comparisons for a call already made: w holds the inputs
    before it (CPU), wd the GPU tensors after it."""
    ref = oracle_ring(w, restart=restart)
    assert_output_close(f64(out), ref["out"])
    idx = w.state_indices.numpy().astype(np.int64)
    hist0 = w.ring["hist_len"].numpy()
    assert_state_close(f64(wd.state)[idx], ref["state"][idx], "checkpoint")
    for n in idx:
        if hist0[n] < w.ring["flush_min"]:
            assert np.array_equal(f64(wd.state)[n], f64(w.state)[n])
    assert np.array_equal(f64(wd.ring["hist_len"])[idx], ref["hist_len"][idx])
    ring_teacher_forced(w, wd, out)
