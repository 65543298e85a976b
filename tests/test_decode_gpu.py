"""kda_decode (T = 1) on the GPU against the fp64 oracle, through the C ABI.

Sizes: element-wise comparisons at B up to 32 (several CTAs per head, every
tile size, ragged batches), the 512-row serving batch compared on sampled
rows plus properties checked everywhere, and the edge cases of the pages'
decode kernel (out-of-range slots, empty pool, misaligned and strided
tensors, padded pools, CUDA-graph replay, non-default streams).
"""

import numpy as np
import pytest
import torch

from harness import (DRIFT_ULPS, assert_drift_close, assert_output_close, assert_state_close, f64,
                     gpu_decode, oracle_decode, output_excess, state_ulps, with_state)
from linear_attention_ssm_step_gb300 import kda, workloads

pytestmark = pytest.mark.gpu

DRIFT_ULPS_512 = 2.0  # the 512-step drift diagnostic holds the state tolerance (measured worst: 1 ulp)


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def run_and_check(w, dev, scale=1.0, **kw):
    """Run one decode on the GPU and compare everything with the oracle."""
    wd = w.to(dev)
    out = gpu_decode(wd, scale=scale, **kw)
    torch.cuda.synchronize()
    ref_state, ref_out = oracle_decode(w, scale=scale)
    got_state, got_out = f64(wd.state), f64(out)
    idx = w.state_indices.numpy().astype(np.int64)
    active = (idx >= 0) & (idx < w.N)
    assert (got_out[~active] == 0).all(), "inactive rows must give exactly zero"
    assert_output_close(got_out, ref_out)
    slots = idx[active]
    assert_state_close(got_state[slots], ref_state[slots])
    untouched = np.setdiff1d(np.arange(w.N), slots)
    assert np.array_equal(got_state[untouched], f64(w.state)[untouched]), "untouched slots changed"
    return wd, out


@pytest.mark.parametrize("B", [1, 3, 13, 32])
@pytest.mark.parametrize("layout", ["separate", "packed", "fused"])
def test_decode_matches_oracle(dev, B, layout):
    w = workloads.decode_inputs(B, B + 5, seed=100 + B, layout=layout, inactive_frac=0.2 if B > 3 else 0.0)
    run_and_check(w, dev)


@pytest.mark.parametrize("H", [1, 3, 64])
@pytest.mark.parametrize("config", [0, 3])
def test_decode_other_head_counts(dev, H, config):
    """H from 1 to the largest the boundary accepts, on the smallest and the whole-head tile."""
    w = workloads.decode_inputs(3, 5, seed=120 + H, H=H, inactive_frac=0.0)
    run_and_check(w, dev, config_override=config)


def test_decode_large_batch_sampled(dev):
    """B = 2048 (24576 CTAs of the whole-head tile); 16 rows compared with the oracle, the
    inactive rule checked on every row."""
    w = workloads.decode_inputs(2048, 2112, seed=121, inactive_frac=0.05)
    wd = w.to(dev)
    out = gpu_decode(wd)
    torch.cuda.synchronize()
    idx = w.state_indices.numpy().astype(np.int64)
    active = (idx >= 0) & (idx < w.N)
    assert (f64(out)[~active] == 0).all()
    rows = np.sort(np.random.default_rng(5).choice(np.nonzero(active)[0], 16, replace=False))
    sub = w.select_rows(rows)
    ref_state, ref_out = oracle_decode(sub)
    assert_output_close(f64(out)[rows], ref_out)
    assert_state_close(f64(wd.state)[idx[rows]], ref_state[idx[rows]])


@pytest.mark.parametrize("config", range(4))
def test_every_config_gives_the_same_bits(dev, config):
    w = workloads.decode_inputs(9, 16, seed=7, layout="packed", inactive_frac=0.2)
    wd = w.to(dev)
    out = gpu_decode(wd, config_override=config)
    wd0 = w.to(dev)
    out0 = gpu_decode(wd0, config_override=3)
    torch.cuda.synchronize()
    assert torch.equal(out.view(torch.int16), out0.view(torch.int16))
    assert torch.equal(wd.state.view(torch.int16), wd0.state.view(torch.int16))
    if config == 0:
        run_and_check(w, dev, config_override=0)


def test_single_row_sixteen_steps(dev):
    """B = 1, pool of 4 slots, slot 2, 16 steps with fresh inputs every step.
    Every step is held, per element, to one oracle step from the GPU's own
    state before it; the oracle also runs its own chain from the first state,
    which the GPU's chain stays within the drift bound of."""
    state = workloads.decode_inputs(1, 4, seed=0).state
    ref = f64(state)  # the oracle's own chain
    gstate = state.to(dev)
    for step in range(16):
        w = workloads.decode_inputs(1, 4, seed=1000 + step, indices=[2])
        before = f64(gstate)[2:3]
        wd = w.to(dev)
        wd.state = gstate
        out = gpu_decode(wd)
        tf_state, tf_out = oracle_decode(with_state(w, before))
        assert_output_close(f64(out), tf_out, f"step {step} output")
        assert_state_close(f64(gstate)[2:3], tf_state, f"step {step} state")
        w.state = torch.from_numpy(ref).to(torch.bfloat16)  # bf16-exact
        ref, ref_out = oracle_decode(w)
        assert_output_close(f64(out), ref_out, f"step {step} output against the oracle's chain")
        assert_drift_close(f64(gstate)[2:3], ref[2:3], f"step {step} chains")
        assert np.array_equal(f64(gstate)[[0, 1, 3]], f64(state)[[0, 1, 3]])


def test_thirtytwo_rows_sixty_four_chained_steps(dev):
    """B = 32 packed rows, pool of 64, 64 chained steps. Every step is held, per
    element, to one oracle step from the GPU's own state before it; the oracle
    also runs its own chain (drift diagnostic: outputs within tolerance and the
    two chains within 2 bf16 ulps of the head scale at every step)."""
    w0 = workloads.decode_inputs(32, 64, seed=1, layout="packed")
    idx = w0.state_indices
    slots = idx.numpy().astype(np.int64)
    ref = f64(w0.state)
    gstate = w0.state.to(dev)
    worst_out, worst_ulps, worst_tf = 0.0, 0.0, 0.0
    for step in range(64):
        w = workloads.decode_inputs(32, 64, seed=2000 + step, layout="packed", indices=idx)
        before = f64(gstate)[slots]
        wd = w.to(dev)
        wd.state = gstate
        out = gpu_decode(wd)
        tf_state, tf_out = oracle_decode(with_state(w, before))
        assert_output_close(f64(out), tf_out, f"step {step} output")
        got = f64(gstate)
        assert_state_close(got[slots], tf_state, f"step {step} state")
        worst_tf = max(worst_tf, float(state_ulps(got[slots], tf_state).max()))
        w.state = torch.from_numpy(ref).to(torch.bfloat16)
        ref, ref_out = oracle_decode(w)
        worst_out = max(worst_out, output_excess(f64(out), ref_out))
        worst_ulps = max(worst_ulps, float(state_ulps(got, ref, floor=1.0).max()))
    print(f"64 chained steps at B = 32: worst step {worst_tf:.2f} bf16 ulps per element; chains "
          f"{worst_ulps:.2f} ulps of the head scale apart, outputs at {worst_out:.3f} x tolerance")
    assert worst_out <= 1.0, f"output error reached {worst_out:.3f} x tolerance over 64 steps"
    assert worst_ulps <= DRIFT_ULPS, f"the chains drifted {worst_ulps:.2f} bf16 ulps of the head scale apart"


def test_serving_batch_512_sampled(dev):
    """B = 512, pool of 640, q/k/v strided views of a [512, 4672] projection
    buffer, about 5% of rows inactive: every row checked for the inactive rule
    and untouched slots, 40 rows checked against the oracle."""
    w = workloads.decode_inputs(512, 640, seed=2, layout="fused", inactive_frac=0.05)
    assert w.qkv.shape == (512, 4672)
    wd = w.to(dev)
    out = gpu_decode(wd)
    torch.cuda.synchronize()
    idx = w.state_indices.numpy().astype(np.int64)
    active = (idx >= 0) & (idx < 640)
    assert 20 <= (~active).sum() <= 32
    got_out = f64(out)
    assert (got_out[~active] == 0).all()
    untouched = np.setdiff1d(np.arange(640), idx[active])
    assert np.array_equal(f64(wd.state)[untouched], f64(w.state)[untouched])
    rng = np.random.default_rng(0)
    rows = np.sort(rng.choice(np.nonzero(active)[0], 40, replace=False))
    ref_state, ref_out = oracle_decode(w.select_rows(rows))
    assert_output_close(got_out[rows], ref_out)
    assert_state_close(f64(wd.state)[idx[rows]], ref_state[idx[rows]])


def test_all_inactive_is_a_bitwise_no_op(dev):
    w = workloads.decode_inputs(6, 8, seed=3, indices=[-1, 8, 9, -7, 2 ** 31 - 1, -(2 ** 31)])
    wd = w.to(dev)
    before = wd.state.clone()
    out = gpu_decode(wd)
    torch.cuda.synchronize()
    assert torch.equal(wd.state.view(torch.int16), before.view(torch.int16))
    assert (out.float() == 0).all()


def test_empty_pool_and_empty_batch(dev):
    w = workloads.decode_inputs(4, 4, seed=4)
    wd = w.to(dev)
    empty = torch.empty((0, 12, 128, 128), dtype=torch.bfloat16, device=dev)
    out = kda.kda_decode(empty, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                         wd.A_log, wd.dt_bias)
    torch.cuda.synchronize()
    assert (out.float() == 0).all()
    w0 = workloads.decode_inputs(0, 4, seed=5)
    w0d = w0.to(dev)
    out0 = gpu_decode(w0d)
    assert out0.shape == (0, 12, 128)


def test_misaligned_state_uses_plain_loads_with_same_bits(dev):
    w = workloads.decode_inputs(5, 7, seed=6, inactive_frac=0.2)
    wd = w.to(dev)
    flat = torch.empty(7 * 12 * 128 * 128 + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[1:1 + 7 * 12 * 128 * 128].view(7, 12, 128, 128)  # 2-byte aligned only
    mis.copy_(wd.state)
    assert mis.data_ptr() % 16 == 2
    out_a = gpu_decode(wd)
    wd.state = mis
    out_b = gpu_decode(wd)
    torch.cuda.synchronize()
    ref = w.to(dev)
    gpu_decode(ref)
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(mis.view(torch.int16), ref.state.view(torch.int16))


def test_padded_pool_and_guard_slots(dev):
    """A pool with padding between slots, and sentinel-filled guard slots and
    guard output rows around the real ones: nothing outside the real rows moves."""
    w = workloads.decode_inputs(6, 10, seed=8, inactive_frac=0.34)
    wd = w.to(dev)
    slot = 12 * 128 * 128
    raw = torch.full((12, slot + 64), -7.0, dtype=torch.bfloat16, device=dev)  # slots 0 and 11 are guards
    pool = raw[1:11, :slot].view(10, 12, 128, 128)
    pool.copy_(wd.state)
    guard_before = raw.clone()
    out_raw = torch.full((8, 12, 128), 3.0, dtype=torch.bfloat16, device=dev)
    out = out_raw[1:7]
    wd.state = pool
    kda.kda_decode(pool, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log,
                   wd.dt_bias, out=out)
    torch.cuda.synchronize()
    keep = torch.ones_like(raw, dtype=torch.bool)
    keep[1:11, :slot] = False
    assert torch.equal(raw[keep].view(torch.int16), guard_before[keep].view(torch.int16))
    assert (out_raw[0].float() == 3).all() and (out_raw[7].float() == 3).all()
    ref_state, ref_out = oracle_decode(w)
    assert_output_close(f64(out), ref_out)
    idx = w.state_indices.numpy().astype(np.int64)
    act = idx[(idx >= 0) & (idx < 10)]
    assert_state_close(f64(pool)[act], ref_state[act])


def test_odd_strides_and_shifted_tensors(dev):
    """q/k/v/g/beta/out views with odd strides and 2-byte offsets (the pages'
    shifted-tensor tests): same results as contiguous copies."""
    w = workloads.decode_inputs(5, 9, seed=9)
    wd = w.to(dev)

    def shifted(t, pad):
        """A copy of t whose base is 2 bytes past a 16-byte boundary and whose
        rows are pad elements longer than the data (odd strides)."""
        d = t.shape[-1]
        flat = torch.zeros(t[..., 0].numel() * (d + pad) + 1, dtype=t.dtype, device=dev)
        v = flat[1:].view(t.shape[:-1] + (d + pad,))[..., :d]
        v.copy_(t)
        assert v.data_ptr() % 16 == 2 and v.stride(-2) % 2 == 1
        return v

    q, k, v, g = (shifted(x, 3) for x in (wd.q, wd.k, wd.v, wd.g_raw))
    beta_big = torch.zeros((5, 12, 3), dtype=torch.bfloat16, device=dev)
    beta = beta_big[:, :, 1]
    beta.copy_(wd.beta_logit)
    out_big = torch.zeros((5, 12, 131), dtype=torch.bfloat16, device=dev)
    out = out_big[:, :, 3:]
    st = wd.state.clone()
    kda.kda_decode(st, wd.state_indices, q, k, v, g, beta, wd.A_log, wd.dt_bias, out=out)
    out_ref = gpu_decode(wd)
    torch.cuda.synchronize()
    assert torch.equal(out.contiguous().view(torch.int16), out_ref.view(torch.int16))
    assert torch.equal(st.view(torch.int16), wd.state.view(torch.int16))
    assert (out_big[:, :, :3].float() == 0).all()


def test_special_values(dev):
    """beta = 0 with decay 1 leaves the state bitwise unchanged; decay 1 with
    beta = 1 maps k_hat onto v (S^T k_hat = v up to bf16 rounding)."""
    w = workloads.decode_inputs(3, 5, seed=10)
    w.beta_logit[:] = float("-inf")
    w.g_raw[:] = float("-inf")
    wd, out = run_and_check(w, dev)
    idx = w.state_indices.long()
    assert torch.equal(wd.state.cpu()[idx].view(torch.int16), w.state[idx].view(torch.int16))
    w2 = workloads.decode_inputs(3, 5, seed=11)
    w2.beta_logit[:] = float("inf")
    w2.g_raw[:] = float("-inf")
    wd2, _ = run_and_check(w2, dev)
    S = f64(wd2.state)[w2.state_indices.numpy()]  # [B, H, V, K]
    kh = f64(w2.k) / np.sqrt((f64(w2.k) ** 2).sum(-1, keepdims=True) + 1e-6)
    back = np.einsum("bhvk,bhk->bhv", S, kh)
    assert np.abs(back - f64(w2.v)).max() < 0.05


def test_output_scale(dev):
    w = workloads.decode_inputs(4, 6, seed=12)
    run_and_check(w, dev, scale=0.0883883)


def test_cuda_graph_replay_is_deterministic_and_tracks_inputs(dev):
    w = workloads.decode_inputs(8, 12, seed=13, layout="packed", inactive_frac=0.25)
    wd = w.to(dev)
    init = wd.state.clone()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        gpu_decode(wd)  # warm-up outside capture
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    wd.state.copy_(init)
    out = torch.empty((8, 12, 128), dtype=torch.bfloat16, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_decode(wd, out=out)
    results = []
    for _ in range(2):
        wd.state.copy_(init)
        graph.replay()
        torch.cuda.synchronize()
        results.append((out.clone(), wd.state.clone()))
    assert torch.equal(results[0][0].view(torch.int16), results[1][0].view(torch.int16))
    assert torch.equal(results[0][1].view(torch.int16), results[1][1].view(torch.int16))
    # new inputs and new indices copied into the captured buffers
    w2 = workloads.decode_inputs(8, 12, seed=14, layout="packed", inactive_frac=0.25)
    w2.state, w2.A_log, w2.dt_bias = w.state, w.A_log, w.dt_bias  # not re-copied into the graph
    for name in ("qkv", "g_raw", "beta_logit", "state_indices"):
        getattr(wd, name).copy_(getattr(w2, name).to(dev))
    wd.state.copy_(init)
    graph.replay()
    torch.cuda.synchronize()
    ref_state, ref_out = oracle_decode(w2)
    assert_output_close(f64(out), ref_out)
    idx = w2.state_indices.numpy().astype(np.int64)
    act = idx[(idx >= 0) & (idx < 12)]
    assert_state_close(f64(wd.state)[act], ref_state[act])


def test_runs_on_the_callers_stream(dev):
    w = workloads.decode_inputs(4, 6, seed=15)
    wd = w.to(dev)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        torch.cuda._sleep(2_000_000)  # keep the side stream busy; the call must queue behind it
        out = gpu_decode(wd)
    s.synchronize()
    ref_state, ref_out = oracle_decode(w)
    assert_output_close(f64(out), ref_out)


def test_error_word_stays_clear(dev):
    w = workloads.decode_inputs(4, 6, seed=16)
    wd = w.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    gpu_decode(wd, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == 0


@pytest.mark.parametrize("B", [3, 32])
def test_precomputed_gate_convention(dev, B):
    """Log-space g and beta given directly (the API-default convention of the
    pages' recurrent_kda); A_log and dt_bias are not passed."""
    w = workloads.decode_inputs(B, B + 4, seed=40 + B, layout="packed", inactive_frac=0.2, gate_mode=1)
    w.A_log = w.dt_bias = None
    run_and_check(w, dev)


def test_prepared_decode_equals_direct_call(dev):
    """kda.prepare_decode binds the tensors once; each call runs on their
    current contents and gives the bits of a direct kda_decode."""
    w = workloads.decode_inputs(8, 12, seed=130, layout="fused", inactive_frac=0.25)
    wa, wb = w.to(dev), w.to(dev)
    call = kda.prepare_decode(wa.state, wa.state_indices, wa.q, wa.k, wa.v, wa.g_raw, wa.beta_logit, wa.A_log,
                              wa.dt_bias)
    w2 = workloads.decode_inputs(8, 12, seed=131, layout="fused", inactive_frac=0.25)
    for step in range(3):  # refill the bound inputs between calls, as a serving loop does
        src = (w if step % 2 == 0 else w2).to(dev)
        for name in ("qkv", "g_raw", "beta_logit"):
            getattr(wa, name).copy_(getattr(src, name))
            getattr(wb, name).copy_(getattr(src, name))
        out_a = call()
        out_b = kda.kda_decode(wb.state, wb.state_indices, wb.q, wb.k, wb.v, wb.g_raw, wb.beta_logit, wb.A_log,
                               wb.dt_bias)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b) and torch.equal(wa.state, wb.state)


def test_long_chain_drift_diagnostic(dev):
    """512 chained decode steps at B = 1 (the pages' long-run drift diagnostic):
    GPU and oracle each run their own chain; outputs stay within tolerance at
    every step and the state within 2 bf16 ulps of the head scale (no drift:
    the worst seen was 1 ulp, outputs at 0.04 of the tolerance). The worst
    drift seen is printed."""
    ref = f64(workloads.decode_inputs(1, 4, seed=3000, indices=[1]).state)
    gstate = torch.from_numpy(ref).to(torch.bfloat16).to(dev)
    worst_out, worst_ulps, at = 0.0, 0.0, 0
    for step in range(512):
        w = workloads.decode_inputs(1, 4, seed=3001 + step, indices=[1])
        w.state = torch.from_numpy(ref).to(torch.bfloat16)
        wd = w.to(dev)
        wd.state = gstate
        out = gpu_decode(wd)
        ref, ref_out = oracle_decode(w)
        worst_out = max(worst_out, output_excess(f64(out), ref_out))
        u = float(state_ulps(f64(gstate)[1:2], ref[1:2], floor=1.0).max())
        if u > worst_ulps:
            worst_ulps, at = u, step
    print(f"512-step drift: worst output {worst_out:.3f} x tolerance, worst state {worst_ulps:.2f} bf16 ulps "
          f"of the head scale (step {at})")
    assert worst_out <= 1.0
    assert worst_ulps <= DRIFT_ULPS_512
