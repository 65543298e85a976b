"""kda_prefill_ws in its two-stage configurations (5: the preparation kernel,
then the chain kernel; 6: both in one cooperative launch, the chains waiting
for each chunk's ready flag; both with a caller's workspace) on the GPU against
the fp64 prefill oracle, through the C ABI, with the tolerances of
test_prefill_gpu (outputs 2e-2 + 2e-2 |o_ref|; final states 2 bf16 ulps at
max(|s_ref|, F_L M)); against the single-kernel configurations, which compute
the same reading with other fp32 rounding; and 6 against 5, bit for bit.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import assert_output_close, assert_prefill_state_close, assert_state_close, f64
from linear_attention_ssm_step_gb300 import kda, workloads
from test_prefill_gpu import LB, LENGTHS, SENTINEL, check_prefill, gpu_prefill

pytestmark = pytest.mark.gpu

CHAIN = 5
FUSED = 6
BOTH = pytest.mark.parametrize("cfg", [CHAIN, FUSED])


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def workspace_for(wd):
    return kda.prefill_workspace(wd.q.shape[0], wd.cu_seqlens.shape[0] - 1, wd.H, wd.q.device)


def chain_prefill(wd, out=None, workspace=None, cfg=CHAIN, **kw):
    if workspace is None:
        workspace = workspace_for(wd)
    kw.setdefault("config_override", cfg)
    return gpu_prefill(wd, out=out, workspace=workspace, **kw)


@pytest.mark.parametrize("cfg,H", [(CHAIN, 12), (FUSED, 4)])
def test_chain_matches_oracle(dev, cfg, H):
    w = workloads.prefill_inputs(LENGTHS, 12, seed=170, inactive_frac=0.25, layout="fused", H=H)
    wd = w.to(dev)
    out = chain_prefill(wd, cfg=cfg)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


@BOTH
def test_chain_precomputed_gate_and_scale(dev, cfg):
    w = workloads.prefill_inputs([7, 20, 1], 5, seed=171, gate_mode=1)
    wd = w.to(dev)
    out = chain_prefill(wd, cfg=cfg, scale=0.5)
    torch.cuda.synchronize()
    check_prefill(w, wd, out, scale=0.5)


@BOTH
def test_chain_three_heads_packed(dev, cfg):
    w = workloads.prefill_inputs([9, 3, 25], 6, seed=172, H=3, layout="packed")
    wd = w.to(dev)
    out = chain_prefill(wd, cfg=cfg)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


@BOTH
def test_chain_long_sequence(dev, cfg):
    """One 1000-token sequence (63 chunks, prepared by many CTAs) and two short ones."""
    w = workloads.prefill_inputs([1000, 3, 12], 4, seed=173)
    wd = w.to(dev)
    out = chain_prefill(wd, cfg=cfg)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


@BOTH
@pytest.mark.parametrize("lengths", [[15, 16, 17], [31, 32, 33, 48], [47, 64, 1, 2]])
def test_chain_chunk_boundaries(dev, lengths, cfg):
    w = workloads.prefill_inputs(lengths, len(lengths) + 3, seed=185 + sum(lengths))
    wd = w.to(dev)
    out = chain_prefill(wd, cfg=cfg)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


def test_one_launch_equals_two_launches(dev):
    """Configurations 6 and 5 run the same arithmetic: the same bits, here on
    two long sequences (250 and 44 chunks) at H = 8."""
    w = workloads.prefill_inputs([4000, 700], 3, seed=188, H=8)
    a, b = w.to(dev), w.to(dev)
    oa = chain_prefill(a, cfg=FUSED)
    ob = chain_prefill(b, cfg=CHAIN)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_one_launch_conditions(dev):
    """Configuration 6 asked for outside its conditions (too many chains;
    token rows not 16-byte aligned) is refused; the library's own choice then
    falls back to configuration 5 (the same bits)."""
    w = workloads.prefill_inputs([600] * 8, 9, seed=189, H=12)  # 96 chains: more than half the SMs
    wd = w.to(dev)
    with pytest.raises(kda.KdaError) as e:
        chain_prefill(wd, cfg=FUSED)
    assert e.value.status == kda.KDA_EUNSUPPORTED
    w = workloads.prefill_inputs([1200, 40], 3, seed=190, H=4)  # 620 tokens per sequence: the library picks 6
    assert kda.kda_select_prefill_ws_config(1240, 2, 4) == FUSED
    a, b = w.to(dev), w.to(dev)
    wide = torch.zeros((b.q.shape[0], 4, 136), dtype=torch.bfloat16, device=dev)
    wide[:, :, 1:129].copy_(b.q)
    q_off = wide[:, :, 1:129]  # rows 2 bytes past a 16-byte boundary
    assert q_off.data_ptr() % 16 == 2

    def call_b(cfg):
        out = torch.empty((b.q.shape[0], 4, 128), dtype=torch.bfloat16, device=dev)
        return kda.kda_prefill(b.state, b.state_indices, b.cu_seqlens, q_off, b.k, b.v, b.g_raw, b.beta_logit,
                               b.A_log, b.dt_bias, out=out, lower_bound=LB, gate_mode=b.gate_mode,
                               config_override=cfg, workspace=workspace_for(b))

    with pytest.raises(kda.KdaError) as e:
        call_b(FUSED)
    assert e.value.status == kda.KDA_EUNSUPPORTED
    ob = call_b(-1)  # the library's choice (6) falls back to 5
    oa = chain_prefill(a, cfg=CHAIN)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_chain_one_token_sequences_match_decode(dev):
    """One-token sequences: one decode step per slot, to the single-step bound."""
    B = 37
    w = workloads.prefill_inputs([1] * B, B + 20, seed=174, inactive_frac=0.1, layout="fused")
    a, b = w.to(dev), w.to(dev)
    out_p = chain_prefill(a)
    out_d = kda.kda_decode(b.state, b.state_indices, b.q, b.k, b.v, b.g_raw, b.beta_logit, b.A_log, b.dt_bias,
                           lower_bound=LB)
    torch.cuda.synchronize()
    idx = w.state_indices.numpy().astype(np.int64)
    act = idx[(idx >= 0) & (idx < w.N)]
    assert_output_close(f64(out_p), f64(out_d))
    assert_state_close(f64(a.state)[act], f64(b.state)[act], "two-stage one-token prefill against a decode step")
    check_prefill(w, a, out_p)


@BOTH
def test_chain_against_single_kernel_configs(dev, cfg):
    """Against the chunked single kernel (4) and the token-by-token one (2):
    outputs within the output tolerance, states within the prefill bound."""
    lens = [300, 7, 64, 129, 16]
    w = workloads.prefill_inputs(lens, 8, seed=186, layout="packed")
    a = w.to(dev)
    oa = chain_prefill(a, cfg=cfg)
    torch.cuda.synchronize()
    for config in (4, 2):
        b = w.to(dev)
        ob = gpu_prefill(b, config_override=config)
        torch.cuda.synchronize()
        assert_output_close(f64(oa), f64(ob))
        for i, n in enumerate(w.state_indices.tolist()):
            assert_prefill_state_close(f64(a.state)[n], f64(b.state)[n], lens[i], f"sequence {i}, config {config}")


def test_chain_many_items_per_cta(dev):
    """More (sequence, head) items than the chain's grid has CTAs (one per SM),
    with mixed lengths and inactive sequences: 400 sequences of 0..60 tokens at H = 4."""
    rng = np.random.default_rng(187)
    lens = [int(x) for x in rng.integers(0, 61, 400)]
    w = workloads.prefill_inputs(lens, 420, seed=187, H=4, inactive_frac=0.1)
    wd = w.to(dev)
    out = chain_prefill(wd)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


@BOTH
def test_chain_misaligned_pool_same_bits(dev, cfg):
    """A 2-byte aligned pool takes plain loads and stores: the same bits."""
    w = workloads.prefill_inputs([6, 21, 40], 4, seed=176)
    a, b = w.to(dev), w.to(dev)
    flat = torch.empty(b.state.numel() + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[1:1 + b.state.numel()].view(b.state.shape)
    mis.copy_(b.state)
    assert mis.data_ptr() % 16 == 2
    b.state = mis
    oa, ob = chain_prefill(a, cfg=cfg), chain_prefill(b, cfg=cfg)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


@BOTH
def test_chain_bad_bounds_set_the_error_bit(dev, cfg):
    """Sequences with bad bounds are skipped and flagged; the valid ones keep
    their own chunk images even when a bad sequence sits between two valid
    ones whose rows come out of order (rows 32..47, then 0..31)."""
    w = workloads.prefill_inputs([5, 4, 6], 6, seed=177)
    w.cu_seqlens = torch.tensor([0, 5, 9, 3], dtype=torch.int32)  # sequence 2 runs backwards
    wd = w.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = chain_prefill(wd, cfg=cfg, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda.KDA_ERR_SEQLENS
    check_prefill(w, wd, out, err_expected=oracle.PREFILL_ERR_SEQLENS)

    w = workloads.prefill_inputs([16, 16, 16], 6, seed=178)
    w.cu_seqlens = torch.tensor([32, 48, 0, 32], dtype=torch.int32)
    wd = w.to(dev)
    err.zero_()
    out = chain_prefill(wd, cfg=cfg, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda.KDA_ERR_SEQLENS
    check_prefill(w, wd, out, err_expected=oracle.PREFILL_ERR_SEQLENS)


@BOTH
def test_chain_graph_replays_are_identical(dev, cfg):
    w = workloads.prefill_inputs([12, 1, 90], 5, seed=178)
    wd = w.to(dev)
    st0 = wd.state.clone()
    ws = workspace_for(wd)
    out = torch.empty((wd.q.shape[0], 12, 128), dtype=torch.bfloat16, device=dev)
    fn = lambda: chain_prefill(wd, out=out, workspace=ws, cfg=cfg)  # noqa: E731
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fn()
    res = []
    for _ in range(3):
        wd.state.copy_(st0)
        g.replay()
        torch.cuda.synchronize()
        res.append((out.view(torch.int16).clone(), wd.state.view(torch.int16).clone()))
    for o, s in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(s, res[0][1])


@BOTH
def test_chain_workspace_contents_do_not_matter(dev, cfg):
    """A workspace full of garbage, and one reused from a different call, give the same bits."""
    w = workloads.prefill_inputs([33, 70], 3, seed=179)
    a, b = w.to(dev), w.to(dev)
    ws = workspace_for(a)
    ws.fill_(0xFF)
    oa = chain_prefill(a, workspace=ws, cfg=cfg)
    ws.random_(0, 256)
    ob = chain_prefill(b, workspace=ws, cfg=cfg)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_chain_empty_calls(dev):
    """Three empty sequences, and no sequence at all: nothing is written."""
    w = workloads.prefill_inputs([0, 0, 0], 4, seed=179)
    wd = w.to(dev)
    st0 = wd.state.clone()
    out = torch.full((wd.q.shape[0], 12, 128), SENTINEL, dtype=torch.bfloat16, device=dev)
    chain_prefill(wd, out=out)
    w2 = workloads.prefill_inputs([4, 0, 2], 4, seed=180)
    wd2 = w2.to(dev)
    cu0 = torch.zeros(1, dtype=torch.int32, device=dev)
    idx0 = torch.zeros(0, dtype=torch.int32, device=dev)
    o2 = torch.full((6, 12, 128), SENTINEL, dtype=torch.bfloat16, device=dev)
    kda.kda_prefill(wd2.state, idx0, cu0, wd2.q, wd2.k, wd2.v, wd2.g_raw, wd2.beta_logit, wd2.A_log, wd2.dt_bias,
                    out=o2, config_override=CHAIN, workspace=torch.empty(0, dtype=torch.uint8, device=dev))
    torch.cuda.synchronize()
    assert torch.equal(wd.state, st0)
    assert torch.all(o2.float() == SENTINEL), "no sequence: nothing written"
    assert torch.equal(wd2.state, w2.state.to(dev))


def test_chain_rejects_bad_workspaces(dev):
    w = workloads.prefill_inputs([3, 40], 4, seed=181)
    wd = w.to(dev)
    need = kda.prefill_workspace_bytes(wd.q.shape[0], 2, wd.H)
    images = ((43 + 15) // 16 + 2) * 12
    assert need == images * 45568 + (images * 4 + 15) // 16 * 16
    with pytest.raises(kda.KdaError) as e:  # configuration 5 without a workspace
        gpu_prefill(wd, config_override=CHAIN)
    assert e.value.status == kda.KDA_EINVAL
    small = torch.empty(need - 16, dtype=torch.uint8, device=dev)
    with pytest.raises(kda.KdaError) as e:
        chain_prefill(wd, workspace=small)
    assert e.value.status == kda.KDA_EINVAL and "workspace" in str(e.value)
    big = torch.empty(need + 64, dtype=torch.uint8, device=dev)
    with pytest.raises(kda.KdaError) as e:  # not 16-byte aligned
        chain_prefill(wd, workspace=big[1:1 + need])
    assert e.value.status == kda.KDA_EINVAL
    out = torch.empty((wd.q.shape[0], 12, 128), dtype=torch.bfloat16, device=dev)
    ov = torch.empty(need + out.numel() * 2, dtype=torch.uint8, device=dev)
    out_in_ws = ov[:out.numel() * 2].view(torch.bfloat16).view(out.shape)
    with pytest.raises(kda.KdaError) as e:  # overlapping the output
        chain_prefill(wd, out=out_in_ws, workspace=ov[:need])
    assert e.value.status == kda.KDA_EINVAL and "overlaps" in str(e.value)


def test_chain_selector(dev):
    assert kda.kda_select_prefill_ws_config(4096, 1, 12) == FUSED
    assert kda.kda_select_prefill_ws_config(8 * 2048, 8, 12) == CHAIN
    assert kda.kda_select_prefill_ws_config(512 * 16, 512, 12) == 4
    assert kda.kda_select_prefill_ws_config(64 * 256, 64, 12) == 4
    w = workloads.prefill_inputs([700, 400], 3, seed=182)
    a, b = w.to(dev), w.to(dev)
    oa = chain_prefill(a, cfg=-1)
    ob = chain_prefill(b, cfg=FUSED)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16)), "the library's choice is configuration 6"


def test_chain_bench_shape_1x4096_full(dev):
    """The bench's 1 x 4096 shape (H = 12) in its launch configuration: every
    output and the final state against the oracle."""
    w = workloads.prefill_inputs([4096], 9, seed=91, layout="fused")
    wd = w.to(dev)
    out = chain_prefill(wd, config_override=-1)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


@pytest.mark.parametrize("S,L", [(8, 2048), (64, 256)])
def test_chain_bench_shapes_sampled(dev, S, L):
    """The bench's multi-sequence shapes in the two-stage configuration:
    sampled sequences against the oracle, every other slot untouched and every
    row written."""
    w = workloads.prefill_inputs([L] * S, S + 8, seed=90 + S, layout="fused")
    wd = w.to(dev)
    out = chain_prefill(wd)
    torch.cuda.synchronize()
    got_out, got_state = f64(out), f64(wd.state)
    assert np.all(got_out != SENTINEL), "every row belongs to a sequence"
    rng = np.random.default_rng(S)
    for i in rng.choice(S, size=2 if L > 1000 else 6, replace=False):
        rows = slice(i * L, (i + 1) * L)
        n = int(w.state_indices[i])
        ref_state, ref_out, _, err = oracle.kda_prefill(
            f64(w.state[n:n + 1]), np.array([0]), np.array([0, L]), f64(w.q[rows]), f64(w.k[rows]),
            f64(w.v[rows]), f64(w.g_raw[rows]), f64(w.beta_logit[rows]), f64(w.A_log), f64(w.dt_bias),
            lower_bound=LB)
        assert err == 0
        assert_output_close(got_out[rows], ref_out, f"outputs of sequence {i}")
        assert_prefill_state_close(got_state[n], ref_state[0], L, f"final state of sequence {i}")
    owned = set(int(x) for x in w.state_indices)
    rest = [n for n in range(w.N) if n not in owned]
    assert np.array_equal(got_state[rest], f64(w.state)[rest])


def test_chain_h16_16384_against_chunked_kernel(dev):
    """The pages' H16 x 16384-token shape: the two-stage path against the
    single-kernel chunked one on every output and the final state (both
    carry fp32 states; outputs within the output tolerance of each other,
    states within the prefill bound)."""
    w = workloads.prefill_inputs([16384], 2, seed=96, layout="fused", H=16)
    a, b = w.to(dev), w.to(dev)
    oa = chain_prefill(a, config_override=-1)
    ob = gpu_prefill(b, config_override=4)
    torch.cuda.synchronize()
    assert_output_close(f64(oa), f64(ob), "two-stage against chunked outputs")
    n = int(w.state_indices[0])
    assert_prefill_state_close(f64(a.state)[n], f64(b.state)[n], 16384, "final state")


def test_chain_h16_16384_sampled_heads_against_oracle(dev):
    """The pages' H16 x 16384-token shape in the library's launch
    configuration (one launch, two stages): two sampled heads' outputs for
    every token and their final states against the oracle (heads are
    independent; the oracle runs those two alone)."""
    L = 16384
    w = workloads.prefill_inputs([L], 2, seed=96, layout="fused", H=16)
    wd = w.to(dev)
    assert kda.kda_select_prefill_ws_config(L, 1, 16) == FUSED
    out = chain_prefill(wd, config_override=-1)
    torch.cuda.synchronize()
    got_out, got_state = f64(out), f64(wd.state)
    n = int(w.state_indices[0])
    for h in (3, 12):
        hs = slice(h, h + 1)
        ref_state, ref_out, _, err = oracle.kda_prefill(
            f64(w.state[n:n + 1, hs]), np.array([0]), np.array([0, L]), f64(w.q[:, hs]), f64(w.k[:, hs]),
            f64(w.v[:, hs]), f64(w.g_raw[:, hs]), f64(w.beta_logit[:, hs]), f64(w.A_log[hs]),
            f64(w.dt_bias[hs]), lower_bound=LB)
        assert err == 0
        assert_output_close(got_out[:, hs], ref_out, f"outputs of head {h}")
        assert_prefill_state_close(got_state[n, hs], ref_state[0], L, f"final state of head {h}")
