"""kda_prefill (varlen prefill on the bf16 pool) on the GPU against the fp64
prefill oracle, through the C ABI.

What is compared:
  * outputs: the decode's tolerance, 2e-2 + 2e-2 |o_ref|;
  * final states: one-token sequences are one decode step, held to the
    single-step bound (2 bf16 ulps at max(|s_ref|, 2^-12 M)); an L-token one
    to 2 bf16 ulps at max(|s_ref|, F_L M), F_L = max(2^-12, L 2^-11) up to 1.
    The kernel carries the state in fp32 across the tokens and the oracle in
    fp64: their difference grows by at most about 2^-19 M per token (the step
    map is non-expansive), and the final rounding to bf16 can fall on either
    side of a boundary (harness module docstring);
  * rows of inactive sequences: exactly zero; rows no valid sequence covers
    and slots no active sequence owns: bit for bit unchanged;
  * one-token sequences against kda_decode on the same rows: bit for bit on
    the CUDA cores (configurations 0-3), to the single-step bound in the
    chunked tensor-core configuration (4, the default), whose products round
    differently;
  * the chunked kernel at chunk boundaries, against the token-by-token one,
    and with more (sequence, head) items than its persistent grid has CTAs.
"""

import numpy as np
import pytest
import torch

import oracle
from harness import assert_output_close, assert_prefill_state_close, assert_state_close, f64
from linear_attention_ssm_step_gb300 import kda, workloads

pytestmark = pytest.mark.gpu

LB = -5.0
SENTINEL = 7.0  # written into out before a call: rows the call must not touch keep it


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def gpu_prefill(wd, out=None, **kw):
    kw.setdefault("gate_mode", wd.gate_mode)
    if out is None:
        out = torch.full((wd.q.shape[0], wd.H, 128), SENTINEL, dtype=torch.bfloat16, device=wd.q.device)
    return kda.kda_prefill(wd.state, wd.state_indices, wd.cu_seqlens, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                           wd.A_log, wd.dt_bias, out=out, lower_bound=LB, **kw)


def oracle_prefill(w, scale=1.0):
    return oracle.kda_prefill(f64(w.state), f64(w.state_indices), f64(w.cu_seqlens), f64(w.q), f64(w.k), f64(w.v),
                              f64(w.g_raw), f64(w.beta_logit), f64(w.A_log), f64(w.dt_bias),
                              lower_bound=LB, scale=scale, gate_mode=w.gate_mode)


def check_prefill(w, wd, out, scale=1.0, err_expected=0):
    new_ref, out_ref, written, err = oracle_prefill(w, scale)
    assert err == err_expected
    got = f64(out)
    assert_output_close(got[written], out_ref[written], "outputs")
    assert np.all(got[~written] == SENTINEL), "rows no sequence covers must keep their contents"
    st = f64(wd.state)
    st0 = f64(w.state)
    idx = w.state_indices.tolist()
    cu = w.cu_seqlens.tolist()
    owned = set()
    for i, n in enumerate(idx):
        t0, t1 = cu[i], cu[i + 1]
        if not (0 <= n < w.N) or not (0 <= t0 <= t1 <= w.q.shape[0]) or t0 == t1:
            continue
        owned.add(n)
        assert_prefill_state_close(st[n], new_ref[n], t1 - t0, f"final state of sequence {i} ({t1 - t0} tokens)")
    for i, n in enumerate(idx):
        t0, t1 = cu[i], cu[i + 1]
        if not (0 <= n < w.N) and 0 <= t0 <= t1 <= w.q.shape[0]:
            assert np.all(got[t0:t1] == 0.0), f"inactive sequence {i} must write zeros"
    rest = [n for n in range(w.N) if n not in owned]
    assert np.array_equal(st[rest], st0[rest]), "slots no active sequence owns must be untouched"


LENGTHS = [1, 17, 0, 40, 5, 16, 33, 2]


@pytest.mark.parametrize("config", [-1, 0, 1, 2, 3, 4])
def test_prefill_matches_oracle(dev, config):
    w = workloads.prefill_inputs(LENGTHS, 12, seed=70 + config, inactive_frac=0.25, layout="fused")
    wd = w.to(dev)
    out = gpu_prefill(wd, config_override=config)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


def test_prefill_precomputed_gate_and_scale(dev):
    w = workloads.prefill_inputs([7, 20, 1], 5, seed=71, gate_mode=1)
    wd = w.to(dev)
    out = gpu_prefill(wd, scale=0.5)
    torch.cuda.synchronize()
    check_prefill(w, wd, out, scale=0.5)


def test_prefill_three_heads_packed(dev):
    w = workloads.prefill_inputs([9, 3, 25], 6, seed=72, H=3, layout="packed")
    wd = w.to(dev)
    out = gpu_prefill(wd)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


def test_prefill_long_sequence(dev):
    """One 1000-token sequence and two short ones; every output and both states."""
    w = workloads.prefill_inputs([1000, 3, 12], 4, seed=73)
    wd = w.to(dev)
    out = gpu_prefill(wd)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


@pytest.mark.parametrize("config", [0, 2, 3])
def test_single_token_sequences_equal_decode_bit_for_bit(dev, config):
    """On the CUDA cores (configurations 0-3) a prefill of one-token sequences
    is one decode step per slot, bit for bit."""
    B = 37
    w = workloads.prefill_inputs([1] * B, B + 20, seed=74, inactive_frac=0.1, layout="fused")
    a, b = w.to(dev), w.to(dev)
    out_p = gpu_prefill(a, config_override=config)
    out_d = kda.kda_decode(b.state, b.state_indices, b.q, b.k, b.v, b.g_raw, b.beta_logit, b.A_log, b.dt_bias,
                           lower_bound=LB)
    torch.cuda.synchronize()
    assert torch.equal(out_p.view(torch.int16), out_d.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_single_token_sequences_chunked_match_decode(dev):
    """The chunked tensor-core kernel on one-token sequences: one decode step
    per slot to the single-step bound (its products round differently), and
    against the oracle."""
    B = 37
    w = workloads.prefill_inputs([1] * B, B + 20, seed=74, inactive_frac=0.1, layout="fused")
    a, b = w.to(dev), w.to(dev)
    out_p = gpu_prefill(a, config_override=4)
    out_d = kda.kda_decode(b.state, b.state_indices, b.q, b.k, b.v, b.g_raw, b.beta_logit, b.A_log, b.dt_bias,
                           lower_bound=LB)
    torch.cuda.synchronize()
    idx = w.state_indices.numpy().astype(np.int64)
    act = idx[(idx >= 0) & (idx < w.N)]
    assert_output_close(f64(out_p), f64(out_d))
    assert_state_close(f64(a.state)[act], f64(b.state)[act], "chunked one-token prefill against a decode step")
    check_prefill(w, a, out_p)


@pytest.mark.parametrize("lengths", [[15, 16, 17], [31, 32, 33, 48], [47, 64, 1, 2]])
def test_prefill_chunk_boundaries(dev, lengths):
    """Sequences that end just before, on and just after a 16-token chunk
    boundary, in the chunked kernel and in the token-by-token one."""
    for config in (4, 2):
        w = workloads.prefill_inputs(lengths, len(lengths) + 3, seed=85 + sum(lengths) + config)
        wd = w.to(dev)
        out = gpu_prefill(wd, config_override=config)
        torch.cuda.synchronize()
        check_prefill(w, wd, out)


def test_prefill_chunked_against_token_by_token(dev):
    """The two kernels compute the same reading with different fp32 rounding:
    their outputs within the output tolerance of each other and their states
    within the prefill bound."""
    lens = [200, 7, 64, 129]
    w = workloads.prefill_inputs(lens, 8, seed=86, layout="packed")
    a, b = w.to(dev), w.to(dev)
    oa = gpu_prefill(a, config_override=4)
    ob = gpu_prefill(b, config_override=2)
    torch.cuda.synchronize()
    assert_output_close(f64(oa), f64(ob))
    for i, n in enumerate(w.state_indices.tolist()):
        assert_prefill_state_close(f64(a.state)[n], f64(b.state)[n], lens[i], f"sequence {i}")


def test_prefill_many_sequences_per_cta(dev):
    """More (sequence, head) items than the persistent grid has CTAs, with mixed
    lengths and inactive sequences: 400 sequences of 0..40 tokens at H = 4."""
    rng = np.random.default_rng(87)
    lens = [int(x) for x in rng.integers(0, 41, 400)]
    w = workloads.prefill_inputs(lens, 420, seed=87, H=4, inactive_frac=0.1)
    wd = w.to(dev)
    out = gpu_prefill(wd)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


def test_prefill_configs_agree_bit_for_bit(dev):
    """The tile size changes only which CTA runs a row, not its arithmetic."""
    w = workloads.prefill_inputs([5, 30, 18], 5, seed=75)
    res = []
    for config in (0, 1, 2, 3):
        wd = w.to(dev)
        out = gpu_prefill(wd, config_override=config)
        torch.cuda.synchronize()
        res.append((out.view(torch.int16).clone(), wd.state.view(torch.int16).clone()))
    for o, s in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(s, res[0][1])


@pytest.mark.parametrize("config", [2, 4])
def test_prefill_misaligned_pool_same_bits(dev, config):
    """A 2-byte aligned pool takes plain loads and stores: the same bits."""
    w = workloads.prefill_inputs([6, 21], 4, seed=76)
    a, b = w.to(dev), w.to(dev)
    flat = torch.empty(b.state.numel() + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[1:1 + b.state.numel()].view(b.state.shape)
    mis.copy_(b.state)
    assert mis.data_ptr() % 16 == 2
    b.state = mis
    oa, ob = gpu_prefill(a, config_override=config), gpu_prefill(b, config_override=config)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_prefill_misaligned_token_views_same_bits(dev):
    """Token views off a 16-byte boundary take per-lane loads in place of the
    chunked kernel's tensor-map copies of the token rows: the same bits."""
    w = workloads.prefill_inputs([6, 40, 17], 5, seed=78)
    a, b = w.to(dev), w.to(dev)

    def shifted(x):
        flat = torch.empty(x.numel() + 8, dtype=x.dtype, device=dev)
        y = flat[1:1 + x.numel()].view(x.shape)
        y.copy_(x)
        return y

    b.q_sep, b.k_sep, b.v_sep, b.g_raw = (shifted(x) for x in (b.q_sep, b.k_sep, b.v_sep, b.g_raw))
    assert b.q_sep.data_ptr() % 16 == 2
    oa, ob = gpu_prefill(a, config_override=4), gpu_prefill(b, config_override=4)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_prefill_bad_bounds_set_the_error_bit(dev):
    w = workloads.prefill_inputs([5, 4, 6], 6, seed=77)
    w.cu_seqlens = torch.tensor([0, 5, 9, 3], dtype=torch.int32)  # sequence 2 runs backwards
    wd = w.to(dev)
    err = torch.zeros(1, dtype=torch.int32, device=dev)
    out = gpu_prefill(wd, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda.KDA_ERR_SEQLENS
    check_prefill(w, wd, out, err_expected=oracle.PREFILL_ERR_SEQLENS)
    w.cu_seqlens = torch.tensor([0, 5, 9, 16], dtype=torch.int32)  # sequence 2 ends past the last row
    wd = w.to(dev)
    err.zero_()
    out = gpu_prefill(wd, error_word=err)
    torch.cuda.synchronize()
    assert int(err.item()) == kda.KDA_ERR_SEQLENS
    check_prefill(w, wd, out, err_expected=oracle.PREFILL_ERR_SEQLENS)


def test_prefill_graph_replays_are_identical(dev):
    w = workloads.prefill_inputs([12, 1, 30], 5, seed=78)
    wd = w.to(dev)
    st0 = wd.state.clone()
    out = torch.empty((wd.q.shape[0], 12, 128), dtype=torch.bfloat16, device=dev)
    fn = lambda: gpu_prefill(wd, out=out)  # noqa: E731
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


def test_prefill_empty_calls(dev):
    w = workloads.prefill_inputs([0, 0, 0], 4, seed=79)
    wd = w.to(dev)
    st0 = wd.state.clone()
    out = torch.full((1, 12, 128), SENTINEL, dtype=torch.bfloat16, device=dev)
    q = torch.zeros((0, 12, 128), dtype=torch.bfloat16, device=dev)
    b = torch.zeros((0, 12), dtype=torch.bfloat16, device=dev)
    kda.kda_prefill(wd.state, wd.state_indices, wd.cu_seqlens, q, q, q, q, b, wd.A_log, wd.dt_bias, out=out[:0])
    w2 = workloads.prefill_inputs([4, 0, 2], 4, seed=80)
    wd2 = w2.to(dev)
    cu0 = torch.zeros(1, dtype=torch.int32, device=dev)
    idx0 = torch.zeros(0, dtype=torch.int32, device=dev)
    o2 = torch.full((6, 12, 128), SENTINEL, dtype=torch.bfloat16, device=dev)
    kda.kda_prefill(wd2.state, idx0, cu0, wd2.q, wd2.k, wd2.v, wd2.g_raw, wd2.beta_logit, wd2.A_log, wd2.dt_bias,
                    out=o2)
    torch.cuda.synchronize()
    assert torch.equal(wd.state, st0)
    assert torch.all(o2.float() == SENTINEL), "no sequence: nothing written"
    assert torch.equal(wd2.state, w2.state.to(dev))


def test_prefill_rejects_bad_arguments(dev):
    w = workloads.prefill_inputs([3, 2], 4, seed=81)
    wd = w.to(dev)
    with pytest.raises(kda.KdaError) as e:
        gpu_prefill(wd, config_override=5)
    assert e.value.status == kda.KDA_EINVAL
    with pytest.raises(TypeError):
        kda.kda_prefill(wd.state, wd.state_indices, wd.cu_seqlens.long(), wd.q, wd.k, wd.v, wd.g_raw,
                        wd.beta_logit, wd.A_log, wd.dt_bias)
    with pytest.raises(ValueError):
        kda.kda_prefill(wd.state, wd.state_indices[:1], wd.cu_seqlens, wd.q, wd.k, wd.v, wd.g_raw,
                        wd.beta_logit, wd.A_log, wd.dt_bias)


@pytest.mark.parametrize("S,L", [(512, 16), (64, 256)])
def test_prefill_bench_shapes_sampled(dev, S, L):
    """The bench's workloads in its launch configuration: 12 sampled sequences
    against the oracle (outputs and final states), every other slot untouched
    and every row written."""
    w = workloads.prefill_inputs([L] * S, S + 8, seed=90 + S, layout="fused")
    wd = w.to(dev)
    out = gpu_prefill(wd)
    torch.cuda.synchronize()
    got_out, got_state = f64(out), f64(wd.state)
    assert np.all(got_out != SENTINEL), "every row belongs to a sequence"
    rng = np.random.default_rng(S)
    picks = rng.choice(S, size=12, replace=False)
    for i in picks:
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


def test_prefill_sixty_four_heads(dev):
    """The largest head count the library takes."""
    w = workloads.prefill_inputs([3, 18], 3, seed=82, H=64)
    wd = w.to(dev)
    out = gpu_prefill(wd)
    torch.cuda.synchronize()
    check_prefill(w, wd, out)


def test_prefill_on_a_side_stream_same_bits(dev):
    """Launched on a caller's stream: the same bits as on the current stream."""
    w = workloads.prefill_inputs([11, 4, 27], 5, seed=83)
    a, b = w.to(dev), w.to(dev)
    oa = gpu_prefill(a)
    side = torch.cuda.Stream(device=dev)
    side.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(side):
        ob = gpu_prefill(b, stream=side)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_prefill_empty_pool_writes_zeros(dev):
    """N = 0: every sequence is inactive, its rows are zero, nothing else is read."""
    w = workloads.prefill_inputs([4, 9], 2, seed=84)
    wd = w.to(dev)
    empty = torch.empty((0, 12, 128, 128), dtype=torch.bfloat16, device=dev)
    out = torch.full((13, 12, 128), SENTINEL, dtype=torch.bfloat16, device=dev)
    kda.kda_prefill(empty, wd.state_indices, wd.cu_seqlens, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                    wd.A_log, wd.dt_bias, out=out)
    torch.cuda.synchronize()
    assert torch.all(out.float() == 0.0)
