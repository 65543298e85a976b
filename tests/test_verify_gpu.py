"""kda_verify (T tokens) on the GPU: against the oracle token by token, and
bit for bit against T chained kda_decode calls (the CUDA-core configurations
0-3). Every state comparison is per element at the single-step bound: the
oracle step for token t starts from the GPU's own state after t tokens
(harness.verify_teacher_forced). The tensor-core configuration (4) sums the
dot products in another order than the CUDA-core ones: each of its tokens is
held to that bound against the oracle, and against one GPU decode step from
its own previous state; it is bitwise deterministic on its own."""

import numpy as np
import pytest
import torch

from harness import (assert_output_close, assert_state_close, decode_token, f64, gpu_decode, gpu_verify,
                     identity_tokens, token_slice, verify_teacher_forced)
from linear_attention_ssm_step_gb300 import kda, workloads

TC = 4  # the tensor-core configuration

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def check_verify(w, dev, rows=None, **kw):
    wd, out, _ = verify_teacher_forced(w, dev, rows=rows, **kw)
    torch.cuda.synchronize()
    if rows is None:  # slots no active row owns are untouched
        idx = w.state_indices.numpy().astype(np.int64)
        owned = set(idx[(idx >= 0) & (idx < w.N)].tolist())
        rest = [n for n in range(w.N) if n not in owned]
        assert torch.equal(wd.state.cpu()[rest].view(torch.int16), w.state[rest].view(torch.int16))
    return wd, out


@pytest.mark.parametrize("T", [1, 2, 8, 16])
@pytest.mark.parametrize("B", [1, 5, 32])
def test_verify_matches_oracle(dev, B, T):
    if B == 32 and T == 16:
        pytest.skip("covered by the T=8 case; keeps the oracle time short")
    w = workloads.decode_inputs(B, B + 64, seed=300 + 17 * B + T, T=T, inactive_frac=0.2 if B == 5 else 0.0)
    check_verify(w, dev)


@pytest.mark.parametrize("T", [2, 8, 16])
@pytest.mark.parametrize("B", [1, 5, 32])
def test_verify_tensor_cores_match_oracle(dev, B, T):
    if B == 32 and T == 16:
        pytest.skip("covered by the T=8 case; keeps the oracle time short")
    w = workloads.decode_inputs(B, B + 64, seed=310 + 17 * B + T, T=T, inactive_frac=0.2 if B == 5 else 0.0)
    check_verify(w, dev, config_override=TC)


@pytest.mark.parametrize("H", [1, 3, 64])
@pytest.mark.parametrize("config", [3, TC])
def test_verify_other_head_counts(dev, H, config):
    w = workloads.decode_inputs(2, 4, seed=320 + H, T=4, H=H)
    check_verify(w, dev, config_override=config)


def test_verify_large_batch_sampled(dev):
    """T = 8, B = 2048 on the default (tensor-core) configuration; 12 rows compared with the oracle."""
    w = workloads.decode_inputs(2048, 2112, seed=321, T=8, inactive_frac=0.05)
    idx = w.state_indices.numpy().astype(np.int64)
    active = np.nonzero((idx >= 0) & (idx < w.N))[0]
    rows = np.sort(np.random.default_rng(6).choice(active, 12, replace=False))
    check_verify(w, dev, rows=rows)


def test_verify_tensor_cores_match_decode_steps(dev):
    """Configuration 4 token by token against the GPU's own T = 1 decode: the
    state after t + 1 tokens of a tensor-core verify equals one kda_decode step
    from its state after t tokens to the single-step bound, and so do the
    outputs to theirs. (The two sum the dot products in different orders.)"""
    T = 8
    w = workloads.decode_inputs(7, 20, seed=408, T=T, inactive_frac=0.15, layout="packed")
    idx = w.state_indices.numpy().astype(np.int64)
    act = idx[(idx >= 0) & (idx < w.N)]
    wd = w.to(dev)
    out_v = gpu_verify(wd, config_override=TC)
    for t in range(T):
        if t == 0:
            pre = w.to(dev)
        else:
            pre = (identity_tokens(token_slice(w, 0, 2), 1) if t == 1 else token_slice(w, 0, t)).to(dev)
            gpu_verify(pre, config_override=TC)
        nxt = wd if t == T - 1 else (identity_tokens(token_slice(w, 0, 2), 1) if t == 0 else
                                      token_slice(w, 0, t + 1)).to(dev)
        if t < T - 1:
            gpu_verify(nxt, config_override=TC)
        step = decode_token(w, t).to(dev)
        step.state = pre.state
        out_d = gpu_decode(step)
        torch.cuda.synchronize()
        assert_state_close(f64(nxt.state)[act], f64(pre.state)[act], f"token {t}: verify against a decode step")
        assert_output_close(f64(out_v)[:, t], f64(out_d), f"token {t} output")


def test_identity_token_leaves_the_tensor_core_state_unchanged(dev):
    """The one-token prefix of the teacher-forced checks pads configuration 4 with
    an identity token: a trailing identity token changes no state bit."""
    w = workloads.decode_inputs(5, 12, seed=409, T=3, inactive_frac=0.2)
    a = identity_tokens(w, 2).to(dev)
    b = token_slice(w, 0, 2).to(dev)
    oa = gpu_verify(a, config_override=TC)
    ob = gpu_verify(b, config_override=TC)
    torch.cuda.synchronize()
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))
    assert torch.equal(oa[:, :2].view(torch.int16), ob.view(torch.int16))


def test_verify_tensor_cores_serving_batch_512_sampled(dev):
    w = workloads.decode_inputs(512, 576, seed=3, T=8)
    rows = np.sort(np.random.default_rng(2).choice(512, 24, replace=False))
    check_verify(w, dev, rows=rows, config_override=TC)


def test_verify_tensor_cores_misaligned_state_same_bits(dev):
    w = workloads.decode_inputs(4, 6, seed=5, T=4)
    wd = w.to(dev)
    flat = torch.empty(6 * 12 * 128 * 128 + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[3:3 + 6 * 12 * 128 * 128].view(6, 12, 128, 128)
    mis.copy_(wd.state)
    out_a = gpu_verify(wd, config_override=TC)
    wd.state = mis
    out_b = gpu_verify(wd, config_override=TC)
    ref = w.to(dev)
    gpu_verify(ref, config_override=TC)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(mis.view(torch.int16), ref.state.view(torch.int16))


def _shifted(x, dev):
    """x copied to a buffer one element (2 bytes) off a 16-byte boundary."""
    flat = torch.empty(x.numel() + 8, dtype=x.dtype, device=dev)
    y = flat[1:1 + x.numel()].view(x.shape)
    y.copy_(x)
    return y


def test_verify_tensor_cores_misaligned_token_views_same_bits(dev):
    """Token views off a 16-byte boundary take per-lane loads in place of the
    tensor-map copies of the token inputs: the same values, the same bits."""
    w = workloads.decode_inputs(6, 10, seed=17, T=8, inactive_frac=0.2)
    a, b = w.to(dev), w.to(dev)
    b.q_sep, b.k_sep, b.v_sep, b.g_raw = (_shifted(x, dev) for x in (b.q_sep, b.k_sep, b.v_sep, b.g_raw))
    assert b.q_sep.data_ptr() % 16 == 2
    oa, ob = gpu_verify(a, config_override=TC), gpu_verify(b, config_override=TC)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))


def test_verify_tensor_cores_cuda_graph_bitwise(dev):
    w = workloads.decode_inputs(6, 10, seed=6, T=8)
    wd = w.to(dev)
    init = wd.state.clone()
    gpu_verify(wd, config_override=TC)
    torch.cuda.synchronize()
    out = torch.empty((6, 8, 12, 128), dtype=torch.bfloat16, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_verify(wd, out=out, config_override=TC)
    res = []
    for _ in range(3):
        wd.state.copy_(init)
        graph.replay()
        torch.cuda.synchronize()
        res.append((out.clone(), wd.state.clone()))
    for o, s in res[1:]:
        assert torch.equal(o.view(torch.int16), res[0][0].view(torch.int16))
        assert torch.equal(s.view(torch.int16), res[0][1].view(torch.int16))


def test_verify_tensor_cores_precomputed_gate_convention(dev):
    w = workloads.decode_inputs(5, 12, seed=8, T=8, inactive_frac=0.2, gate_mode=1)
    w.A_log = w.dt_bias = None
    check_verify(w, dev, config_override=TC)


def test_tensor_core_configuration_needs_several_tokens(dev):
    w = workloads.decode_inputs(3, 6, seed=9, T=1)
    wd = w.to(dev)
    with pytest.raises(kda.KdaError):
        gpu_verify(wd, config_override=TC)
    w1 = workloads.decode_inputs(3, 6, seed=9)
    with pytest.raises(kda.KdaError):
        gpu_decode(w1.to(dev), config_override=TC)


@pytest.mark.parametrize("T", [2, 8])
@pytest.mark.parametrize("config", [0, 1, 2, 3])
def test_verify_equals_chained_decodes_bitwise(dev, T, config):
    kw = {} if config is None else {"config_override": config}
    w = workloads.decode_inputs(7, 20, seed=400 + T, T=T, inactive_frac=0.15, layout="packed")
    wd = w.to(dev)
    out_v = gpu_verify(wd, **kw)
    wc = w.to(dev)
    outs = []
    for t in range(T):
        outs.append(gpu_decode(_token(wc, t), **kw))
    torch.cuda.synchronize()
    assert torch.equal(wd.state.view(torch.int16), wc.state.view(torch.int16))
    assert torch.equal(out_v.view(torch.int16), torch.stack(outs, dim=1).view(torch.int16))


def _token(w, t):
    """Token t of a T-token workload as a decode workload sharing the pool."""
    from dataclasses import replace
    return replace(w, T=None, g_raw=w.g_raw[:, t], beta_logit=w.beta_logit[:, t],
                   qkv=None if w.qkv is None else w.qkv[:, t],
                   q_sep=None if w.q_sep is None else w.q_sep[:, t],
                   k_sep=None if w.k_sep is None else w.k_sep[:, t],
                   v_sep=None if w.v_sep is None else w.v_sep[:, t])


def test_verify_serving_batch_512_sampled(dev):
    """T = 8, B = 512, pool of 576: all rows run, 24 compared with the oracle."""
    w = workloads.decode_inputs(512, 576, seed=3, T=8)
    rows = np.sort(np.random.default_rng(1).choice(512, 24, replace=False))
    check_verify(w, dev, rows=rows)


def test_verify_misaligned_state_same_bits(dev):
    w = workloads.decode_inputs(4, 6, seed=5, T=4)
    wd = w.to(dev)
    flat = torch.empty(6 * 12 * 128 * 128 + 8, dtype=torch.bfloat16, device=dev)
    mis = flat[3:3 + 6 * 12 * 128 * 128].view(6, 12, 128, 128)
    mis.copy_(wd.state)
    out_a = gpu_verify(wd)
    wd.state = mis
    out_b = gpu_verify(wd)
    ref = w.to(dev)
    gpu_verify(ref)
    torch.cuda.synchronize()
    assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
    assert torch.equal(mis.view(torch.int16), ref.state.view(torch.int16))


def test_verify_cuda_graph_bitwise(dev):
    w = workloads.decode_inputs(6, 10, seed=6, T=8)
    wd = w.to(dev)
    init = wd.state.clone()
    gpu_verify(wd)
    torch.cuda.synchronize()
    out = torch.empty((6, 8, 12, 128), dtype=torch.bfloat16, device=dev)
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        gpu_verify(wd, out=out)
    res = []
    for _ in range(3):
        wd.state.copy_(init)
        graph.replay()
        torch.cuda.synchronize()
        res.append((out.clone(), wd.state.clone()))
    for o, s in res[1:]:
        assert torch.equal(o.view(torch.int16), res[0][0].view(torch.int16))
        assert torch.equal(s.view(torch.int16), res[0][1].view(torch.int16))


def test_verify_precomputed_gate_convention(dev):
    w = workloads.decode_inputs(5, 12, seed=7, T=8, inactive_frac=0.2, gate_mode=1)
    w.A_log = w.dt_bias = None
    check_verify(w, dev)
