"""Prepared calls (kda.prepare_*): bound once to their tensors, each call gives
the bits of the direct call on the same inputs."""

import pytest
import torch

from linear_attention_ssm_step_gb300 import kda, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def test_prepared_verify(dev):
    w = workloads.decode_inputs(6, 9, seed=700, T=8, inactive_frac=0.2)
    a, b = w.to(dev), w.to(dev)
    call = kda.prepare_verify(a.state, a.state_indices, a.q, a.k, a.v, a.g_raw, a.beta_logit, a.A_log, a.dt_bias)
    for _ in range(2):  # chained: the state advances in place
        out_a = call()
        out_b = kda.kda_verify(b.state, b.state_indices, b.q, b.k, b.v, b.g_raw, b.beta_logit, b.A_log, b.dt_bias)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b) and torch.equal(a.state, b.state)


def test_prepared_verify_ring(dev):
    w = workloads.ring_inputs(5, 9, T=8, W=32, flush_min=9, fold_frac=0.5, seed=701)
    a, b = w.to(dev), w.to(dev)
    ra, rb = a.ring, b.ring
    call = kda.prepare_verify_ring(a.state, a.state_indices, a.q, a.k, a.v, a.g_raw, a.beta_logit, a.A_log,
                                   a.dt_bias, ra["k_cache"], ra["u_cache"], ra["g_cache"], ra["hist_len"], 9)
    out_a = call()
    out_b = kda.kda_verify_ring(b.state, b.state_indices, b.q, b.k, b.v, b.g_raw, b.beta_logit, b.A_log,
                                b.dt_bias, rb["k_cache"], rb["u_cache"], rb["g_cache"], rb["hist_len"], 9)
    torch.cuda.synchronize()
    assert torch.equal(out_a, out_b) and torch.equal(a.state, b.state)
    for name in ("k_cache", "u_cache", "g_cache", "hist_len"):
        assert torch.equal(ra[name].nan_to_num(7.0), rb[name].nan_to_num(7.0)), name


def test_prepared_decode_fp8(dev):
    w = workloads.decode_inputs(7, 10, seed=702, layout="packed", inactive_frac=0.2)
    codes, scales = workloads.fp8_pool(10, seed=703)
    a = w.to(dev)
    ca, sa = codes.to(dev), scales.to(dev)
    cb, sb = codes.to(dev), scales.to(dev)
    call = kda.prepare_decode_fp8(ca, sa, a.state_indices, a.q, a.k, a.v, a.g_raw, a.beta_logit, a.A_log,
                                  a.dt_bias)
    for _ in range(2):
        out_a = call()
        out_b = kda.kda_decode_fp8(cb, sb, a.state_indices, a.q, a.k, a.v, a.g_raw, a.beta_logit, a.A_log,
                                   a.dt_bias)
        torch.cuda.synchronize()
        assert torch.equal(out_a, out_b) and torch.equal(ca, cb) and torch.equal(sa, sb)


def test_prepared_prefill(dev):
    """Bound once; refilling the bound input buffers between calls (new tokens of
    the same sequence lengths) gives the direct call's bits."""
    w = workloads.prefill_inputs([7, 0, 19], 5, seed=703, inactive_frac=0.3)
    w2 = workloads.prefill_inputs([7, 0, 19], 5, seed=704)
    a, b = w.to(dev), w.to(dev)
    call = kda.prepare_prefill(a.state, a.state_indices, a.cu_seqlens, a.q_sep, a.k_sep, a.v_sep, a.g_raw,
                               a.beta_logit, a.A_log, a.dt_bias)
    for step in range(2):
        if step == 1:  # the next step's token inputs, into the bound buffers
            for name in ("q_sep", "k_sep", "v_sep", "g_raw", "beta_logit"):
                getattr(a, name).copy_(getattr(w2, name))
                getattr(b, name).copy_(getattr(w2, name))
        out_a = call()
        out_b = kda.kda_prefill(b.state, b.state_indices, b.cu_seqlens, b.q, b.k, b.v, b.g_raw, b.beta_logit,
                                b.A_log, b.dt_bias)
        torch.cuda.synchronize()
        assert torch.equal(out_a.view(torch.int16), out_b.view(torch.int16))
        assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16))
