"""kda_verify_fp8 (T-token verify on an fp8 state pool) on the GPU, through the C ABI.

The reading: T kda_decode_fp8 steps on the same slot, the row requantized
after every token, so a verify of T tokens equals T decode calls bit for bit
(checked here for every configuration and T up to 16). Each token is also
checked against the fp8 oracle teacher-forced: the oracle's decode step starts
from the GPU's own pool before that token (the pool after a verify of the
first t tokens, or the initial pool), and its output and requantized pool are
compared with the verify's output for token t and the pool after t + 1 tokens,
with the fp8 decode's tolerances (test_fp8_gpu.check_state; outputs
2e-2 + 2e-2 |o_ref|).
"""

import numpy as np
import pytest
import torch

import oracle
from harness import assert_output_close, decode_token, f64, token_slice
from linear_attention_ssm_step_gb300 import kda, workloads
from test_fp8_gpu import LB, check_state

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def make(B, N, T, seed, layout="fused", inactive_frac=0.0, H=12, gate_mode=0):
    w = workloads.decode_inputs(B, N, seed=seed, T=T, layout=layout, inactive_frac=inactive_frac, H=H,
                                gate_mode=gate_mode)
    codes, scales = workloads.fp8_pool(N, H=H, seed=seed + 7)
    return w, codes, scales


def verify(wd, c, s, **kw):
    return kda.kda_verify_fp8(c, s, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log,
                              wd.dt_bias, lower_bound=LB, gate_mode=wd.gate_mode, **kw)


def decode(wd, c, s, **kw):
    return kda.kda_decode_fp8(c, s, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log,
                              wd.dt_bias, lower_bound=LB, gate_mode=wd.gate_mode, **kw)


@pytest.mark.parametrize("B,T,config", [(1, 2, -1), (5, 8, -1), (5, 8, 0), (40, 16, -1), (40, 3, 3), (64, 8, -1)])
def test_fp8_verify_equals_chained_decodes(dev, B, T, config):
    w, codes, scales = make(B, B + 4, T, seed=600 + B + T, inactive_frac=0.2 if B > 1 else 0.0)
    wd = w.to(dev)
    ca, sa = codes.to(dev), scales.to(dev)
    cb, sb = codes.to(dev), scales.to(dev)
    out_v = verify(wd, ca, sa, config_override=config)
    outs = [decode(decode_token(wd, t), cb, sb, config_override=config if config != -1 else -1) for t in range(T)]
    torch.cuda.synchronize()
    for t in range(T):
        assert torch.equal(out_v[:, t].view(torch.int16), outs[t].view(torch.int16)), f"token {t}"
    assert torch.equal(ca, cb) and torch.equal(sa.view(torch.int32), sb.view(torch.int32))
    idx = w.state_indices.numpy().astype(np.int64)
    inactive = (idx < 0) | (idx >= w.N)
    assert (f64(out_v)[inactive] == 0).all(), "inactive rows give exactly zero"


@pytest.mark.parametrize("gate_mode", [0, 1])
def test_fp8_verify_teacher_forced_against_oracle(dev, gate_mode):
    B, T, N = 5, 6, 9
    w, codes, scales = make(B, N, T, seed=620 + gate_mode, gate_mode=gate_mode)
    wd = w.to(dev)
    c_full, s_full = codes.to(dev), scales.to(dev)
    out_full = f64(verify(wd, c_full, s_full))
    torch.cuda.synchronize()
    idx = w.state_indices.numpy().astype(np.int64)
    pools = [(codes.numpy(), scales.double().numpy())]  # the GPU's pool before token t
    for t in range(1, T + 1):
        c_t, s_t = codes.to(dev), scales.to(dev)
        verify(token_slice(wd, 0, t), c_t, s_t)
        torch.cuda.synchronize()
        pools.append((c_t.cpu().numpy(), s_t.cpu().double().numpy()))
    assert np.array_equal(pools[T][0], c_full.cpu().numpy()), "a prefix of T tokens is the full call"
    for t in range(T):
        wt = decode_token(w, t)
        c0, s0 = pools[t]
        ref_c, ref_s, ref_out, info = oracle.kda_decode_fp8(
            c0, s0, wt.state_indices.numpy(), f64(wt.q), f64(wt.k), f64(wt.v), f64(wt.g_raw), f64(wt.beta_logit),
            None if w.A_log is None else f64(w.A_log), None if w.dt_bias is None else f64(w.dt_bias), LB, 1.0,
            gate_mode)
        assert_output_close(out_full[:, t], ref_out, what=f"output of token {t}")
        got_c, got_s = pools[t + 1]
        check_state(got_c[idx], got_s[idx], ref_c[idx], ref_s[idx], info["S_new"])


def test_fp8_verify_plain_path_equals_bulk_path(dev):
    """Codes at an odd offset take plain loads and stores: the same bits."""
    w, codes, scales = make(6, 8, 5, seed=640)
    wd = w.to(dev)
    ca, sa = codes.to(dev), scales.to(dev)
    flat = torch.empty(codes.numel() + 16, dtype=torch.uint8, device=dev)
    cb = flat[1:1 + codes.numel()].view(codes.shape)
    cb.copy_(codes.to(dev))
    sb = scales.to(dev)
    assert cb.data_ptr() % 16 == 1
    oa, ob = verify(wd, ca, sa), verify(wd, cb, sb)
    torch.cuda.synchronize()
    assert torch.equal(oa.view(torch.int16), ob.view(torch.int16))
    assert torch.equal(ca, cb) and torch.equal(sa.view(torch.int32), sb.view(torch.int32))


def test_fp8_verify_graph_replay_is_deterministic(dev):
    w, codes, scales = make(32, 36, 8, seed=650)
    wd = w.to(dev)
    c, s = codes.to(dev), scales.to(dev)
    c0, s0 = c.clone(), s.clone()
    out = torch.empty((32, 8, 12, 128), dtype=torch.bfloat16, device=dev)
    verify(wd, c, s, out=out)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        verify(wd, c, s, out=out)
    results = []
    for _ in range(2):
        c.copy_(c0)
        s.copy_(s0)
        g.replay()
        torch.cuda.synchronize()
        results.append((out.clone(), c.clone(), s.clone()))
    assert all(torch.equal(a, b) for a, b in zip(results[0], results[1]))


def test_fp8_verify_rejects_bad_arguments(dev):
    w, codes, scales = make(2, 3, 4, seed=660)
    wd = w.to(dev)
    c, s = codes.to(dev), scales.to(dev)
    with pytest.raises(kda.KdaError) as e:
        verify(wd, c, s, config_override=4)
    assert e.value.status == kda.KDA_EUNSUPPORTED
    w17, codes17, scales17 = make(1, 2, 16, seed=661)
    with pytest.raises(kda.KdaError) as e:
        verify(token_slice(w17.to(dev), 0, 16), c[:2], s[:2], config_override=5)
    assert e.value.status == kda.KDA_EINVAL
    with pytest.raises(TypeError):
        kda.kda_verify_fp8(c, s.double(), wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit,
                           wd.A_log, wd.dt_bias)
