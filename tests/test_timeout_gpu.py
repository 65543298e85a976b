"""Failure detection on the GPU without a fault: the kernels' bounded waits.

The "waittest" build of the library (linear_attention_ssm_step_gb300/_build.py,
KDA_WITHHOLD_LOADS in csrc/kda_device.cuh) is the same source with every
asynchronous global -> shared copy left unissued while its mbarrier still
expects the bytes, and a wait limit of 2 ms: each kernel's wait for its state
copy runs out exactly as on a copy that never lands, with nothing in flight.
Every call must then
  * OR KDA_ERR_TIMEOUT into the caller's error word,
  * give zero outputs for the rows it skipped (here: every row),
  * leave the state pool (and the ring, and the fp8 scales) bit for bit as
    they were,
and the CUDA context must stay usable: the regular library runs a decode
afterwards and matches the oracle.
"""

import ctypes

import numpy as np
import pytest
import torch

from harness import assert_output_close, assert_state_close, f64, gpu_decode, oracle_decode
from linear_attention_ssm_step_gb300 import _build, kda, workloads

pytestmark = pytest.mark.gpu

LB = -5.0


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


@pytest.fixture(scope="module")
def wlib(dev):
    """The failure-detection build, loaded beside the regular library."""
    return kda.bind_library(_build.build(variant="waittest"))


def _err(dev):
    return torch.zeros(1, dtype=torch.int32, device=dev)


def _params(wd, out, err, T=None, config=-1, n_indices=None):
    return kda._params(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log,
                       wd.dt_bias, out, T, LB, 1.0, err, config, wd.gate_mode, n_indices=n_indices)


def _sentinel_out(shape, dev):
    return torch.full(shape, 3.0, dtype=torch.bfloat16, device=dev)


def _expect_timeout(err, out, rows=None):
    torch.cuda.synchronize()
    assert int(err.item()) & kda.KDA_ERR_TIMEOUT, "the error word must report the bounded wait that gave up"
    o = out if rows is None else out[rows]
    assert (o.float() == 0).all(), "skipped rows give zero output"


@pytest.mark.parametrize("B", [3, 40])
def test_decode_timeout_skips_and_reports(dev, wlib, B):
    w = workloads.decode_inputs(B, B + 4, seed=700 + B, layout="packed")
    wd = w.to(dev)
    out, err = _sentinel_out((B, 12, 128), dev), _err(dev)
    p = _params(wd, out, err)
    assert wlib.kda_decode(ctypes.byref(p), kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(wd.state.cpu().view(torch.int16), w.state.view(torch.int16))


@pytest.mark.parametrize("config", [2, 4])
def test_verify_timeout_skips_and_reports(dev, wlib, config):
    """CUDA-core verify (bulk copies) and tensor-core verify (tensor-map loads,
    tensor memory released on the way out)."""
    w = workloads.decode_inputs(6, 10, seed=710 + config, T=8)
    wd = w.to(dev)
    out, err = _sentinel_out((6, 8, 12, 128), dev), _err(dev)
    p = _params(wd, out, err, T=8, config=config)
    assert wlib.kda_verify(ctypes.byref(p), 8, kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(wd.state.cpu().view(torch.int16), w.state.view(torch.int16))


def test_ring_timeout_skips_and_reports(dev, wlib):
    """The persistent ring kernel: the first wait gives up, the CTA issues
    nothing more, skips all its items, and releases its tensor memory. The
    checkpoint and the ring are untouched; hist_len is reset as after any
    call for rows that reach flush_min (the reset kernel runs in stream order
    and does not see the skip)."""
    w = workloads.ring_inputs(6, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=720)
    wd = w.to(dev)
    out, err = _sentinel_out((6, 8, 12, 128), dev), _err(dev)
    p = _params(wd, out, err, T=8)
    r = wd.ring
    rp = kda._ring_params(wd.state, 12, r["k_cache"], r["u_cache"], r["g_cache"], r["hist_len"], r["flush_min"],
                          True, None)
    assert wlib.kda_verify_ring(ctypes.byref(p), 8, ctypes.byref(rp), kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(wd.state.cpu().view(torch.int16), w.state.view(torch.int16))
    for name in ("k_cache", "u_cache", "g_cache"):
        assert np.array_equal(f64(r[name]), f64(w.ring[name]), equal_nan=True), name
    hist0 = w.ring["hist_len"].clone()
    idx = w.state_indices.long()
    want = hist0.clone()
    want[idx] = torch.where(hist0[idx] >= 9, torch.zeros_like(hist0[idx]), hist0[idx])
    assert torch.equal(r["hist_len"].cpu(), want)


def test_prefill_timeout_skips_and_reports(dev, wlib):
    w = workloads.prefill_inputs([5, 19, 1, 40], 8, seed=730)
    wd = w.to(dev)
    L = w.q.shape[0]
    out, err = _sentinel_out((L, 12, 128), dev), _err(dev)
    p = _params(wd, out, err, n_indices=4)
    sq = kda.KdaSeqs(wd.cu_seqlens.data_ptr(), 4)
    assert wlib.kda_prefill(ctypes.byref(p), ctypes.byref(sq), kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(wd.state.cpu().view(torch.int16), w.state.view(torch.int16))


@pytest.mark.parametrize("config", [5, 6])
def test_prefill_two_stage_timeout_skips_and_reports(dev, wlib, config):
    """Configurations 5 and 6: the chain's waits for the state and for its
    chunk images run out; the preparation, which waits for nothing (and in
    configuration 6 publishes every image it writes), still fills the
    workspace."""
    w = workloads.prefill_inputs([5, 19, 1, 70], 8, seed=735)
    wd = w.to(dev)
    L = w.q.shape[0]
    out, err = _sentinel_out((L, 12, 128), dev), _err(dev)
    p = _params(wd, out, err, n_indices=4)
    p.config_override = config
    sq = kda.KdaSeqs(wd.cu_seqlens.data_ptr(), 4)
    ws = torch.empty(int(wlib.kda_prefill_workspace_bytes(L, 4, 12)), dtype=torch.uint8, device=dev)
    assert wlib.kda_prefill_ws(ctypes.byref(p), ctypes.byref(sq), ws.data_ptr(), ws.numel(),
                               kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(wd.state.cpu().view(torch.int16), w.state.view(torch.int16))


def test_fp8_decode_timeout_skips_and_reports(dev, wlib):
    w = workloads.decode_inputs(4, 6, seed=740)
    codes, scales = workloads.fp8_pool(6, seed=741)
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    out, err = _sentinel_out((4, 12, 128), dev), _err(dev)
    p = kda._params(c_d, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log, wd.dt_bias, out,
                    None, LB, 1.0, err, -1, wd.gate_mode, state_dtype=torch.uint8)
    f = kda._fp8_pool(c_d, s_d)
    assert wlib.kda_decode_fp8(ctypes.byref(p), ctypes.byref(f), kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(c_d.cpu(), codes)
    assert torch.equal(s_d.cpu().view(torch.int32), scales.view(torch.int32))


def test_fp8_ring_timeout_skips_and_reports(dev, wlib):
    """The ring on an fp8 checkpoint pool: its bulk copy of the codes is never
    issued, the first wait gives up, and codes, scales and the ring stay as
    they were (hist_len reset as in the bf16 ring's case)."""
    w = workloads.ring_inputs(6, 12, T=8, W=32, flush_min=9, fold_frac=0.5, seed=745)
    codes, scales = workloads.fp8_pool(12, seed=746)
    wd = w.to(dev)
    c_d, s_d = codes.to(dev), scales.to(dev)
    out, err = _sentinel_out((6, 8, 12, 128), dev), _err(dev)
    p = kda._params(c_d, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log, wd.dt_bias, out,
                    8, LB, 1.0, err, -1, wd.gate_mode, state_dtype=torch.uint8)
    r = wd.ring
    rp = kda._ring_params(c_d, 12, r["k_cache"], r["u_cache"], r["g_cache"], r["hist_len"], r["flush_min"],
                          True, None)
    f = kda._fp8_pool(c_d, s_d)
    assert wlib.kda_verify_ring_fp8(ctypes.byref(p), 8, ctypes.byref(rp), ctypes.byref(f),
                                    kda._stream_handle(None, dev)) == kda.KDA_OK
    _expect_timeout(err, out)
    assert torch.equal(c_d.cpu(), codes)
    assert torch.equal(s_d.cpu().view(torch.int32), scales.view(torch.int32))
    for name in ("k_cache", "u_cache", "g_cache"):
        assert np.array_equal(f64(r[name]), f64(w.ring[name]), equal_nan=True), name


def test_context_usable_after_timeouts(dev, wlib):
    """After the calls that gave up, the regular library's decode still runs and
    matches the oracle."""
    w = workloads.decode_inputs(5, 9, seed=750, inactive_frac=0.2)
    wd = w.to(dev)
    out = gpu_decode(wd)
    torch.cuda.synchronize()
    ref_state, ref_out = oracle_decode(w)
    idx = w.state_indices.numpy().astype(np.int64)
    act = idx[(idx >= 0) & (idx < w.N)]
    assert_output_close(f64(out), ref_out)
    assert_state_close(f64(wd.state)[act], ref_state[act])
