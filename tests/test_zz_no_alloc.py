"""kda_prefill_static: the two-stage prefill with its workspace in a fixed
array inside the library, for callers that cannot allocate device memory when
they run a prefill (a step captured in global capture mode, a plugin host that
owns all device memory, a server that reserved all of it at start-up).

Through the C ABI, against kda_prefill_ws with a caller-allocated workspace on
the same inputs, with the prefill tolerances (outputs 2e-2 + 2e-2 |o_ref|,
states 2 bf16 ulps at max(|s_ref|, F_L M)), on two calls in a row: the second
call finds the first one's contents in the shared array. Also the size limit.
This file is collected last on purpose, so that a run stopping at the first
failure has run every other test before it.
"""

import ctypes

import pytest
import torch

from harness import assert_output_close, assert_prefill_state_close, f64
from linear_attention_ssm_step_gb300 import kda, workloads

pytestmark = pytest.mark.gpu

LB = -5.0


@pytest.fixture(scope="module")
def dev():
    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    import __graft_entry__
    __graft_entry__.build()
    return torch.device("cuda:0")


def _params(wd, out, config=-1):
    S = wd.cu_seqlens.shape[0] - 1
    p = kda._params(wd.state, wd.state_indices, wd.q, wd.k, wd.v, wd.g_raw, wd.beta_logit, wd.A_log, wd.dt_bias,
                    out, None, LB, 1.0, None, config, wd.gate_mode, n_indices=S)
    return p, kda.KdaSeqs(wd.cu_seqlens.data_ptr(), S)


def _static_call(wd):
    out = torch.full((wd.q.shape[0], wd.H, 128), 7.0, dtype=torch.bfloat16, device=wd.q.device)
    p, sq = _params(wd, out)
    st = kda.load_library().kda_prefill_static(ctypes.byref(p), ctypes.byref(sq),
                                               kda._stream_handle(None, wd.q.device))
    assert st == kda.KDA_OK, kda.kda_last_error()
    return out


def _workspace_call(wd):
    out = torch.full((wd.q.shape[0], wd.H, 128), 7.0, dtype=torch.bfloat16, device=wd.q.device)
    p, sq = _params(wd, out, config=5)
    ws = kda.prefill_workspace(wd.q.shape[0], sq.num_seqs, wd.H, wd.q.device)
    st = kda.load_library().kda_prefill_ws(ctypes.byref(p), ctypes.byref(sq), ws.data_ptr(), ws.numel(),
                                           kda._stream_handle(None, wd.q.device))
    assert st == kda.KDA_OK, kda.kda_last_error()
    return out


@pytest.mark.parametrize("lengths,H,seed", [([700, 33, 5, 0, 300], 12, 301), ([1200, 64, 17], 8, 302)])
def test_no_alloc_prefill_matches_workspace_prefill_twice(dev, lengths, H, seed):
    """Two calls in a row on different inputs, each against kda_prefill_ws."""
    for call in range(2):
        w = workloads.prefill_inputs(lengths, len(lengths) + 3, seed=seed + 10 * call, H=H, inactive_frac=0.2)
        a, b = w.to(dev), w.to(dev)
        oa = _static_call(a)
        ob = _workspace_call(b)
        torch.cuda.synchronize()
        assert_output_close(f64(oa), f64(ob), f"outputs, call {call}")
        for i, n in enumerate(w.state_indices.tolist()):
            if 0 <= n < w.N:
                assert_prefill_state_close(f64(a.state)[n], f64(b.state)[n], max(lengths[i], 1),
                                           f"state of sequence {i}, call {call}")
        assert torch.equal(a.state.view(torch.int16), b.state.view(torch.int16)), "the same kernels: the same bits"


def test_no_alloc_prefill_rejects_calls_beyond_its_workspace(dev):
    """A call that needs more than the fixed 64 MiB is refused before anything runs."""
    w = workloads.prefill_inputs([40], 2, seed=303)
    wd = w.to(dev)
    out = torch.empty((wd.q.shape[0], 12, 128), dtype=torch.bfloat16, device=dev)
    p, sq = _params(wd, out)
    p.B = 16 * 2000  # (2000 + 1) chunk slots x 12 heads x 45568 bytes > 64 MiB; checked before any pointer is used
    st = kda.load_library().kda_prefill_static(ctypes.byref(p), ctypes.byref(sq), kda._stream_handle(None, dev))
    assert st == kda.KDA_EUNSUPPORTED
    assert "kda_prefill_ws" in kda.kda_last_error()
    p.B = wd.q.shape[0]
    p.config_override = 4
    st = kda.load_library().kda_prefill_static(ctypes.byref(p), ctypes.byref(sq), kda._stream_handle(None, dev))
    assert st == kda.KDA_EINVAL
    torch.cuda.synchronize()
    assert torch.equal(wd.state.cpu().view(torch.int16), w.state.view(torch.int16)), "nothing ran"
