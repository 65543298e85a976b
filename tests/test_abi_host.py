"""The C ABI on the host, without a GPU: the library loads, exports every
function include/kda.h and include/kda_fp8.h declare, lays out its structs as the binding does,
and rejects malformed arguments before touching CUDA. No call here passes
validation with a non-zero batch, so nothing is ever launched."""

import ctypes
import os
import re
import subprocess
import tempfile

import pytest
import torch

from linear_attention_ssm_step_gb300 import _build, kda

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "kda.h")
HEADERS = [os.path.join(ROOT, "include", h) for h in sorted(os.listdir(os.path.join(ROOT, "include")))
           if h.endswith(".h")]


# The checks that call the entry points pass fake host addresses, which
# validation rejects before any launch. They run only where no GPU is visible,
# so that a validation bug can never launch a kernel on fake pointers.
no_gpu = pytest.mark.skipif(torch.cuda.is_available(), reason="fake-pointer checks run only without a GPU")


@pytest.fixture(scope="module")
def lib():
    _build.build()
    return kda.load_library()


def declared_functions():
    names = set()
    for path in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(path).read(), flags=re.S)
        names |= set(re.findall(r"\b(kda_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_every_declared_function_is_exported(lib):
    names = declared_functions()
    assert {"kda_decode", "kda_verify", "kda_verify_ring", "kda_select_config", "kda_last_error",
            "kda_decode_fp8"} <= set(names)
    for name in names:
        assert hasattr(lib, name), f"{name} declared in a header but not exported"
    assert set(names) == set(kda.EXPORTS), "binding and header disagree"


def test_header_constants_match_binding():
    text = open(HEADER).read()
    for name in ("KDA_ERR_HIST_LEN", "KDA_ERR_TIMEOUT", "KDA_ERR_CACHE_BASE", "KDA_GATE_RAW",
                 "KDA_GATE_PRECOMPUTED", "KDA_MAX_T"):
        m = re.search(r"#define\s+" + name + r"\s+(\d+)u?", text)
        assert m, name
        assert int(m.group(1)) == getattr(kda, name), name
    text = open(os.path.join(ROOT, "include", "kda_prefill.h")).read()
    m = re.search(r"#define\s+KDA_ERR_SEQLENS\s+(\d+)u?", text)
    assert m and int(m.group(1)) == kda.KDA_ERR_SEQLENS


def test_struct_layout_matches_header(tmp_path):
    src = tmp_path / "layout.c"
    src.write_text(r"""
#include <stddef.h>
#include <stdio.h>
#include "kda.h"
#include "kda_fp8.h"
#include "kda_prefill.h"
#define P(s, f) printf(#s "." #f " %zu\n", offsetof(s, f))
int main(void) {
  printf("kda_view %zu\nkda_params %zu\nkda_ring_params %zu\nkda_fp8_pool %zu\nkda_seqs %zu\n",
         sizeof(kda_view), sizeof(kda_params), sizeof(kda_ring_params), sizeof(kda_fp8_pool),
         sizeof(kda_seqs));
  P(kda_fp8_pool, scale); P(kda_fp8_pool, scale_slot_stride);
  P(kda_seqs, cu_seqlens); P(kda_seqs, num_seqs);
  P(kda_params, q); P(kda_params, beta_logit); P(kda_params, A_log); P(kda_params, lower_bound);
  P(kda_params, state); P(kda_params, state_indices); P(kda_params, out); P(kda_params, out_h_stride);
  P(kda_params, error_word); P(kda_params, config_override); P(kda_params, gate_mode);
  P(kda_ring_params, g_slot_stride); P(kda_ring_params, hist_len); P(kda_ring_params, W);
  P(kda_ring_params, restart_hist_on_flush); P(kda_ring_params, cache_base);
  return 0;
}
""")
    exe = tmp_path / "layout"
    subprocess.run(["gcc", "-std=c99", "-I", os.path.join(ROOT, "include"), str(src), "-o", str(exe)], check=True)
    got = dict(line.rsplit(" ", 1) for line in subprocess.check_output([str(exe)], text=True).split("\n") if line)
    assert int(got["kda_view"]) == ctypes.sizeof(kda.KdaView)
    assert int(got["kda_params"]) == ctypes.sizeof(kda.KdaParams)
    assert int(got["kda_ring_params"]) == ctypes.sizeof(kda.KdaRingParams)
    assert int(got["kda_fp8_pool"]) == ctypes.sizeof(kda.KdaFp8Pool)
    assert int(got["kda_seqs"]) == ctypes.sizeof(kda.KdaSeqs)
    for key, val in got.items():
        if "." in key:
            s, f = key.split(".")
            cls = {"kda_params": kda.KdaParams, "kda_ring_params": kda.KdaRingParams,
                   "kda_fp8_pool": kda.KdaFp8Pool, "kda_seqs": kda.KdaSeqs}[s]
            assert getattr(cls, f).offset == int(val), key


def fake_params(B=4, N=8, H=12):
    """Parameters pointing at aligned fake host addresses; only ever used with
    calls that validation rejects, or with B = 0."""
    p = kda.KdaParams()
    p.B, p.H, p.K, p.V, p.N = B, H, 128, 128, N
    base = 1 << 32
    for i, name in enumerate(("q", "k", "v", "g_raw")):
        setattr(p, name, kda.KdaView(base + i * (1 << 24), 3 * H * 128, 0, 128))
    p.beta_logit = kda.KdaView(base + 5 * (1 << 24), H, 0, 1)
    p.A_log = base + 6 * (1 << 24)
    p.dt_bias = base + 7 * (1 << 24)
    p.lower_bound, p.scale = -5.0, 1.0
    p.state = base + (1 << 30)
    p.state_slot_stride = H * 128 * 128
    p.state_indices = base + 8 * (1 << 24)
    p.out = base + 9 * (1 << 24)
    p.out_b_stride, p.out_t_stride, p.out_h_stride = H * 128, 0, 128
    p.error_word = None
    p.config_override = -1
    return p


def status(lib, p, T=None, ring=None):
    if ring is not None:
        return lib.kda_verify_ring(ctypes.byref(p), T, ctypes.byref(ring), None)
    if T is None:
        return lib.kda_decode(ctypes.byref(p), None)
    return lib.kda_verify(ctypes.byref(p), T, None)


@no_gpu
def test_null_params(lib):
    assert lib.kda_decode(None, None) == kda.KDA_EINVAL
    assert "NULL" in kda.kda_last_error()


@no_gpu
def test_empty_batch_is_ok_without_launch(lib):
    p = fake_params(B=0)
    assert status(lib, p) == kda.KDA_OK
    assert kda.kda_last_error() == ""
    assert status(lib, p, T=8) == kda.KDA_OK


@no_gpu
@pytest.mark.parametrize("mutate,expect,msg", [
    (lambda p: setattr(p, "K", 64), kda.KDA_EUNSUPPORTED, "128"),
    (lambda p: setattr(p, "V", 256), kda.KDA_EUNSUPPORTED, "128"),
    (lambda p: setattr(p, "H", 0), kda.KDA_EUNSUPPORTED, "H"),
    (lambda p: setattr(p, "H", 65), kda.KDA_EUNSUPPORTED, "H"),
    (lambda p: setattr(p, "B", -1), kda.KDA_EINVAL, "B"),
    (lambda p: setattr(p, "N", -3), kda.KDA_EINVAL, "N"),
    (lambda p: setattr(p, "q", kda.KdaView(0, 1, 0, 1)), kda.KDA_EINVAL, "q.ptr"),
    (lambda p: setattr(p, "k", kda.KdaView((1 << 32) + 1, 1, 0, 1)), kda.KDA_EINVAL, "aligned"),
    (lambda p: setattr(p, "v", kda.KdaView(1 << 32, -1, 0, 1)), kda.KDA_EINVAL, "negative"),
    (lambda p: setattr(p, "A_log", (1 << 32) + 2), kda.KDA_EINVAL, "A_log"),
    (lambda p: setattr(p, "dt_bias", None), kda.KDA_EINVAL, "dt_bias"),
    (lambda p: setattr(p, "state_indices", None), kda.KDA_EINVAL, "state_indices"),
    (lambda p: setattr(p, "out", None), kda.KDA_EINVAL, "out"),
    (lambda p: setattr(p, "out_h_stride", -128), kda.KDA_EINVAL, "negative"),
    (lambda p: setattr(p, "state", None), kda.KDA_EINVAL, "state"),
    (lambda p: setattr(p, "state", (1 << 32) + 1), kda.KDA_EINVAL, "state"),
    (lambda p: setattr(p, "state_slot_stride", 100), kda.KDA_EINVAL, "slot_stride"),
    (lambda p: setattr(p, "config_override", 99), kda.KDA_EINVAL, "config_override"),
    (lambda p: setattr(p, "lower_bound", float("nan")), kda.KDA_EINVAL, "lower_bound"),
    (lambda p: setattr(p, "scale", float("inf")), kda.KDA_EINVAL, "scale"),
    (lambda p: setattr(p, "out", p.state + 4096), kda.KDA_EINVAL, "overlaps"),
    (lambda p: setattr(p, "error_word", (1 << 32) + 2), kda.KDA_EINVAL, "error_word"),
    (lambda p: setattr(p, "gate_mode", 2), kda.KDA_EINVAL, "gate_mode"),
    # A_log and dt_bias are not needed in the pre-computed convention: the next check fires instead
    (lambda p: (setattr(p, "gate_mode", 1), setattr(p, "A_log", None), setattr(p, "dt_bias", None),
                setattr(p, "state_indices", None)), kda.KDA_EINVAL, "state_indices"),
])
def test_decode_rejects(lib, mutate, expect, msg):
    p = fake_params()
    mutate(p)
    assert status(lib, p) == expect
    assert msg in kda.kda_last_error()


@no_gpu
def test_tensor_core_configuration_is_verify_only(lib):
    p = fake_params()
    p.config_override = 4
    assert status(lib, p) == kda.KDA_EUNSUPPORTED  # decode
    assert "T > 1" in kda.kda_last_error()
    assert status(lib, p, T=1) == kda.KDA_EUNSUPPORTED
    assert status(lib, p, T=8, ring=ring()) == kda.KDA_EUNSUPPORTED  # the ring takes whole-head tiles only
    assert kda.kda_config_tile_v(4) == 128


@no_gpu
def test_verify_token_range(lib):
    for T in (0, -1, 17):
        assert status(lib, fake_params(), T=T) == kda.KDA_EUNSUPPORTED
        assert "T" in kda.kda_last_error()


def ring(W=32, flush_min=9, N=8, H=12):
    r = kda.KdaRingParams()
    base = 1 << 36
    r.k_cache, r.u_cache, r.g_cache = base, base + (1 << 28), base + (1 << 29)
    r.k_slot_stride = r.u_slot_stride = r.g_slot_stride = H * W * 128
    r.hist_len = base + (1 << 30)
    r.W, r.flush_min, r.restart_hist_on_flush = W, flush_min, 1
    return r


@no_gpu
@pytest.mark.parametrize("T,mut,expect,msg", [
    (8, lambda r: setattr(r, "W", 0), kda.KDA_EUNSUPPORTED, "W"),
    (8, lambda r: setattr(r, "W", 65), kda.KDA_EUNSUPPORTED, "W"),
    (8, lambda r: setattr(r, "W", 4), kda.KDA_EINVAL, "exceeds"),
    (8, lambda r: setattr(r, "flush_min", 0), kda.KDA_EINVAL, "flush_min"),
    (8, lambda r: setattr(r, "flush_min", 26), kda.KDA_EINVAL, "flush_min"),
    (8, lambda r: setattr(r, "k_cache", None), kda.KDA_EINVAL, "NULL"),
    (8, lambda r: setattr(r, "g_cache", (1 << 36) + 8), kda.KDA_EINVAL, "16-byte"),
    (8, lambda r: setattr(r, "u_slot_stride", 12), kda.KDA_EINVAL, "stride"),
    (8, lambda r: setattr(r, "cache_base", (1 << 36) + 2), kda.KDA_EINVAL, "cache_base"),
])
def test_ring_rejects(lib, T, mut, expect, msg):
    p = fake_params()
    r = ring()
    mut(r)
    assert status(lib, p, T=T, ring=r) == expect
    assert msg in kda.kda_last_error()


@no_gpu
@pytest.mark.parametrize("config", [0, 1, 2])
def test_ring_rejects_partial_head_tiles(lib, config):
    p = fake_params()
    p.config_override = config
    assert status(lib, p, T=8, ring=ring()) == kda.KDA_EUNSUPPORTED
    assert "whole-head" in kda.kda_last_error()


@no_gpu
def test_ring_null_and_empty(lib):
    p = fake_params()
    assert lib.kda_verify_ring(ctypes.byref(p), 8, None, None) == kda.KDA_EINVAL
    p0 = fake_params(B=0)
    assert status(lib, p0, T=8, ring=ring()) == kda.KDA_OK


def test_config_table_and_selector(lib):
    n = kda.kda_num_configs()
    tiles = [kda.kda_config_tile_v(i) for i in range(n)]
    assert tiles == sorted(tiles) and all(128 % t == 0 and t % 16 == 0 for t in tiles)
    assert kda.kda_config_tile_v(-1) == -1 and kda.kda_config_tile_v(n) == -1
    assert kda.kda_select_config(-1, 1) == -1 and kda.kda_select_config(4, 0) == -1
    assert kda.kda_select_config(4, 17) == -1
    prev = 0
    for B in (1, 2, 8, 16, 32, 64, 128, 256, 512, 4096):
        c = kda.kda_select_config(B, 1)
        assert 0 <= c < n and c >= prev  # tiles never shrink as the batch grows
        prev = c
    assert kda.kda_config_tile_v(kda.kda_select_config(512, 1)) == 128
    for B in (0, 1, 2, 8, 16, 32, 64, 128, 512, 4096):  # the ring kernel always takes whole heads
        for T in (1, 4, 8, 16):
            assert kda.kda_config_tile_v(kda.kda_select_ring_config(B, T)) == 128
    assert kda.kda_select_ring_config(-1, 8) == -1 and kda.kda_select_ring_config(4, 17) == -1


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(kda, "_lib", None)
    monkeypatch.setattr(kda, "lib_path", lambda: str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        kda.load_library()


@no_gpu
def test_fp8_decode_validation(lib):
    """kda_decode_fp8 rejects a missing pool or scale array, short scale slot
    strides, the tensor-core configuration and out overlapping the scales."""
    p = fake_params()
    call = lambda f: lib.kda_decode_fp8(ctypes.byref(p), None if f is None else ctypes.byref(f), None)  # noqa: E731
    assert call(None) == kda.KDA_EINVAL and "fp8 pool" in kda.kda_last_error()
    assert call(kda.KdaFp8Pool(None, 12 * 128)) == kda.KDA_EINVAL and "scale" in kda.kda_last_error()
    assert call(kda.KdaFp8Pool(p.state + (1 << 26) + 2, 12 * 128)) == kda.KDA_EINVAL  # 2-byte aligned
    assert call(kda.KdaFp8Pool(p.state + (1 << 26), 12 * 128 - 1)) == kda.KDA_EINVAL
    assert "scale_slot_stride" in kda.kda_last_error()
    f = kda.KdaFp8Pool(p.out, 12 * 128)  # the scales where the output goes
    assert call(f) == kda.KDA_EINVAL and "overlaps" in kda.kda_last_error()
    p.config_override = 4
    assert call(kda.KdaFp8Pool(p.state + (1 << 26), 12 * 128)) == kda.KDA_EUNSUPPORTED
    p.config_override = -1
    p.B = 0
    assert call(kda.KdaFp8Pool(p.state + (1 << 26), 12 * 128)) == kda.KDA_OK


@no_gpu
def test_prefill_validation(lib):
    """kda_prefill rejects missing arguments, a negative sequence count, a
    configuration index past the last and an unaligned cu_seqlens; an empty
    call launches nothing; the selector picks the chunked tensor-core kernel."""
    p = fake_params()
    call = lambda sq: lib.kda_prefill(ctypes.byref(p), None if sq is None else ctypes.byref(sq), None)  # noqa: E731
    cu = (1 << 32) + 10 * (1 << 24)
    assert lib.kda_prefill(None, ctypes.byref(kda.KdaSeqs(cu, 1)), None) == kda.KDA_EINVAL
    assert call(None) == kda.KDA_EINVAL and "seqs" in kda.kda_last_error()
    assert call(kda.KdaSeqs(cu, -1)) == kda.KDA_EINVAL and "num_seqs" in kda.kda_last_error()
    assert call(kda.KdaSeqs(None, 2)) == kda.KDA_EINVAL and "cu_seqlens" in kda.kda_last_error()
    assert call(kda.KdaSeqs(cu + 2, 2)) == kda.KDA_EINVAL and "cu_seqlens" in kda.kda_last_error()
    p.config_override = 5
    assert call(kda.KdaSeqs(cu, 2)) == kda.KDA_EINVAL and "config_override" in kda.kda_last_error()
    p.config_override = -1
    p.K = 64
    assert call(kda.KdaSeqs(cu, 2)) == kda.KDA_EUNSUPPORTED
    p.K = 128
    assert call(kda.KdaSeqs(None, 0)) == kda.KDA_OK  # no sequence: nothing to do
    p.B = 0
    assert call(kda.KdaSeqs(cu, 2)) == kda.KDA_OK  # no token rows: nothing launched
    assert [lib.kda_select_prefill_config(s, 12) for s in (1, 8, 512)] == [4, 4, 4]
    assert lib.kda_select_prefill_config(-1, 12) == -1 and lib.kda_select_prefill_config(1, 0) == -1


@no_gpu
def test_prefill_ws_validation(lib):
    """kda_prefill_ws: configuration 5 needs a workspace of the size
    kda_prefill_workspace_bytes gives, 16-byte aligned and apart from the
    call's other buffers; other configurations go to kda_prefill's checks; the
    selector takes the two stages from an average of 512 tokens per
    sequence, in one launch (6) for at most 32 sequences and 64 chains."""
    p = fake_params(B=40)
    cu = (1 << 32) + 10 * (1 << 24)
    sq = kda.KdaSeqs(cu, 2)
    images = ((40 + 15) // 16 + 2) * 12
    need = images * 45568 + (images * 4 + 15) // 16 * 16  # the chunk images, then their ready flags
    assert lib.kda_prefill_workspace_bytes(40, 2, 12) == need
    assert [lib.kda_prefill_workspace_bytes(*a) for a in ((0, 2, 12), (40, 0, 12), (40, 2, 0), (-1, 2, 12))] == [0] * 4
    ws = (1 << 32) + 32 * (1 << 24)

    def call(w, n, s=sq):
        return lib.kda_prefill_ws(ctypes.byref(p), None if s is None else ctypes.byref(s), w, n, None)

    p.config_override = 5
    assert call(None, need) == kda.KDA_EINVAL and "workspace" in kda.kda_last_error()
    assert call(ws + 8, need) == kda.KDA_EINVAL and "aligned" in kda.kda_last_error()
    assert call(ws, need - 16) == kda.KDA_EINVAL and "workspace_bytes" in kda.kda_last_error()
    assert call(p.out, need) == kda.KDA_EINVAL and "overlaps out" in kda.kda_last_error()
    assert call(p.state, need) == kda.KDA_EINVAL and "state pool" in kda.kda_last_error()
    assert call(p.q.ptr, need) == kda.KDA_EINVAL and "overlaps q" in kda.kda_last_error()
    assert call(ws, need, None) == kda.KDA_EINVAL and "seqs" in kda.kda_last_error()
    assert call(ws, need, kda.KdaSeqs(None, 2)) == kda.KDA_EINVAL and "cu_seqlens" in kda.kda_last_error()
    assert call(ws, need, kda.KdaSeqs(cu, -1)) == kda.KDA_EINVAL
    assert call(None, 0, kda.KdaSeqs(None, 0)) == kda.KDA_OK  # no sequence: nothing to do
    p.K = 64
    assert call(ws, need) == kda.KDA_EUNSUPPORTED
    p.K = 128
    p.config_override = 6  # the one-launch schedule: the same workspace checks
    assert call(None, need) == kda.KDA_EINVAL and "workspace" in kda.kda_last_error()
    assert call(ws, need - 16) == kda.KDA_EINVAL and "workspace_bytes" in kda.kda_last_error()
    p.config_override = 7
    assert call(ws, need) == kda.KDA_EINVAL and "config_override" in kda.kda_last_error()
    p.config_override = 4  # a single-kernel configuration: kda_prefill's checks, no workspace needed
    assert call(None, 0, kda.KdaSeqs(cu + 2, 2)) == kda.KDA_EINVAL and "cu_seqlens" in kda.kda_last_error()
    p.config_override = 5
    p.B = 0
    assert call(None, 0) == kda.KDA_OK  # no token rows: nothing launched
    sel = lib.kda_select_prefill_ws_config
    assert [sel(4096, 1, 12), sel(16384, 1, 16), sel(512 * 3, 3, 12), sel(512 * 4, 4, 16)] == [6, 6, 6, 6]
    assert [sel(8 * 2048, 8, 12), sel(512 * 40, 40, 1), sel(512 * 5, 5, 13)] == [5, 5, 5]
    assert [sel(64 * 256, 64, 12), sel(512 * 16, 512, 12), sel(511 * 10, 10, 12), sel(100, 0, 12)] == [4, 4, 4, 4]
    assert sel(-1, 1, 12) == -1 and sel(16, -1, 12) == -1 and sel(16, 1, 0) == -1
