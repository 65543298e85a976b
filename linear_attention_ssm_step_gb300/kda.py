"""Thin ctypes binding of libkda_gb300.so (include/kda.h).

Argument marshalling only: torch tensors supply device pointers, strides and
the current CUDA stream; every step of the computation runs in the library's
kernels. There is no CPU or fallback path: if the library is missing or a
call is rejected, this module raises.
"""

import ctypes
import os

import torch

from . import _build

KDA_OK, KDA_EINVAL, KDA_EUNSUPPORTED, KDA_ELAUNCH = 0, 1, 2, 3
KDA_ERR_HIST_LEN = 1
KDA_ERR_TIMEOUT = 2
KDA_ERR_CACHE_BASE = 4
KDA_ERR_SEQLENS = 8
KDA_MAX_T = 16
KDA_GATE_RAW, KDA_GATE_PRECOMPUTED = 0, 1
STATUS_NAMES = {0: "KDA_OK", 1: "KDA_EINVAL", 2: "KDA_EUNSUPPORTED", 3: "KDA_ELAUNCH"}


class KdaError(RuntimeError):
    def __init__(self, status, message):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class KdaView(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("b_stride", ctypes.c_int64),
                ("t_stride", ctypes.c_int64), ("h_stride", ctypes.c_int64)]


class KdaParams(ctypes.Structure):
    _fields_ = [
        ("B", ctypes.c_int32), ("H", ctypes.c_int32), ("K", ctypes.c_int32),
        ("V", ctypes.c_int32), ("N", ctypes.c_int32),
        ("q", KdaView), ("k", KdaView), ("v", KdaView), ("g_raw", KdaView),
        ("beta_logit", KdaView),
        ("A_log", ctypes.c_void_p), ("dt_bias", ctypes.c_void_p),
        ("lower_bound", ctypes.c_float), ("scale", ctypes.c_float),
        ("state", ctypes.c_void_p), ("state_slot_stride", ctypes.c_int64),
        ("state_indices", ctypes.c_void_p),
        ("out", ctypes.c_void_p), ("out_b_stride", ctypes.c_int64),
        ("out_t_stride", ctypes.c_int64), ("out_h_stride", ctypes.c_int64),
        ("error_word", ctypes.c_void_p), ("config_override", ctypes.c_int32),
        ("gate_mode", ctypes.c_int32),
    ]


class KdaRingParams(ctypes.Structure):
    _fields_ = [
        ("k_cache", ctypes.c_void_p), ("u_cache", ctypes.c_void_p), ("g_cache", ctypes.c_void_p),
        ("k_slot_stride", ctypes.c_int64), ("u_slot_stride", ctypes.c_int64),
        ("g_slot_stride", ctypes.c_int64),
        ("hist_len", ctypes.c_void_p), ("W", ctypes.c_int32), ("flush_min", ctypes.c_int32),
        ("restart_hist_on_flush", ctypes.c_int32), ("cache_base", ctypes.c_void_p),
    ]


class KdaFp8Pool(ctypes.Structure):
    """kda_fp8_pool of include/kda_fp8.h."""

    _fields_ = [("scale", ctypes.c_void_p), ("scale_slot_stride", ctypes.c_int64)]


class KdaSeqs(ctypes.Structure):
    """kda_seqs of include/kda_prefill.h."""

    _fields_ = [("cu_seqlens", ctypes.c_void_p), ("num_seqs", ctypes.c_int32)]


EXPORTS = {
    "kda_decode": ([ctypes.POINTER(KdaParams), ctypes.c_void_p], ctypes.c_int),
    "kda_decode_fp8": ([ctypes.POINTER(KdaParams), ctypes.POINTER(KdaFp8Pool), ctypes.c_void_p], ctypes.c_int),
    "kda_verify_fp8": ([ctypes.POINTER(KdaParams), ctypes.c_int32, ctypes.POINTER(KdaFp8Pool), ctypes.c_void_p],
                       ctypes.c_int),
    "kda_verify_ring_fp8": ([ctypes.POINTER(KdaParams), ctypes.c_int32, ctypes.POINTER(KdaRingParams),
                             ctypes.POINTER(KdaFp8Pool), ctypes.c_void_p], ctypes.c_int),
    "kda_verify": ([ctypes.POINTER(KdaParams), ctypes.c_int32, ctypes.c_void_p], ctypes.c_int),
    "kda_prefill": ([ctypes.POINTER(KdaParams), ctypes.POINTER(KdaSeqs), ctypes.c_void_p], ctypes.c_int),
    "kda_select_prefill_config": ([ctypes.c_int32, ctypes.c_int32], ctypes.c_int32),
    "kda_prefill_ws": ([ctypes.POINTER(KdaParams), ctypes.POINTER(KdaSeqs), ctypes.c_void_p, ctypes.c_size_t,
                        ctypes.c_void_p], ctypes.c_int),
    "kda_prefill_workspace_bytes": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32], ctypes.c_size_t),
    "kda_prefill_static": ([ctypes.POINTER(KdaParams), ctypes.POINTER(KdaSeqs), ctypes.c_void_p], ctypes.c_int),
    "kda_select_prefill_ws_config": ([ctypes.c_int32, ctypes.c_int32, ctypes.c_int32], ctypes.c_int32),
    "kda_verify_ring": ([ctypes.POINTER(KdaParams), ctypes.c_int32, ctypes.POINTER(KdaRingParams),
                         ctypes.c_void_p], ctypes.c_int),
    "kda_num_configs": ([], ctypes.c_int32),
    "kda_config_tile_v": ([ctypes.c_int32], ctypes.c_int32),
    "kda_select_config": ([ctypes.c_int32, ctypes.c_int32], ctypes.c_int32),
    "kda_select_ring_config": ([ctypes.c_int32, ctypes.c_int32], ctypes.c_int32),
    "kda_last_error": ([], ctypes.c_char_p),
}

_lib = None


def lib_path():
    return _build.LIB_PATH


def bind_library(path):
    """Open a build of the library at `path` with the C signatures of EXPORTS set."""
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is not built; run __graft_entry__.build() first")
    lib = ctypes.CDLL(path)
    for name, (args, res) in EXPORTS.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    return lib


def load_library():
    """Load libkda_gb300.so (built by __graft_entry__.build()); raise if it is absent."""
    global _lib
    if _lib is None:
        _lib = bind_library(lib_path())
    return _lib


def _check(status):
    if status != KDA_OK:
        raise KdaError(status, load_library().kda_last_error().decode())


def _need(t, name, dtype):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")


def _view(t, name, has_T, D):
    """KdaView of [B, H, D] (has_T False) or [B, T, H, D]; D == 1 drops the last dim."""
    _need(t, name, torch.bfloat16)
    want = (3 if has_T else 2) + (1 if D > 1 else 0)
    if t.dim() != want:
        raise ValueError(f"{name} must have {want} dims, got shape {tuple(t.shape)}")
    if D > 1 and (t.shape[-1] != D or t.stride(-1) != 1):
        raise ValueError(f"{name} must have a contiguous last dim of {D}")
    s = t.stride()
    if has_T:
        return KdaView(t.data_ptr(), s[0], s[1], s[2])
    return KdaView(t.data_ptr(), s[0], 0, s[1])


def _stream_handle(stream, device):
    if stream is None:
        stream = torch.cuda.current_stream(device)
    return ctypes.c_void_p(stream.cuda_stream)


def _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
            lower_bound, scale, error_word, config_override, gate_mode, state_dtype=torch.bfloat16,
            n_indices=None):
    has_T = T is not None
    B = q.shape[0]
    n_idx = B if n_indices is None else n_indices
    H = q.shape[-2]
    _need(state, "state", state_dtype)
    if state.dim() != 4 or state.shape[1:] != (H, 128, 128):
        raise ValueError(f"state must be [N, {H}, 128, 128], got {tuple(state.shape)}")
    if state.stride()[1:] != (128 * 128, 128, 1):
        raise ValueError("each state slot must be contiguous [H][V][K]")
    _need(state_indices, "state_indices", torch.int32)
    if state_indices.shape != (n_idx,) or (n_idx > 0 and state_indices.stride(0) != 1):
        raise ValueError(f"state_indices must be a contiguous [{n_idx}] tensor")
    if gate_mode == KDA_GATE_RAW or A_log is not None:
        _need(A_log, "A_log", torch.float32)
        if A_log.numel() != H or not A_log.is_contiguous():
            raise ValueError("A_log must be a contiguous [H] tensor")
    if gate_mode == KDA_GATE_RAW or dt_bias is not None:
        _need(dt_bias, "dt_bias", torch.float32)
        if dt_bias.numel() != H * 128 or not dt_bias.is_contiguous():
            raise ValueError("dt_bias must be a contiguous [H, 128] tensor")
    _need(out, "out", torch.bfloat16)
    if out.stride(-1) != 1:
        raise ValueError("out must have a contiguous last dim")
    so = out.stride()
    p = KdaParams()
    p.B, p.H, p.K, p.V, p.N = B, H, 128, 128, state.shape[0]
    p.q = _view(q, "q", has_T, 128)
    p.k = _view(k, "k", has_T, 128)
    p.v = _view(v, "v", has_T, 128)
    p.g_raw = _view(g_raw, "g_raw", has_T, 128)
    p.beta_logit = _view(beta_logit, "beta_logit", has_T, 1)
    p.A_log = None if A_log is None else A_log.data_ptr()
    p.dt_bias = None if dt_bias is None else dt_bias.data_ptr()
    p.lower_bound = lower_bound
    p.scale = scale
    p.state = state.data_ptr()
    p.state_slot_stride = state.stride(0)
    p.state_indices = state_indices.data_ptr()
    p.out = out.data_ptr()
    if has_T:
        p.out_b_stride, p.out_t_stride, p.out_h_stride = so[0], so[1], so[2]
    else:
        p.out_b_stride, p.out_t_stride, p.out_h_stride = so[0], 0, so[1]
    if error_word is not None:
        _need(error_word, "error_word", torch.int32)
        p.error_word = error_word.data_ptr()
    p.config_override = config_override
    p.gate_mode = gate_mode
    return p


def kda_decode(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
               lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
               stream=None):
    """T=1 decode. q, k, v, g_raw: bf16 [B, H, 128] views (any row and head stride);
    beta_logit: bf16 [B, H]; state: bf16 [N, H, 128, 128] pool updated in place;
    returns out bf16 [B, H, 128]. With gate_mode=KDA_GATE_PRECOMPUTED, g_raw holds
    log-space g, beta_logit holds beta, and A_log / dt_bias may be None."""
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 128), dtype=torch.bfloat16, device=q.device)
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, None,
                lower_bound, scale, error_word, config_override, gate_mode)
    _check(load_library().kda_decode(ctypes.byref(p), _stream_handle(stream, q.device)))
    return out


class PreparedCall:
    """A library call bound to fixed tensors: argument checks and the C parameter
    struct are done once, and each call() launches the kernel on the tensors'
    current contents, on the stream given (or current) at preparation. The bound
    tensors must stay alive and keep their storage; `out` is the output tensor.
    For serving loops that refill the same input buffers every step."""

    def __init__(self, fn, args, out, keep):
        self._fn, self._args = fn, args  # ctypes arguments, structs passed by reference
        self.out = out
        self._keep = keep  # the structs and bound tensors, kept alive with the call

    def __call__(self):
        _check(self._fn(*self._args))
        return self.out


def prepare_decode(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                   lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                   stream=None):
    """kda_decode bound to these tensors (see PreparedCall); same arguments."""
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 128), dtype=torch.bfloat16, device=q.device)
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, None,
                lower_bound, scale, error_word, config_override, gate_mode)
    keep = (p, state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, error_word)
    return PreparedCall(load_library().kda_decode, (ctypes.byref(p), _stream_handle(stream, q.device)), out, keep)


def kda_decode_fp8(codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                   lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                   stream=None):
    """T=1 decode on an fp8 state pool (include/kda_fp8.h): codes uint8
    [N, H, 128, 128] (E4M3) and scales fp32 [N, H, 128] (powers of two), both
    updated in place for active rows; other arguments as kda_decode."""
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 128), dtype=torch.bfloat16, device=q.device)
    p = _params(codes, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, None,
                lower_bound, scale, error_word, config_override, gate_mode, state_dtype=torch.uint8)
    f = _fp8_pool(codes, scales)
    _check(load_library().kda_decode_fp8(ctypes.byref(p), ctypes.byref(f), _stream_handle(stream, q.device)))
    return out


def kda_verify_fp8(codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                   lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                   stream=None):
    """T-token verify on an fp8 state pool (include/kda_fp8.h): the pool as for
    kda_decode_fp8, the token views and output as for kda_verify
    ([B, T, H, 128]); equal to T kda_decode_fp8 calls, bit for bit."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=q.device)
    p = _params(codes, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
                lower_bound, scale, error_word, config_override, gate_mode, state_dtype=torch.uint8)
    f = _fp8_pool(codes, scales)
    _check(load_library().kda_verify_fp8(ctypes.byref(p), T, ctypes.byref(f), _stream_handle(stream, q.device)))
    return out


def kda_verify_ring_fp8(codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                        k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush=True,
                        out=None, lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1,
                        gate_mode=KDA_GATE_RAW, stream=None, cache_base=None):
    """Ring-cache verify with replay and fold on an fp8 checkpoint pool
    (include/kda_fp8.h): codes and scales as kda_decode_fp8's (a fold
    requantizes the checkpoint in place), the ring and the rest as
    kda_verify_ring's."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=q.device)
    p = _params(codes, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
                lower_bound, scale, error_word, config_override, gate_mode, state_dtype=torch.uint8)
    r = _ring_params(codes, H, k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush, cache_base)
    f = _fp8_pool(codes, scales)
    _check(load_library().kda_verify_ring_fp8(ctypes.byref(p), T, ctypes.byref(r), ctypes.byref(f),
                                              _stream_handle(stream, q.device)))
    return out


def _fp8_pool(codes, scales):
    _need(scales, "scales", torch.float32)
    if scales.dim() != 3 or scales.shape != codes.shape[:3] or scales.stride()[1:] != (128, 1):
        raise ValueError(f"scales must be [N, H, 128] with contiguous slots, got {tuple(scales.shape)}")
    return KdaFp8Pool(scales.data_ptr(), scales.stride(0))


def prepare_decode_fp8(codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                       lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                       stream=None):
    """kda_decode_fp8 bound to these tensors (see PreparedCall); same arguments."""
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 128), dtype=torch.bfloat16, device=q.device)
    p = _params(codes, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, None,
                lower_bound, scale, error_word, config_override, gate_mode, state_dtype=torch.uint8)
    f = _fp8_pool(codes, scales)
    keep = (p, f, codes, scales, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, error_word)
    args = (ctypes.byref(p), ctypes.byref(f), _stream_handle(stream, q.device))
    return PreparedCall(load_library().kda_decode_fp8, args, out, keep)


def kda_verify(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
               lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
               stream=None):
    """T-token verify. q, k, v, g_raw: bf16 [B, T, H, 128]; beta_logit: bf16 [B, T, H];
    returns out bf16 [B, T, H, 128]."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=q.device)
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
                lower_bound, scale, error_word, config_override, gate_mode)
    _check(load_library().kda_verify(ctypes.byref(p), T, _stream_handle(stream, q.device)))
    return out


def prepare_verify(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                   lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                   stream=None):
    """kda_verify bound to these tensors (see PreparedCall); same arguments."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=q.device)
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
                lower_bound, scale, error_word, config_override, gate_mode)
    keep = (p, state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, error_word)
    return PreparedCall(load_library().kda_verify, (ctypes.byref(p), T, _stream_handle(stream, q.device)), out,
                        keep)


def kda_verify_ring(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                    k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush=True,
                    out=None, lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1,
                    gate_mode=KDA_GATE_RAW, stream=None, cache_base=None):
    """Ring-cache verify with replay and fold. k_cache, u_cache: bf16 [N, H, W, 128];
    g_cache: fp32 [N, H, W, 128]; hist_len: int32 [N]; cache_base: optional int32 [N]
    (ring position P of slot n is entry (cache_base[n] + P) mod W). Returns out
    bf16 [B, T, H, 128]."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=q.device)
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
                lower_bound, scale, error_word, config_override, gate_mode)
    r = _ring_params(state, H, k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush, cache_base)
    _check(load_library().kda_verify_ring(ctypes.byref(p), T, ctypes.byref(r),
                                          _stream_handle(stream, q.device)))
    return out


def prepare_verify_ring(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                        k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush=True,
                        out=None, lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1,
                        gate_mode=KDA_GATE_RAW, stream=None, cache_base=None):
    """kda_verify_ring bound to these tensors (see PreparedCall); same arguments."""
    B, T, H = q.shape[0], q.shape[1], q.shape[2]
    if out is None:
        out = torch.empty((B, T, H, 128), dtype=torch.bfloat16, device=q.device)
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, T,
                lower_bound, scale, error_word, config_override, gate_mode)
    r = _ring_params(state, H, k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush, cache_base)
    keep = (p, r, state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, k_cache, u_cache, g_cache,
            hist_len, cache_base, error_word)
    args = (ctypes.byref(p), T, ctypes.byref(r), _stream_handle(stream, q.device))
    return PreparedCall(load_library().kda_verify_ring, args, out, keep)


def _ring_params(state, H, k_cache, u_cache, g_cache, hist_len, flush_min, restart_hist_on_flush, cache_base):
    _need(k_cache, "k_cache", torch.bfloat16)
    _need(u_cache, "u_cache", torch.bfloat16)
    _need(g_cache, "g_cache", torch.float32)
    _need(hist_len, "hist_len", torch.int32)
    W = k_cache.shape[2]
    for name, t in (("k_cache", k_cache), ("u_cache", u_cache), ("g_cache", g_cache)):
        if t.dim() != 4 or t.shape[1:] != (H, W, 128) or t.stride()[1:] != (W * 128, 128, 1):
            raise ValueError(f"{name} must be [N, {H}, {W}, 128] with contiguous slots")
    if hist_len.shape != (state.shape[0],) or not hist_len.is_contiguous():
        raise ValueError("hist_len must be a contiguous [N] tensor")
    if cache_base is not None:
        _need(cache_base, "cache_base", torch.int32)
        if cache_base.shape != (state.shape[0],) or not cache_base.is_contiguous():
            raise ValueError("cache_base must be a contiguous [N] tensor")
    r = KdaRingParams()
    r.k_cache, r.u_cache, r.g_cache = k_cache.data_ptr(), u_cache.data_ptr(), g_cache.data_ptr()
    r.k_slot_stride, r.u_slot_stride, r.g_slot_stride = k_cache.stride(0), u_cache.stride(0), g_cache.stride(0)
    r.hist_len = hist_len.data_ptr()
    r.W, r.flush_min, r.restart_hist_on_flush = W, flush_min, int(bool(restart_hist_on_flush))
    r.cache_base = None if cache_base is None else cache_base.data_ptr()
    return r


def kda_prefill(state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                stream=None, workspace=None):
    """Varlen prefill (include/kda_prefill.h). q, k, v, g_raw: bf16 [L, H, 128]
    views with one row per token (any row and head stride); beta_logit: bf16
    [L, H]; cu_seqlens: int32 [S + 1] on the device, sequence i owning rows
    cu_seqlens[i] .. cu_seqlens[i+1]-1; state_indices: int32 [S], one slot per
    sequence; state: bf16 [N, H, 128, 128] pool, read as each sequence's
    initial state and overwritten with its final state. Returns out bf16
    [L, H, 128] (rows no sequence covers are left as they were).
    workspace: None (kda_prefill, configurations 0-4) or a device byte tensor
    of at least prefill_workspace_bytes(L, S, H) (kda_prefill_ws, which may
    then choose the two-stage configuration 5)."""
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 128), dtype=torch.bfloat16, device=q.device)
    fn, args, _ = _prefill_call(state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                                out, lower_bound, scale, error_word, config_override, gate_mode, stream, workspace)
    _check(fn(*args))
    return out


def _prefill_call(state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias, out,
                  lower_bound, scale, error_word, config_override, gate_mode, stream, workspace):
    _need(cu_seqlens, "cu_seqlens", torch.int32)
    if cu_seqlens.dim() != 1 or cu_seqlens.shape[0] < 1 or not cu_seqlens.is_contiguous():
        raise ValueError("cu_seqlens must be a contiguous [S + 1] tensor")
    S = cu_seqlens.shape[0] - 1
    p = _params(state, state_indices, q, k, v, g_raw, beta_logit, A_log, dt_bias, out, None,
                lower_bound, scale, error_word, config_override, gate_mode, n_indices=S)
    sq = KdaSeqs(cu_seqlens.data_ptr(), S)
    keep = (p, sq, state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias, error_word,
            workspace)
    lib = load_library()
    handle = _stream_handle(stream, q.device)
    if workspace is None:
        return lib.kda_prefill, (ctypes.byref(p), ctypes.byref(sq), handle), keep
    _need(workspace, "workspace", torch.uint8)
    if not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous byte tensor")
    return lib.kda_prefill_ws, (ctypes.byref(p), ctypes.byref(sq), workspace.data_ptr(), workspace.numel(),
                                handle), keep


def prepare_prefill(state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias, out=None,
                    lower_bound=-5.0, scale=1.0, error_word=None, config_override=-1, gate_mode=KDA_GATE_RAW,
                    stream=None, workspace=None):
    """kda_prefill bound to these tensors (see PreparedCall); same arguments. The
    sequence count is fixed by cu_seqlens' length; its contents may change."""
    if out is None:
        out = torch.empty((q.shape[0], q.shape[1], 128), dtype=torch.bfloat16, device=q.device)
    fn, args, keep = _prefill_call(state, state_indices, cu_seqlens, q, k, v, g_raw, beta_logit, A_log, dt_bias,
                                   out, lower_bound, scale, error_word, config_override, gate_mode, stream,
                                   workspace)
    return PreparedCall(fn, args, out, keep)


def prefill_workspace_bytes(B, num_seqs, H):
    """Bytes of the workspace kda_prefill_ws needs (include/kda_prefill.h)."""
    return int(load_library().kda_prefill_workspace_bytes(B, num_seqs, H))


def prefill_workspace(B, num_seqs, H, device):
    """A device workspace for prefill calls of up to B token rows and num_seqs sequences of H heads."""
    return torch.empty(max(16, prefill_workspace_bytes(B, num_seqs, H)), dtype=torch.uint8, device=device)


def kda_select_prefill_ws_config(B, num_seqs, H=12):
    return int(load_library().kda_select_prefill_ws_config(B, num_seqs, H))


def kda_select_prefill_config(num_seqs, H=12):
    return int(load_library().kda_select_prefill_config(num_seqs, H))


def kda_select_config(B, T=1):
    return load_library().kda_select_config(B, T)


def kda_select_ring_config(B, T=8):
    return load_library().kda_select_ring_config(B, T)


def kda_num_configs():
    return load_library().kda_num_configs()


def kda_config_tile_v(config):
    return load_library().kda_config_tile_v(config)


def kda_last_error():
    return load_library().kda_last_error().decode()
