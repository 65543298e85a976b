// kda_api.cu - the C ABI: host-side argument validation, launch-configuration
// selection and dispatch. No device memory is read, nothing is allocated and
// nothing synchronizes; kernels go on the caller's stream.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdint.h>
#include <stdio.h>

#include "kda.h"
#include "kda_fp8.h"
#include "kda_launch.h"
#include "kda_prefill.h"

namespace kda {
// T=1 decode on an fp8 pool (kda_fp8.cu); tile_v and bulk as launch_step's.
cudaError_t launch_decode_fp8(const kda_params& p, const kda_fp8_pool& f, int tile_v, bool bulk, cudaStream_t s);
// T-token verify on an fp8 pool (kda_fp8.cu); tile_v and bulk as above.
cudaError_t launch_verify_fp8(const kda_params& p, const kda_fp8_pool& f, int T, int tile_v, bool bulk,
                              cudaStream_t s);
// Varlen prefill token by token on the CUDA cores (kda_prefill.cu): num_seqs * H * (128 / tile_v) CTAs.
cudaError_t launch_prefill(const kda_params& p, const int32_t* cu, int num_seqs, int tile_v, bool bulk,
                           cudaStream_t s);
// Varlen prefill in chunks of 16 tokens on the tensor cores (kda_prefill_tc.cu), persistent.
cudaError_t launch_prefill_tc(const kda_params& p, const int32_t* cu, int num_seqs, bool bulk, cudaStream_t s);
}  // namespace kda

namespace {

thread_local char g_err[512] = "";

kda_status fail(kda_status s, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_err, sizeof(g_err), fmt, ap);
  va_end(ap);
  return s;
}

kda_status ok() {
  g_err[0] = '\0';
  return KDA_OK;
}

// Rows of V per CTA, by configuration index. Configuration 4 runs whole heads
// with the dot products on the tensor cores (T > 1 only).
constexpr int kTileV[] = {16, 32, 64, 128, 128};
constexpr int kTensorCoreConfig = 4;
constexpr int kNumConfigs = sizeof(kTileV) / sizeof(kTileV[0]);
// Prefill only, with a caller's workspace (kda_prefill_ws): the two stages in
// two launches (5) or in one cooperative launch (6).
constexpr int kChainConfig = 5;
constexpr int kFusedConfig = 6;
constexpr int kFusedMaxSeqs = 32;

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Byte extent [lo, hi) touched by a strided bf16 view [B][T][H][D].
void view_extent(const void* ptr, int B, int T, int H, int D, int64_t bs, int64_t ts, int64_t hs,
                 uintptr_t& lo, uintptr_t& hi) {
  lo = reinterpret_cast<uintptr_t>(ptr);
  const int64_t last = (int64_t)(B - 1) * bs + (int64_t)(T - 1) * ts + (int64_t)(H - 1) * hs + (D - 1);
  hi = lo + (uintptr_t)(last + 1) * 2;
}

bool overlaps(uintptr_t a0, uintptr_t a1, uintptr_t b0, uintptr_t b1) { return a0 < b1 && b0 < a1; }

kda_status check_view(const char* name, const kda_view& v, int D) {
  (void)D;
  if (v.ptr == nullptr) return fail(KDA_EINVAL, "%s.ptr is NULL", name);
  if (!aligned(v.ptr, 2)) return fail(KDA_EINVAL, "%s.ptr is not 2-byte aligned", name);
  if (v.b_stride < 0 || v.t_stride < 0 || v.h_stride < 0)
    return fail(KDA_EINVAL, "%s has a negative stride", name);
  return KDA_OK;
}

// Checks shared by the three calls. On success, sets *bulk.
kda_status check_params(const kda_params* p, int T, bool* bulk) {
  if (p == nullptr) return fail(KDA_EINVAL, "params is NULL");
  if (p->B < 0) return fail(KDA_EINVAL, "B = %d is negative", p->B);
  if (p->N < 0) return fail(KDA_EINVAL, "N = %d is negative", p->N);
  if (p->K != 128 || p->V != 128) return fail(KDA_EUNSUPPORTED, "K = %d, V = %d: only 128 x 128", p->K, p->V);
  if (p->H < 1 || p->H > 64) return fail(KDA_EUNSUPPORTED, "H = %d outside 1..64", p->H);
  if (T < 1 || T > KDA_MAX_T) return fail(KDA_EUNSUPPORTED, "T = %d outside 1..%d", T, KDA_MAX_T);
  if ((long long)p->B * p->H * 128 > 0x7fffffffLL)
    return fail(KDA_EUNSUPPORTED, "B * H = %lld is too large for one launch", (long long)p->B * p->H);
  if (p->gate_mode != KDA_GATE_RAW && p->gate_mode != KDA_GATE_PRECOMPUTED)
    return fail(KDA_EINVAL, "gate_mode = %d is neither KDA_GATE_RAW nor KDA_GATE_PRECOMPUTED", p->gate_mode);
  if (p->config_override < -1 || p->config_override >= kNumConfigs)
    return fail(KDA_EINVAL, "config_override = %d outside -1..%d", p->config_override, kNumConfigs - 1);
  if (!(p->lower_bound == p->lower_bound) || p->lower_bound > 3.0e38f || p->lower_bound < -3.0e38f)
    return fail(KDA_EINVAL, "lower_bound is not finite");
  if (!(p->scale == p->scale) || p->scale > 3.0e38f || p->scale < -3.0e38f)
    return fail(KDA_EINVAL, "scale is not finite");
  *bulk = false;
  if (p->B == 0) return KDA_OK;  // nothing is read or written
  kda_status s;
  if ((s = check_view("q", p->q, 128)) != KDA_OK) return s;
  if ((s = check_view("k", p->k, 128)) != KDA_OK) return s;
  if ((s = check_view("v", p->v, 128)) != KDA_OK) return s;
  if ((s = check_view("g_raw", p->g_raw, 128)) != KDA_OK) return s;
  if ((s = check_view("beta_logit", p->beta_logit, 1)) != KDA_OK) return s;
  if (p->gate_mode == KDA_GATE_RAW) {
    if (p->A_log == nullptr || !aligned(p->A_log, 4))
      return fail(KDA_EINVAL, "A_log is NULL or not 4-byte aligned");
    if (p->dt_bias == nullptr || !aligned(p->dt_bias, 4))
      return fail(KDA_EINVAL, "dt_bias is NULL or not 4-byte aligned");
  }
  if (p->state_indices == nullptr || !aligned(p->state_indices, 4))
    return fail(KDA_EINVAL, "state_indices is NULL or not 4-byte aligned");
  if (p->out == nullptr || !aligned(p->out, 2)) return fail(KDA_EINVAL, "out is NULL or not 2-byte aligned");
  if (p->out_b_stride < 0 || p->out_t_stride < 0 || p->out_h_stride < 0)
    return fail(KDA_EINVAL, "out has a negative stride");
  if (p->error_word != nullptr && !aligned(p->error_word, 4))
    return fail(KDA_EINVAL, "error_word is not 4-byte aligned");
  const int64_t slot = (int64_t)p->H * 128 * 128;
  if (p->N > 0) {
    if (p->state == nullptr) return fail(KDA_EINVAL, "state is NULL with N = %d", p->N);
    if (!aligned(p->state, 2)) return fail(KDA_EINVAL, "state is not 2-byte aligned");
    if (p->N > 1 && p->state_slot_stride < slot)
      return fail(KDA_EINVAL, "state_slot_stride = %lld < H*V*K = %lld", (long long)p->state_slot_stride,
                  (long long)slot);
  }
  *bulk = p->N > 0 && aligned(p->state, 16) && (p->N == 1 || p->state_slot_stride % 8 == 0);
  if (p->B > 0 && p->N > 0) {
    uintptr_t o0, o1, s0, s1;
    view_extent(p->out, p->B, T, p->H, 128, p->out_b_stride, p->out_t_stride, p->out_h_stride, o0, o1);
    s0 = reinterpret_cast<uintptr_t>(p->state);
    s1 = s0 + (uintptr_t)((int64_t)(p->N - 1) * p->state_slot_stride + slot) * 2;
    if (overlaps(o0, o1, s0, s1)) return fail(KDA_EINVAL, "out overlaps the state pool");
  }
  return KDA_OK;
}

int pick_config(const kda_params* p, int T) {
  return p->config_override >= 0 ? p->config_override : kda_select_config(p->B, T);
}

// The ring kernel works on whole heads: the one configuration it runs.
constexpr int kRingConfig = 3;

}  // namespace

extern "C" {

int32_t kda_num_configs(void) { return kNumConfigs; }

int32_t kda_config_tile_v(int32_t config) {
  if (config < 0 || config >= kNumConfigs) return -1;
  return kTileV[config];
}

// Launch-configuration policy, measured on GB300 both with L2 cold between
// calls (CUDA-graph replays) and in warm 16-step decode loops: small batches
// take smaller tiles, so that B * H * (128 / TV) CTAs still cover the 152
// SMs, and whole-head tiles once a batch fills the machine on its own. T = 1
// and T > 1 differ because a verify CTA does T times the work per byte of
// state.
int32_t kda_select_config(int32_t B, int32_t T) {
  if (B < 0 || T < 1 || T > KDA_MAX_T) return -1;
  if (T == 1) {
    if (B <= 4) return 0;   // 16 rows
    if (B <= 8) return 1;   // 32 rows
    if (B <= 32) return 2;  // 64 rows
    return 3;               // 128 rows
  }
  if (B <= 2) return 0;   // 16 rows
  if (B <= 8) return 2;   // 64 rows, 8 warps
  if (B <= 32) return 3;  // 128 rows, 8 warps
  return 4;               // 128 rows, dot products on the tensor cores
}

// The ring kernel runs one CTA per (row, head): its state rows enter one
// 128-row tensor-core product, so it has a single configuration.
int32_t kda_select_ring_config(int32_t B, int32_t T) {
  if (B < 0 || T < 1 || T > KDA_MAX_T) return -1;
  return kRingConfig;  // 128 rows
}

// Prefill: the chunked kernel on the tensor cores (configuration 4) does the
// per-token work of a 16-token chunk as two products and a 16-step scalar
// recurrence per value row, instead of 16 passes over the state; the
// token-by-token CUDA-core kernel (configurations 0-3, of which 64-row tiles
// were the fastest on every shape measured) stays selectable.
int32_t kda_select_prefill_config(int32_t num_seqs, int32_t H) {
  if (num_seqs < 0 || H < 1) return -1;
  return kTensorCoreConfig;
}

// Prefill with a workspace: the two stages once the sequences average 512
// tokens (32 chunks) or more, where the chain's short per-chunk step outweighs
// the workspace round trip (measured on GB300: 1 x 4096 and 8 x 2048 tokens
// faster in two stages, 64 x 256 and 512 x 16 faster in the chunked single
// kernel); in one launch (6) when there are few chains (at most 32 sequences
// and 64 (sequence, head) chains), where the preparation then runs beside the
// chains instead of before them; the chunked single kernel (4) below 512.
int32_t kda_select_prefill_ws_config(int32_t B, int32_t num_seqs, int32_t H) {
  if (B < 0 || num_seqs < 0 || H < 1) return -1;
  if (num_seqs > 0 && (long long)B >= 512LL * num_seqs)
    return (num_seqs <= kFusedMaxSeqs && (long long)num_seqs * H <= 64) ? kFusedConfig : kChainConfig;
  return kTensorCoreConfig;
}

size_t kda_prefill_workspace_bytes(int32_t B, int32_t num_seqs, int32_t H) {
  if (B <= 0 || num_seqs <= 0 || H < 1) return 0;
  return kda::prefill_workspace_size(B, num_seqs, H);
}

const char* kda_last_error(void) { return g_err; }

kda_status kda_decode(const kda_params* p, void* stream) {
  bool bulk = false;
  kda_status s = check_params(p, 1, &bulk);
  if (s != KDA_OK) return s;
  if (p->config_override == kTensorCoreConfig)
    return fail(KDA_EUNSUPPORTED, "config_override = %d (tensor-core verify) needs T > 1", kTensorCoreConfig);
  if (p->B == 0) return ok();
  cudaError_t e = kda::launch_step(*p, 1, kTileV[pick_config(p, 1)], bulk, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_decode launch: %s", cudaGetErrorString(e));
  return ok();
}

kda_status kda_verify(const kda_params* p, int32_t T, void* stream) {
  bool bulk = false;
  kda_status s = check_params(p, T, &bulk);
  if (s != KDA_OK) return s;
  if (T == 1 && p->config_override == kTensorCoreConfig)
    return fail(KDA_EUNSUPPORTED, "config_override = %d (tensor-core verify) needs T > 1", kTensorCoreConfig);
  if (p->B == 0) return ok();
  const int cfg = pick_config(p, T);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cfg == kTensorCoreConfig ? kda::launch_verify_tc(*p, T, bulk, st)
                                           : kda::launch_step(*p, T, kTileV[cfg], bulk, st);
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_verify launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"

namespace {

// The ring's own checks (after the shared ones).
kda_status check_ring(const kda_params* p, int T, const kda_ring_params* r) {
  if (r == nullptr) return fail(KDA_EINVAL, "ring params is NULL");
  if (r->W < 1 || r->W > 64) return fail(KDA_EUNSUPPORTED, "W = %d outside 1..64", r->W);
  if (T > r->W) return fail(KDA_EINVAL, "T = %d exceeds the ring width W = %d", T, r->W);
  if (r->flush_min < 1 || (r->flush_min - 1) + T > r->W)
    return fail(KDA_EINVAL, "flush_min = %d: need flush_min >= 1 and flush_min - 1 + T <= W (T = %d, W = %d)",
                r->flush_min, T, r->W);
  if (p->N > 0 && p->B > 0) {
    if (r->k_cache == nullptr || r->u_cache == nullptr || r->g_cache == nullptr || r->hist_len == nullptr)
      return fail(KDA_EINVAL, "a ring buffer is NULL");
    if (!aligned(r->k_cache, 16) || !aligned(r->u_cache, 16) || !aligned(r->g_cache, 16))
      return fail(KDA_EINVAL, "k_cache, u_cache and g_cache must be 16-byte aligned");
    if (!aligned(r->hist_len, 4)) return fail(KDA_EINVAL, "hist_len is not 4-byte aligned");
    if (r->cache_base != nullptr && !aligned(r->cache_base, 4))
      return fail(KDA_EINVAL, "cache_base is not 4-byte aligned");
    const int64_t ring = (int64_t)p->H * r->W * 128;
    if (p->N > 1 && (r->k_slot_stride < ring || r->u_slot_stride < ring || r->g_slot_stride < ring))
      return fail(KDA_EINVAL, "a ring slot stride is below H*W*128 = %lld", (long long)ring);
    if (r->k_slot_stride % 8 || r->u_slot_stride % 8 || r->g_slot_stride % 4)
      return fail(KDA_EINVAL, "ring slot strides must keep slots 16-byte aligned");
  }
  if (p->config_override >= 0 && p->config_override != kRingConfig)
    return fail(KDA_EUNSUPPORTED, "config_override = %d: kda_verify_ring runs whole-head tiles only (configuration %d)",
                p->config_override, kRingConfig);
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_verify_ring(const kda_params* p, int32_t T, const kda_ring_params* r, void* stream) {
  bool bulk = false;
  kda_status s = check_params(p, T, &bulk);
  if (s != KDA_OK) return s;
  if ((s = check_ring(p, T, r)) != KDA_OK) return s;
  if (p->B == 0) return ok();
  cudaError_t e = kda::launch_ring(*p, T, *r, bulk, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_verify_ring launch: %s", cudaGetErrorString(e));
  return ok();
}

kda_status kda_prefill(const kda_params* p, const kda_seqs* sq, void* stream) {
  if (p == nullptr) return fail(KDA_EINVAL, "params is NULL");
  if (sq == nullptr) return fail(KDA_EINVAL, "seqs is NULL");
  if (sq->num_seqs < 0) return fail(KDA_EINVAL, "num_seqs = %d is negative", sq->num_seqs);
  if (sq->num_seqs == 0) return ok();  // nothing to read or write (state_indices may be empty)
  bool bulk = false;
  kda_status s = check_params(p, 1, &bulk);
  if (s != KDA_OK) return s;
  if (p->B == 0) return ok();
  if (sq->cu_seqlens == nullptr || !aligned(sq->cu_seqlens, 4))
    return fail(KDA_EINVAL, "cu_seqlens is NULL or not 4-byte aligned");
  const int cfg = p->config_override >= 0 ? p->config_override : kda_select_prefill_config(sq->num_seqs, p->H);
  if ((long long)sq->num_seqs * p->H * (128 / kTileV[cfg]) > 0x7fffffffLL)
    return fail(KDA_EUNSUPPORTED, "num_seqs * H = %lld is too large for one launch",
                (long long)sq->num_seqs * p->H);
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cfg == kTensorCoreConfig ? kda::launch_prefill_tc(*p, sq->cu_seqlens, sq->num_seqs, bulk, st)
                                           : kda::launch_prefill(*p, sq->cu_seqlens, sq->num_seqs, kTileV[cfg], bulk, st);
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_prefill launch: %s", cudaGetErrorString(e));
  return ok();
}

kda_status kda_prefill_ws(const kda_params* p, const kda_seqs* sq, void* workspace, size_t workspace_bytes,
                          void* stream) {
  if (p == nullptr) return fail(KDA_EINVAL, "params is NULL");
  if (sq == nullptr) return fail(KDA_EINVAL, "seqs is NULL");
  if (sq->num_seqs < 0) return fail(KDA_EINVAL, "num_seqs = %d is negative", sq->num_seqs);
  int cfg = p->config_override >= 0 ? p->config_override : kda_select_prefill_ws_config(p->B, sq->num_seqs, p->H);
  if (cfg != kChainConfig && cfg != kFusedConfig) {  // the single-kernel configurations; the workspace is not used
    if (p->config_override < 0) {
      kda_params q = *p;
      q.config_override = cfg;
      return kda_prefill(&q, sq, stream);
    }
    return kda_prefill(p, sq, stream);
  }
  if (sq->num_seqs == 0) return ok();
  kda_params q = *p;
  q.config_override = -1;  // configurations 5 and 6 are prefill-only; the shared checks see "library's choice"
  bool bulk = false;
  kda_status s = check_params(&q, 1, &bulk);
  if (s != KDA_OK) return s;
  if (p->B == 0) return ok();
  if (sq->cu_seqlens == nullptr || !aligned(sq->cu_seqlens, 4))
    return fail(KDA_EINVAL, "cu_seqlens is NULL or not 4-byte aligned");
  if ((long long)sq->num_seqs * p->H > 0x7fffffffLL)
    return fail(KDA_EUNSUPPORTED, "num_seqs * H = %lld is too large for one launch",
                (long long)sq->num_seqs * p->H);
  const size_t need = kda_prefill_workspace_bytes(p->B, sq->num_seqs, p->H);
  if (workspace == nullptr || !aligned(workspace, 16))
    return fail(KDA_EINVAL, "workspace is NULL or not 16-byte aligned (configuration %d)", kChainConfig);
  if (workspace_bytes < need)
    return fail(KDA_EINVAL, "workspace_bytes = %zu is below the %zu this call needs (kda_prefill_workspace_bytes)",
                workspace_bytes, need);
  {  // the workspace must not overlap anything the call reads or writes
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + need;
    struct {
      const char* name;
      const kda_view* v;
      int D;
    } views[] = {{"q", &p->q, 128}, {"k", &p->k, 128}, {"v", &p->v, 128}, {"g_raw", &p->g_raw, 128},
                 {"beta_logit", &p->beta_logit, 1}};
    for (const auto& e : views) {
      uintptr_t a0, a1;
      view_extent(e.v->ptr, p->B, 1, p->H, e.D, e.v->b_stride, 0, e.v->h_stride, a0, a1);
      if (overlaps(w0, w1, a0, a1)) return fail(KDA_EINVAL, "workspace overlaps %s", e.name);
    }
    uintptr_t o0, o1;
    view_extent(p->out, p->B, 1, p->H, 128, p->out_b_stride, 0, p->out_h_stride, o0, o1);
    if (overlaps(w0, w1, o0, o1)) return fail(KDA_EINVAL, "workspace overlaps out");
    if (p->N > 0) {
      const uintptr_t s0 = reinterpret_cast<uintptr_t>(p->state);
      const uintptr_t s1 = s0 + (uintptr_t)((int64_t)(p->N - 1) * p->state_slot_stride + (int64_t)p->H * 128 * 128) * 2;
      if (overlaps(w0, w1, s0, s1)) return fail(KDA_EINVAL, "workspace overlaps the state pool");
    }
  }
  if (cfg == kFusedConfig) {  // one cooperative launch: few chains, 16-byte aligned token rows
    int dev = 0, sms = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return fail(KDA_ELAUNCH, "kda_prefill_ws: no current device");
    const bool fits = sq->num_seqs <= kFusedMaxSeqs && 2LL * sq->num_seqs * p->H <= sms;
    const bool aligned_rows = kda::prefill_rows_aligned16(*p);
    if (!fits || !aligned_rows) {
      if (p->config_override == kFusedConfig)
        return fail(KDA_EUNSUPPORTED,
                    "configuration %d needs num_seqs <= %d, 2 * num_seqs * H <= %d SMs and q, k, v, g_raw rows "
                    "16-byte aligned (num_seqs = %d, H = %d)",
                    kFusedConfig, kFusedMaxSeqs, sms, sq->num_seqs, p->H);
      cfg = kChainConfig;  // the library's choice falls back to two launches
    }
  }
  const cudaStream_t st = static_cast<cudaStream_t>(stream);
  cudaError_t e = cfg == kFusedConfig ? kda::launch_prefill_fused(*p, sq->cu_seqlens, sq->num_seqs, workspace, bulk, st)
                                      : kda::launch_prefill_chain(*p, sq->cu_seqlens, sq->num_seqs, workspace, bulk, st);
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_prefill_ws launch: %s", cudaGetErrorString(e));
  return ok();
}

kda_status kda_prefill_static(const kda_params* p, const kda_seqs* sq, void* stream) {
  if (p == nullptr) return fail(KDA_EINVAL, "params is NULL");
  if (sq == nullptr) return fail(KDA_EINVAL, "seqs is NULL");
  if (p->config_override != -1 && p->config_override != kChainConfig)
    return fail(KDA_EINVAL, "config_override = %d: kda_prefill_static runs configuration %d only (or -1)",
                p->config_override, kChainConfig);
  kda_params q = *p;
  q.config_override = kChainConfig;
  if (sq->num_seqs <= 0 || p->B <= 0) return kda_prefill_ws(&q, sq, nullptr, 0, stream);  // nothing is launched
  const size_t need = kda_prefill_workspace_bytes(p->B, sq->num_seqs, p->H);
  if (need > (size_t)KDA_PREFILL_STATIC_BYTES)
    return fail(KDA_EUNSUPPORTED,
                "kda_prefill_static: B = %d, num_seqs = %d, H = %d need %zu bytes of workspace, above its fixed %zu; "
                "use kda_prefill_ws",
                p->B, sq->num_seqs, p->H, need, (size_t)KDA_PREFILL_STATIC_BYTES);
  void* ws = nullptr;
  const cudaError_t e = kda::prefill_static_workspace(&ws);
  if (e != cudaSuccess)
    return fail(KDA_ELAUNCH, "kda_prefill_static: the workspace's device address: %s", cudaGetErrorString(e));
  return kda_prefill_ws(&q, sq, ws, KDA_PREFILL_STATIC_BYTES, stream);
}

}  // extern "C"

namespace {

// The checks of the fp8-pool calls for T tokens: the shared ones without the
// bf16 pool's, then the fp8 pool's. On success, sets *bulk.
kda_status check_fp8(const kda_params* p, int T, const kda_fp8_pool* f, bool* bulk_out) {
  if (p == nullptr) return fail(KDA_EINVAL, "params is NULL");
  kda_params common = *p;
  common.N = 0;
  bool unused = false;
  kda_status s = check_params(&common, T, &unused);
  if (s != KDA_OK) return s;
  if (p->config_override == kTensorCoreConfig)
    return fail(KDA_EUNSUPPORTED, T == 1 ? "config_override = %d (tensor-core verify) needs T > 1"
                                         : "config_override = %d (tensor-core verify) has no fp8-pool form",
                kTensorCoreConfig);
  if (f == nullptr) return fail(KDA_EINVAL, "fp8 pool is NULL");
  const int64_t slot = (int64_t)p->H * 128 * 128, sslot = (int64_t)p->H * 128;
  bool bulk = false;
  if (p->N > 0) {
    if (p->state == nullptr) return fail(KDA_EINVAL, "state is NULL with N = %d", p->N);
    if (f->scale == nullptr || !aligned(f->scale, 4))
      return fail(KDA_EINVAL, "scale is NULL or not 4-byte aligned with N = %d", p->N);
    if (p->N > 1 && p->state_slot_stride < slot)
      return fail(KDA_EINVAL, "state_slot_stride = %lld < H*V*K = %lld", (long long)p->state_slot_stride,
                  (long long)slot);
    if (p->N > 1 && f->scale_slot_stride < sslot)
      return fail(KDA_EINVAL, "scale_slot_stride = %lld < H*V = %lld", (long long)f->scale_slot_stride,
                  (long long)sslot);
    bulk = aligned(p->state, 16) && aligned(f->scale, 16) &&
           (p->N == 1 || (p->state_slot_stride % 16 == 0 && f->scale_slot_stride % 4 == 0));
    if (p->B > 0) {
      uintptr_t o0, o1;
      view_extent(p->out, p->B, T, p->H, 128, p->out_b_stride, p->out_t_stride, p->out_h_stride, o0, o1);
      const uintptr_t c0 = reinterpret_cast<uintptr_t>(p->state);
      const uintptr_t c1 = c0 + (uintptr_t)((int64_t)(p->N - 1) * p->state_slot_stride + slot);
      const uintptr_t s0 = reinterpret_cast<uintptr_t>(f->scale);
      const uintptr_t s1 = s0 + (uintptr_t)((int64_t)(p->N - 1) * f->scale_slot_stride + sslot) * 4;
      if (overlaps(o0, o1, c0, c1)) return fail(KDA_EINVAL, "out overlaps the fp8 codes");
      if (overlaps(o0, o1, s0, s1)) return fail(KDA_EINVAL, "out overlaps the fp8 scales");
    }
  }
  *bulk_out = bulk;
  return KDA_OK;
}

}  // namespace

extern "C" {

kda_status kda_decode_fp8(const kda_params* p, const kda_fp8_pool* f, void* stream) {
  bool bulk = false;
  const kda_status s = check_fp8(p, 1, f, &bulk);
  if (s != KDA_OK) return s;
  if (p->B == 0) return ok();
  cudaError_t e = kda::launch_decode_fp8(*p, *f, kTileV[pick_config(p, 1)], bulk, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_decode_fp8 launch: %s", cudaGetErrorString(e));
  return ok();
}

kda_status kda_verify_fp8(const kda_params* p, int32_t T, const kda_fp8_pool* f, void* stream) {
  bool bulk = false;
  const kda_status s = check_fp8(p, T, f, &bulk);
  if (s != KDA_OK) return s;
  if (p->B == 0) return ok();
  // The library's choice: kda_select_config's tile, whole heads where it picks
  // the tensor-core configuration (which has no fp8-pool form).
  const int cfg = p->config_override >= 0 ? p->config_override : kda_select_config(p->B, T);
  const int tile_v = cfg == kTensorCoreConfig ? 128 : kTileV[cfg];
  cudaError_t e = kda::launch_verify_fp8(*p, *f, T, tile_v, bulk, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_verify_fp8 launch: %s", cudaGetErrorString(e));
  return ok();
}

kda_status kda_verify_ring_fp8(const kda_params* p, int32_t T, const kda_ring_params* r, const kda_fp8_pool* f,
                               void* stream) {
  bool unused = false;
  kda_status s = check_fp8(p, T, f, &unused);
  if (s != KDA_OK) return s;
  if ((s = check_ring(p, T, r)) != KDA_OK) return s;
  if (p->N > 0 && (!aligned(p->state, 16) || (p->N > 1 && p->state_slot_stride % 16 != 0)))
    return fail(KDA_EINVAL, "kda_verify_ring_fp8 needs 16-byte aligned codes and a slot stride that is a multiple of 16");
  if (p->B == 0) return ok();
  cudaError_t e = kda::launch_ring_fp8(*p, T, *r, *f, static_cast<cudaStream_t>(stream));
  if (e != cudaSuccess) return fail(KDA_ELAUNCH, "kda_verify_ring_fp8 launch: %s", cudaGetErrorString(e));
  return ok();
}

}  // extern "C"
