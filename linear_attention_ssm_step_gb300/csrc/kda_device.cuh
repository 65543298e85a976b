// kda_device.cuh - device building blocks of the KDA serving-step kernels (sm_103a).
//
// The state of one (slot, head) is 128 rows (value index v) of 128 bf16 keys,
// 256 bytes per row, 32 KB per head. A CTA of 128 threads owns one
// (batch row, head, tile of TV value rows). Each warp stages its TV/4 rows in
// shared memory with one bulk asynchronous copy (cp.async.bulk, completion on
// an mbarrier), and writes them back with one bulk store. Inside a warp, 8
// lanes share a row and a warp works on 4 rows at a time: lane j (= lane & 7)
// of a row holds keys 8j..8j+7 and 64+8j..64+8j+7 (two bf16x8 vectors), so
// that the 8 lanes of a row read 128 consecutive bytes per shared-memory
// access (no bank conflicts), and the row's dot products reduce over 8 lanes.
//
// Sources: "feat(kda): add packed-input CuTe decode kernel" (PR #4417),
// "Kernel design" (fused output o = (d*h).q + u*(k.q), packed bf16 state with
// shift/mask unpack and a single cvt.rn.bf16x2.f32 repack); the step itself
// from "T=1 fast path inside recurrent_kda" (raw gate, lower_bound, beta
// logits, q/k L2 norm, fp32 math).
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "kda.h"

namespace kda {

constexpr int KD = 128;      // K = V = 128
constexpr int NTHREADS = 128;
constexpr int NWARPS = NTHREADS / 32;
constexpr float L2_EPS = 1e-6f;

// Bounded waits: a wait that has not finished after this long gives up, sets
// KDA_ERR_TIMEOUT and skips its tile instead of hanging the GPU. The library
// uses 1 s; the failure-detection test build (KDA_WITHHOLD_LOADS below) sets a
// few milliseconds.
#ifndef KDA_WAIT_LIMIT_NS
#define KDA_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr unsigned long long WAIT_LIMIT_NS = KDA_WAIT_LIMIT_NS;
constexpr unsigned WAIT_LIMIT_ITERS = 1u << 28;

// KDA_WITHHOLD_LOADS is defined only in the failure-detection test build of
// the library: there every asynchronous global -> shared copy (bulk and
// tensor-map loads) is left unissued while its mbarrier still expects the
// bytes, so the kernel's wait on it runs out as on a copy that never lands,
// with nothing in flight, and the timeout path (error bit, skipped tile,
// zero output, state untouched) runs.
#ifdef KDA_WITHHOLD_LOADS
constexpr bool kWithholdLoads = true;
#else
constexpr bool kWithholdLoads = false;
#endif

// ---------------------------------------------------------------- PTX wrappers

__device__ __forceinline__ uint32_t smem_addr(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long global_timer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count) : "memory");
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t done;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(done)
      : "r"(smem_addr(bar)), "r"(parity)
      : "memory");
  return done != 0;
}

// Wait for phase `parity` of an mbarrier; false if the bounded wait gave up.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = global_timer_ns();
  for (unsigned it = 1; it < WAIT_LIMIT_ITERS; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 255u) == 0 && global_timer_ns() - t0 > WAIT_LIMIT_NS) return false;
  }
  return false;
}

// After a bounded wait gave up: one more bounded wait on the same phase, so
// that a copy still in flight lands before the CTA leaves and its shared
// memory goes to another CTA.
__device__ __forceinline__ void mbar_drain_bounded(uint64_t* bar, uint32_t parity) {
  (void)mbar_wait_bounded(bar, parity);
}

// Bulk copy global -> shared, completing `bytes` of transaction count on `bar`.
// src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
  if constexpr (kWithholdLoads) return;
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_addr(dst_smem)),
      "l"(src_gmem), "r"(bytes), "r"(smem_addr(bar))
      : "memory");
}

// Bulk copy shared -> global in the current bulk group.
__device__ __forceinline__ void bulk_s2g(void* dst_gmem, const void* src_smem, uint32_t bytes) {
  asm volatile("cp.async.bulk.global.shared::cta.bulk_group [%0], [%1], %2;" ::"l"(dst_gmem),
               "r"(smem_addr(src_smem)), "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }

// Wait until every committed bulk store has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}

// Wait until every committed bulk store has completed (its writes are done).
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

// Named CTA barriers (ids 1..15; count a multiple of 32 threads): bar_arrive
// signals without waiting, bar_sync waits until `count` threads have arrived
// or synced on `id`.
__device__ __forceinline__ void bar_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void bar_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// Make this thread's generic-proxy shared-memory writes visible to the async proxy.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- bf16 helpers

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
  return __uint_as_float(static_cast<uint32_t>(b) << 16);
}

__device__ __forceinline__ uint16_t float_to_bf16_bits(float f) {
  __nv_bfloat16 h = __float2bfloat16_rn(f);
  return *reinterpret_cast<uint16_t*>(&h);
}

// Two bf16 in one 32-bit word: element 2i in the low half, 2i+1 in the high half.
__device__ __forceinline__ void unpack_bf16x2(uint32_t w, float& lo, float& hi) {
  lo = __uint_as_float(w << 16);
  hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);  // cvt.rn.bf16x2.f32
  return *reinterpret_cast<uint32_t*>(&h);
}

__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) x += __shfl_xor_sync(0xffffffffu, x, off);
  return x;
}

// ---------------------------------------------------------------- per-token vectors

// What one token contributes to every state row of one (row, head), in shared memory.
struct TokenSmem {
  float* kh;     // [T][128] k_hat
  float* qh;     // [T][128] q_hat
  float* dd;     // [T][128] exp(g): per-key-channel decay
  float* gg;     // [T][128] g (log-decay), kept for the ring's G
  float* vrow;   // [T][TV] v for this CTA's value rows
  float* beta;   // [KDA_MAX_T]
  float* kappa;  // [KDA_MAX_T] k_hat . q_hat
  float* red;    // [3][128] per-channel products (single-token prologue only)
};

__device__ __forceinline__ float load_bf16(const kda_view& vw, int b, int t, int h, int c) {
  const uint16_t* p = static_cast<const uint16_t*>(vw.ptr);
  return bf16_bits_to_float(p[(int64_t)b * vw.b_stride + (int64_t)t * vw.t_stride + (int64_t)h * vw.h_stride + c]);
}

// The per-token prologue of (row b, head h): L2 norms, k_hat . q_hat, the gate
// and beta, for every token into shared memory. Warp w of NW handles tokens
// w, w + NW, ...; lane l handles key channels l + 32 i (i < 4). A warp's
// token inputs (up to PT tokens) are loaded into registers together, so that
// their latencies overlap; prologue_issue starts those loads (callers issue
// them next to the slot-index load), token_prologue finishes.
//
// Sums over the 128 channels: each lane adds its 4 channels in order, then a
// butterfly over the warp. The order is fixed, so every CTA of a (row, head)
// and every kernel that repeats it (the ring's append kernel) gets the same
// bits.
template <int PT>
struct TokenLoads {
  float q[PT][4], k[PT][4], g[PT][4], v[PT][4], bl[PT];
  float alog, dtb[4];  // A_log[h] and dt_bias[h][lane + 32 i] (raw gate)
};

// A_log[h] and the lane's four dt_bias values, issued with the token loads.
template <int PT>
__device__ __forceinline__ void gate_issue(const kda_params& p, int h, TokenLoads<PT>& L) {
  const int lane = threadIdx.x & 31;
  const bool raw = p.gate_mode == KDA_GATE_RAW;
  L.alog = raw ? p.A_log[h] : 0.0f;
#pragma unroll
  for (int i = 0; i < 4; ++i) L.dtb[i] = raw ? p.dt_bias[(int64_t)h * KD + lane + 32 * i] : 0.0f;
}

template <int PT, int NW = NWARPS>
__device__ __forceinline__ void prologue_issue(const kda_params& p, int b, int h, int T, int v0, int TV,
                                               TokenLoads<PT>& L) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  gate_issue(p, h, L);
#pragma unroll
  for (int s = 0; s < PT; ++s) {
    const int t = warp + NW * s;
    L.bl[s] = 0.0f;
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      L.q[s][i] = L.k[s][i] = L.g[s][i] = L.v[s][i] = 0.0f;
      if (t < T) {
        const int c = lane + 32 * i;
        L.q[s][i] = load_bf16(p.q, b, t, h, c);
        L.k[s][i] = load_bf16(p.k, b, t, h, c);
        L.g[s][i] = load_bf16(p.g_raw, b, t, h, c);
        if (c < TV) L.v[s][i] = load_bf16(p.v, b, t, h, v0 + c);
      }
    }
    if (t < T && lane == 0)
      L.bl[s] = bf16_bits_to_float(static_cast<const uint16_t*>(
          p.beta_logit.ptr)[(int64_t)b * p.beta_logit.b_stride + (int64_t)t * p.beta_logit.t_stride +
                            (int64_t)h * p.beta_logit.h_stride]);
  }
}

// Sum of a lane's 4 channel values, then over the warp (the fixed order above).
__device__ __forceinline__ float sum_channels(float x0, float x1, float x2, float x3) {
  return warp_sum(__fadd_rn(__fadd_rn(__fadd_rn(x0, x1), x2), x3));
}

// 1 / sqrt(sum + eps) for the L2 norm.
__device__ __forceinline__ float inv_norm(float sum_sq) { return __frcp_rn(__fsqrt_rn(__fadd_rn(sum_sq, L2_EPS))); }

// g = lower_bound * sigmoid(exp(A_log) * (g_raw + dt_bias)), given a_h = exp(A_log[h]).
__device__ __forceinline__ float gate_log_decay(float a_h, float g_raw, float dt_bias, float lower_bound) {
  const float z = __fmul_rn(a_h, __fadd_rn(g_raw, dt_bias));
  return __fmul_rn(lower_bound, __frcp_rn(__fadd_rn(1.0f, expf(-z))));
}

__device__ __forceinline__ float sigmoid(float x) { return __frcp_rn(__fadd_rn(1.0f, expf(-x))); }

// The gate of the call's convention (KDA_GATE_RAW or KDA_GATE_PRECOMPUTED):
// log-decay g of one channel, and beta from its input.
struct Gate {
  bool raw;
  float a_h, lower_bound;
  __device__ __forceinline__ Gate(const kda_params& p, int h)
      : raw(p.gate_mode == KDA_GATE_RAW), a_h(raw ? expf(p.A_log[h]) : 0.0f), lower_bound(p.lower_bound) {}
  // The same, from A_log[h] loaded ahead of time.
  __device__ __forceinline__ Gate(const kda_params& p, float alog, bool)
      : raw(p.gate_mode == KDA_GATE_RAW), a_h(raw ? expf(alog) : 0.0f), lower_bound(p.lower_bound) {}
  __device__ __forceinline__ float dt_bias(const kda_params& p, int h, int c) const {
    return raw ? p.dt_bias[(int64_t)h * KD + c] : 0.0f;
  }
  __device__ __forceinline__ float g(float g_in, float dtb) const {
    return raw ? gate_log_decay(a_h, g_in, dtb, lower_bound) : g_in;
  }
  __device__ __forceinline__ float beta(float b_in) const { return raw ? sigmoid(b_in) : b_in; }
};

template <int PT, int NW = NWARPS>
__device__ __forceinline__ void token_prologue(const kda_params& p, int b, int h, int T, int v0, int TV,
                                               const TokenSmem& ts, const TokenLoads<PT>& L) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Gate gate(p, L.alog, true);
  const float* dtb = L.dtb;
  // The sums of all of the warp's tokens first, then their per-channel work,
  // so that the tokens' dependent chains overlap. Slots past T hold zero
  // inputs and store nothing.
  float rq[PT], rk[PT], sqk[PT];
#pragma unroll
  for (int s = 0; s < PT; ++s) {
    float qq[4], kk[4], qk[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      qq[i] = __fmul_rn(L.q[s][i], L.q[s][i]);
      kk[i] = __fmul_rn(L.k[s][i], L.k[s][i]);
      qk[i] = __fmul_rn(L.q[s][i], L.k[s][i]);
    }
    rq[s] = inv_norm(sum_channels(qq[0], qq[1], qq[2], qq[3]));
    rk[s] = inv_norm(sum_channels(kk[0], kk[1], kk[2], kk[3]));
    sqk[s] = sum_channels(qk[0], qk[1], qk[2], qk[3]);
  }
#pragma unroll
  for (int s = 0; s < PT; ++s) {
    const int t = warp + NW * s;
    if (t < T) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        const float g = gate.g(L.g[s][i], dtb[i]);
        ts.gg[t * KD + c] = g;
        ts.dd[t * KD + c] = expf(g);
        ts.qh[t * KD + c] = __fmul_rn(L.q[s][i], rq[s]);
        ts.kh[t * KD + c] = __fmul_rn(L.k[s][i], rk[s]);
        if (c < TV) ts.vrow[t * TV + c] = L.v[s][i];
      }
      if (lane == 0) {
        ts.kappa[t] = __fmul_rn(__fmul_rn(sqk[s], rq[s]), rk[s]);
        ts.beta[t] = gate.beta(L.bl[s]);
      }
    }
  }
  __syncthreads();
}

// The same prologue for a single token, with all 128 threads busy (thread c =
// channel c), for the T = 1 decode. Each thread's channel products go through
// shared memory so that every lane can add channels l, l + 32, l + 64, l + 96
// in the order sum_channels uses before the same butterfly: the results are
// bit-identical to token_prologue's for that token.
struct TokenLoads1 {
  float q, k, g, v, bl;
  float alog, dtb;  // A_log[h] and dt_bias[h][c] (raw gate)
};

__device__ __forceinline__ void prologue_issue1(const kda_params& p, int b, int h, int v0, int TV, TokenLoads1& L) {
  const int c = threadIdx.x;
  const bool raw = p.gate_mode == KDA_GATE_RAW;
  L.alog = raw ? p.A_log[h] : 0.0f;
  L.dtb = raw ? p.dt_bias[(int64_t)h * KD + c] : 0.0f;
  L.q = load_bf16(p.q, b, 0, h, c);
  L.k = load_bf16(p.k, b, 0, h, c);
  L.g = load_bf16(p.g_raw, b, 0, h, c);
  L.v = c < TV ? load_bf16(p.v, b, 0, h, v0 + c) : 0.0f;
  L.bl = c == 0 ? bf16_bits_to_float(static_cast<const uint16_t*>(
                      p.beta_logit.ptr)[(int64_t)b * p.beta_logit.b_stride + (int64_t)h * p.beta_logit.h_stride])
                : 0.0f;
}

__device__ __forceinline__ void token_prologue1(const kda_params& p, int h, int TV, const TokenSmem& ts,
                                                const TokenLoads1& L) {
  const int c = threadIdx.x, lane = c & 31;
  ts.red[c] = __fmul_rn(L.q, L.q);
  ts.red[KD + c] = __fmul_rn(L.k, L.k);
  ts.red[2 * KD + c] = __fmul_rn(L.q, L.k);
  const Gate gate(p, L.alog, true);
  const float g = gate.g(L.g, L.dtb);
  ts.gg[c] = g;
  ts.dd[c] = expf(g);
  if (c < TV) ts.vrow[c] = L.v;
  __syncthreads();
  const float* r = ts.red;
  const float rq = inv_norm(sum_channels(r[lane], r[lane + 32], r[lane + 64], r[lane + 96]));
  const float rk = inv_norm(sum_channels(r[KD + lane], r[KD + lane + 32], r[KD + lane + 64], r[KD + lane + 96]));
  // every lane of every warp takes part in the butterflies; thread 0 stores
  const float sqk =
      sum_channels(r[2 * KD + lane], r[2 * KD + lane + 32], r[2 * KD + lane + 64], r[2 * KD + lane + 96]);
  ts.qh[c] = __fmul_rn(L.q, rq);
  ts.kh[c] = __fmul_rn(L.k, rk);
  if (c == 0) {
    ts.kappa[0] = __fmul_rn(__fmul_rn(sqk, rq), rk);
    ts.beta[0] = gate.beta(L.bl);
  }
  __syncthreads();
}

// ---------------------------------------------------------------- packed fp32 pairs

// Two fp32 values in one 64-bit register pair, for the sm_100+ packed
// instructions mul.rn.f32x2 / fma.rn.f32x2: one issue slot for two IEEE
// operations, each rounded exactly as its scalar counterpart.
typedef unsigned long long f32x2;

__device__ __forceinline__ f32x2 pk2(float lo, float hi) {
  f32x2 r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}

__device__ __forceinline__ void upk2(f32x2 r, float& lo, float& hi) {
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(r));
}

__device__ __forceinline__ f32x2 mul2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ f32x2 fma2(f32x2 a, f32x2 b, f32x2 c) {
  f32x2 d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}

// bf16x2 word -> fp32 pair (exact).
__device__ __forceinline__ f32x2 bf16x2_to_f32x2(uint32_t w) {
  return pk2(__uint_as_float(w << 16), __uint_as_float(w & 0xffff0000u));
}

// fp32 pair -> bf16x2 word, round to nearest even.
__device__ __forceinline__ uint32_t f32x2_to_bf16x2(f32x2 v) {
  float lo, hi;
  upk2(v, lo, hi);
  return pack_bf16x2(lo, hi);
}

// Lane layout of a row: LPR lanes per row, ROWS_PER_WARP rows per warp access.
constexpr int LPR = 8;
constexpr int ROWS_PER_WARP = 32 / LPR;

// Element offset of lane j's first and second 8-key chunk within a row.
__device__ __forceinline__ int chunk0(int j) { return 8 * j; }
__device__ __forceinline__ int chunk1(int j) { return 64 + 8 * j; }

// A lane's 16 keys of one token's vectors, in registers, as 8 pairs each:
// pairs 0..3 are keys 8j..8j+7, pairs 4..7 are keys 64+8j..64+8j+7.
struct LaneVecs {
  f32x2 kh[8], qh[8], dd[8];
};

__device__ __forceinline__ void load_pairs8(const float* v, int j, f32x2 (&out)[8]) {
  const float4* a = reinterpret_cast<const float4*>(v + chunk0(j));
  const float4* b = reinterpret_cast<const float4*>(v + chunk1(j));
  const float4 a0 = a[0], a1 = a[1], b0 = b[0], b1 = b[1];
  out[0] = pk2(a0.x, a0.y);
  out[1] = pk2(a0.z, a0.w);
  out[2] = pk2(a1.x, a1.y);
  out[3] = pk2(a1.z, a1.w);
  out[4] = pk2(b0.x, b0.y);
  out[5] = pk2(b0.z, b0.w);
  out[6] = pk2(b1.x, b1.y);
  out[7] = pk2(b1.z, b1.w);
}

__device__ __forceinline__ void load_lane_vecs(const TokenSmem& ts, int t, int j, LaneVecs& lv) {
  load_pairs8(ts.kh + t * KD, j, lv.kh);
  load_pairs8(ts.qh + t * KD, j, lv.qh);
  load_pairs8(ts.dd + t * KD, j, lv.dd);
}

// A row's 16 keys of lane j, as two bf16x8 vectors.
struct RowBf16 {
  uint4 a, b;
};

__device__ __forceinline__ RowBf16 load_row_bf16(const uint16_t* row, int j) {
  RowBf16 r;
  r.a = *reinterpret_cast<const uint4*>(row + chunk0(j));
  r.b = *reinterpret_cast<const uint4*>(row + chunk1(j));
  return r;
}

__device__ __forceinline__ void store_row_bf16(uint16_t* row, int j, const RowBf16& r) {
  *reinterpret_cast<uint4*>(row + chunk0(j)) = r.a;
  *reinterpret_cast<uint4*>(row + chunk1(j)) = r.b;
}

__device__ __forceinline__ void row_to_f32(const RowBf16& r, f32x2 (&s)[8]) {
  s[0] = bf16x2_to_f32x2(r.a.x);
  s[1] = bf16x2_to_f32x2(r.a.y);
  s[2] = bf16x2_to_f32x2(r.a.z);
  s[3] = bf16x2_to_f32x2(r.a.w);
  s[4] = bf16x2_to_f32x2(r.b.x);
  s[5] = bf16x2_to_f32x2(r.b.y);
  s[6] = bf16x2_to_f32x2(r.b.z);
  s[7] = bf16x2_to_f32x2(r.b.w);
}

__device__ __forceinline__ RowBf16 row_to_bf16(const f32x2 (&s)[8]) {
  RowBf16 r;
  r.a.x = f32x2_to_bf16x2(s[0]);
  r.a.y = f32x2_to_bf16x2(s[1]);
  r.a.z = f32x2_to_bf16x2(s[2]);
  r.a.w = f32x2_to_bf16x2(s[3]);
  r.b.x = f32x2_to_bf16x2(s[4]);
  r.b.y = f32x2_to_bf16x2(s[5]);
  r.b.z = f32x2_to_bf16x2(s[6]);
  r.b.w = f32x2_to_bf16x2(s[7]);
  return r;
}

// Lane j's partial dot products x = a . k_hat and y = a . q_hat over its 16
// keys (two accumulator chains each, summed in a fixed order).
__device__ __forceinline__ void partial_dots(const f32x2 (&a)[8], const LaneVecs& lv, float& x, float& y) {
  f32x2 xa = mul2(lv.kh[0], a[0]), xb = mul2(lv.kh[1], a[1]);
  f32x2 ya = mul2(lv.qh[0], a[0]), yb = mul2(lv.qh[1], a[1]);
#pragma unroll
  for (int i = 2; i < 8; i += 2) {
    xa = fma2(lv.kh[i], a[i], xa);
    xb = fma2(lv.kh[i + 1], a[i + 1], xb);
    ya = fma2(lv.qh[i], a[i], ya);
    yb = fma2(lv.qh[i + 1], a[i + 1], yb);
  }
  float x0, x1, x2, x3, y0, y1, y2, y3;
  upk2(xa, x0, x1);
  upk2(xb, x2, x3);
  upk2(ya, y0, y1);
  upk2(yb, y2, y3);
  x = __fadd_rn(__fadd_rn(x0, x2), __fadd_rn(x1, x3));
  y = __fadd_rn(__fadd_rn(y0, y2), __fadd_rn(y1, y3));
}

// The row's x and y reduced over its 8 lanes, and its u = beta (v - x).
// Transposed butterfly: at the first level lanes j < 4 keep the x half and
// lanes j >= 4 the y half, so the next two levels reduce one value each; a
// last exchange hands u (computed where x is complete) and y to every lane.
// 4 shuffles for the 4 rows of a warp access. Every lane of the row ends with
// the same u and y: each level adds the same two values, in either order, in
// both lanes.
__device__ __forceinline__ void row_reduce(float x, float y, int j, float beta, float vv, float& u, float& y_out) {
  const bool upper = (j & 4) != 0;
  float keep = upper ? y : x;
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, upper ? x : y, 4));
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, 2));
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, 1));
  // lanes j < 4 hold x, lanes j >= 4 hold y
  const float mine = upper ? keep : __fmul_rn(beta, __fsub_rn(vv, keep));
  const float got = __shfl_xor_sync(0xffffffffu, mine, 4);
  u = upper ? got : mine;
  y_out = upper ? keep : got;
}

// One gated delta-rule step on one bf16 state row, shared by its 8 lanes. For
// the row's value index v:
//   a = d * s;  x = a . k_hat;  y = a . q_hat        (reduced over the 8 lanes)
//   u = beta (v - x);  s <- bf16(a + k_hat u);  o = scale (y + u kappa)
// The output uses the fused form o = (D s) . q_hat + u (k_hat . q_hat), which
// equals s_new . q_hat before rounding.
__device__ __forceinline__ float row_step(RowBf16& row, const LaneVecs& lv, int j, float beta, float kappa,
                                          float vv, float scale) {
  f32x2 a[8];
  row_to_f32(row, a);
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = mul2(lv.dd[i], a[i]);
  float x, y, u, yr;
  partial_dots(a, lv, x, y);
  row_reduce(x, y, j, beta, vv, u, yr);
  const f32x2 uu = pk2(u, u);
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fma2(lv.kh[i], uu, a[i]);
  row = row_to_bf16(a);
  return __fmul_rn(scale, __fmaf_rn(u, kappa, yr));
}

}  // namespace kda
