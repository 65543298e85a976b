// kda_device.cuh - device building blocks of the KDA serving-step kernels (sm_103a).
//
// The state of one (slot, head) is 128 rows (value index v) of 128 bf16 keys,
// 256 bytes per row, 32 KB per head. A CTA of 128 threads owns one
// (batch row, head, tile of TV value rows). Each warp stages its TV/4 rows in
// shared memory with one bulk asynchronous copy (cp.async.bulk, completion on
// an mbarrier), and writes them back with one bulk store. Inside a warp, 16
// lanes share a row: lane j holds keys 8j..8j+7 (16 bytes, one bf16x8
// vector), so a warp works on two rows at a time and reduces across 16 lanes.
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
// KDA_ERR_TIMEOUT and skips its tile instead of hanging the GPU.
constexpr unsigned long long WAIT_LIMIT_NS = 1000000000ull;  // 1 s
constexpr unsigned WAIT_LIMIT_ITERS = 1u << 28;

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

// Bulk copy global -> shared, completing `bytes` of transaction count on `bar`.
// src and dst 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_g2s(void* dst_smem, const void* src_gmem, uint32_t bytes, uint64_t* bar) {
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
  float* red;    // [KDA_MAX_T][NWARPS][3] reduction partials
};

__device__ __forceinline__ float load_bf16(const kda_view& vw, int b, int t, int h, int c) {
  const uint16_t* p = static_cast<const uint16_t*>(vw.ptr);
  return bf16_bits_to_float(p[(int64_t)b * vw.b_stride + (int64_t)t * vw.t_stride + (int64_t)h * vw.h_stride + c]);
}

// Raw per-token inputs of thread c (key channel c) for a chunk of PC tokens,
// loaded into registers together so that their global-memory latencies
// overlap instead of adding up token after token.
constexpr int PC = 4;
struct TokenLoads {
  float q[PC], k[PC], g[PC], v[PC], bl[PC];
};

__device__ __forceinline__ void prologue_issue(const kda_params& p, int b, int h, int t0, int T, int v0, int TV,
                                               TokenLoads& L) {
  const int c = threadIdx.x;
#pragma unroll
  for (int i = 0; i < PC; ++i) {
    const int t = t0 + i;
    L.q[i] = L.k[i] = L.g[i] = L.v[i] = L.bl[i] = 0.0f;
    if (t < T) {
      L.q[i] = load_bf16(p.q, b, t, h, c);
      L.k[i] = load_bf16(p.k, b, t, h, c);
      L.g[i] = load_bf16(p.g_raw, b, t, h, c);
      if (c < TV) L.v[i] = load_bf16(p.v, b, t, h, v0 + c);
      if (c == 0)
        L.bl[i] = bf16_bits_to_float(static_cast<const uint16_t*>(
            p.beta_logit.ptr)[(int64_t)b * p.beta_logit.b_stride + (int64_t)t * p.beta_logit.t_stride +
                              (int64_t)h * p.beta_logit.h_stride]);
    }
  }
}

// The per-token prologue of (row b, head h): L2 norms, k_hat . q_hat, the gate
// and beta. Thread c of the CTA handles key channel c; `first` holds the
// already-issued loads of tokens 0..PC-1. Ends with a CTA barrier. Every CTA of
// the same (b, h) computes the same bits: fixed reduction order.
__device__ __forceinline__ void token_prologue(const kda_params& p, int b, int h, int T, int v0, int TV,
                                               const TokenSmem& ts, const TokenLoads& first) {
  const int c = threadIdx.x;
  const int warp = c >> 5, lane = c & 31;
  const float a_h = expf(p.A_log[h]);
  const float dtb = p.dt_bias[(int64_t)h * KD + c];
  TokenLoads L = first;
  for (int t0 = 0; t0 < T; t0 += PC) {
    if (t0 > 0) prologue_issue(p, b, h, t0, T, v0, TV, L);
#pragma unroll
    for (int i = 0; i < PC; ++i) {
      const int t = t0 + i;
      if (t >= T) break;
      const float qc = L.q[i], kc = L.k[i];
      const float sq = warp_sum(__fmul_rn(qc, qc));
      const float sk = warp_sum(__fmul_rn(kc, kc));
      const float sqk = warp_sum(__fmul_rn(qc, kc));
      if (lane == 0) {
        float* r = ts.red + (t * NWARPS + warp) * 3;
        r[0] = sq;
        r[1] = sk;
        r[2] = sqk;
      }
      // g = lower_bound * sigmoid(exp(A_log) * (g_raw + dt_bias)), decay exp(g)
      const float z = __fmul_rn(a_h, __fadd_rn(L.g[i], dtb));
      const float sig = __frcp_rn(__fadd_rn(1.0f, expf(-z)));
      const float g = __fmul_rn(p.lower_bound, sig);
      ts.gg[t * KD + c] = g;
      ts.dd[t * KD + c] = expf(g);
      ts.qh[t * KD + c] = qc;
      ts.kh[t * KD + c] = kc;
      if (c < TV) ts.vrow[t * TV + c] = L.v[i];
      if (c == 0) ts.beta[t] = __frcp_rn(__fadd_rn(1.0f, expf(-L.bl[i])));
    }
  }
  __syncthreads();
  for (int t = 0; t < T; ++t) {
    const float* r = ts.red + t * NWARPS * 3;
    float sq = r[0], sk = r[1], sqk = r[2];
#pragma unroll
    for (int w = 1; w < NWARPS; ++w) {
      sq = __fadd_rn(sq, r[w * 3 + 0]);
      sk = __fadd_rn(sk, r[w * 3 + 1]);
      sqk = __fadd_rn(sqk, r[w * 3 + 2]);
    }
    const float rq = __frcp_rn(__fsqrt_rn(__fadd_rn(sq, L2_EPS)));
    const float rk = __frcp_rn(__fsqrt_rn(__fadd_rn(sk, L2_EPS)));
    ts.qh[t * KD + c] = __fmul_rn(ts.qh[t * KD + c], rq);
    ts.kh[t * KD + c] = __fmul_rn(ts.kh[t * KD + c], rk);
    if (c == 0) ts.kappa[t] = __fmul_rn(__fmul_rn(sqk, rq), rk);
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

// A lane's 8 keys of one token's vectors, in registers, as 4 pairs each.
struct LaneVecs {
  f32x2 kh[4], qh[4], dd[4];
};

__device__ __forceinline__ void load_lane_vecs(const TokenSmem& ts, int t, int j, LaneVecs& lv) {
  const float4* k4 = reinterpret_cast<const float4*>(ts.kh + t * KD + j * 8);
  const float4* q4 = reinterpret_cast<const float4*>(ts.qh + t * KD + j * 8);
  const float4* d4 = reinterpret_cast<const float4*>(ts.dd + t * KD + j * 8);
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const float4 a = k4[i], q = q4[i], d = d4[i];
    lv.kh[2 * i] = pk2(a.x, a.y);
    lv.kh[2 * i + 1] = pk2(a.z, a.w);
    lv.qh[2 * i] = pk2(q.x, q.y);
    lv.qh[2 * i + 1] = pk2(q.z, q.w);
    lv.dd[2 * i] = pk2(d.x, d.y);
    lv.dd[2 * i + 1] = pk2(d.z, d.w);
  }
}

// The two dot products of a row, reduced over the row's 16 lanes (lane j of
// the row, j = lane & 15), and the row's u. Transposed butterfly: at the
// first level the lanes with j < 8 keep the x half and the others the y half,
// so each later level reduces one value instead of two; a last exchange hands
// u (computed where x is complete) and y to every lane. 5 shuffles instead of
// 8, and every lane of the row ends with the same u and y: each level adds the
// same two values, in either order, in both lanes.
__device__ __forceinline__ void row_reduce(f32x2 xp, f32x2 yp, int j, float beta, float vv, float& u, float& y) {
  float x0, x1, y0, y1;
  upk2(xp, x0, x1);
  upk2(yp, y0, y1);
  const float x = __fadd_rn(x0, x1), yy = __fadd_rn(y0, y1);
  const bool upper = (j & 8) != 0;
  float keep = upper ? yy : x;
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, upper ? x : yy, 8));
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, 4));
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, 2));
  keep = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, keep, 1));
  // lanes j < 8 hold x, lanes j >= 8 hold y
  const float mine = upper ? keep : __fmul_rn(beta, __fsub_rn(vv, keep));
  const float got = __shfl_xor_sync(0xffffffffu, mine, 8);
  u = upper ? got : mine;
  y = upper ? keep : got;
}

// One gated delta-rule step on one state row, shared by 16 lanes (lane j holds
// keys 8j..8j+7 as four bf16x2 words). For the row's value index v:
//   a = d * s;  x = a . k_hat;  y = a . q_hat        (reduced over the 16 lanes)
//   u = beta (v - x);  s <- bf16(a + k_hat u);  o = scale (y + u kappa)
// The output uses the fused form o = (D s) . q_hat + u (k_hat . q_hat), which
// equals s_new . q_hat before rounding.
__device__ __forceinline__ float row_step(uint4& s, const LaneVecs& lv, int j, float beta, float kappa, float vv,
                                          float scale) {
  f32x2 a[4];
  a[0] = mul2(lv.dd[0], bf16x2_to_f32x2(s.x));
  a[1] = mul2(lv.dd[1], bf16x2_to_f32x2(s.y));
  a[2] = mul2(lv.dd[2], bf16x2_to_f32x2(s.z));
  a[3] = mul2(lv.dd[3], bf16x2_to_f32x2(s.w));
  f32x2 xp = mul2(lv.kh[0], a[0]), yp = mul2(lv.qh[0], a[0]);
#pragma unroll
  for (int i = 1; i < 4; ++i) {
    xp = fma2(lv.kh[i], a[i], xp);
    yp = fma2(lv.qh[i], a[i], yp);
  }
  float u, y;
  row_reduce(xp, yp, j, beta, vv, u, y);
  const f32x2 uu = pk2(u, u);
  s.x = f32x2_to_bf16x2(fma2(lv.kh[0], uu, a[0]));
  s.y = f32x2_to_bf16x2(fma2(lv.kh[1], uu, a[1]));
  s.z = f32x2_to_bf16x2(fma2(lv.kh[2], uu, a[2]));
  s.w = f32x2_to_bf16x2(fma2(lv.kh[3], uu, a[3]));
  return __fmul_rn(scale, __fmaf_rn(u, kappa, y));
}

}  // namespace kda
