// kda_verify_tc.cu - T-token verify with the dot products on the tensor cores
// (sm_103a).
//
// The step is that of "feat(kda): add packed-input CuTe decode kernel"
// (PR #4417), "T=1 fast path inside recurrent_kda", applied T times with the
// state rounded to bf16 after every token (a T-token verify equals T decode
// steps). Per token and value row v, with a = d * s_v:
//   x = a . k_hat = s_v . (d * k_hat),  y = a . q_hat = s_v . (d * q_hat),
//   u = beta (v - x),  s_v <- bf16(a + k_hat u),  o_v = scale (y + u kappa).
// Both dot products of all 128 rows form one [128 x 128] x [128 x 2] product
// of the bf16 state (exact as stored) with the two vectors d * k_hat and
// d * q_hat, each split into three bf16 parts (exact to 2^-25 relative):
// one tcgen05.mma of N = 16 (6 columns used) per K step of 16, fp32 sums in
// tensor memory. The update and the rounding are the CUDA-core kernel's, per
// element, so only the order of the dot products' sums differs from it.
//
// One CTA of 128 threads per (batch row, head). Thread v is key channel v in
// the per-channel work and reads value row v's sums from tensor memory; in the
// per-row work each thread owns a tile of 16 value rows x 8 keys of the state
// (held in registers as bf16 pairs): lane l of warp w takes rows
// 32 w + 16 (l / 16) .. + 15 and keys 8 (l % 16) .. + 7, so a warp holds
// whole rows 32 w .. 32 w + 31, the rows whose sums it reads.
//   1. slot index; the state arrives by two tensor-map loads into the
//      K-major, 128-byte-swizzled layout of the A operand; the per-token
//      prologue (the CUDA-core verify's, the same bits) runs meanwhile;
//   2. per token: each thread writes its channel of the B operand; one thread
//      issues 8 tcgen05.mma; each thread waits for the product itself, reads
//      its row's sums and computes u and o for that row; u goes to its warp's
//      shared-memory slot; each thread updates its tile with the u of its 16
//      rows and the decay and key of its 8 channels, and writes the tile back
//      to the A operand (one CTA barrier per token, before the product);
//   3. the final rows leave by two tensor-map stores.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "kda_device.cuh"
#include "kda_launch.h"
#include "kda_tc.cuh"

namespace kda {

constexpr int VT_THREADS = 128;
constexpr uint32_t VT_TMEM_COLS = 32;

// Shared-memory carve-up (bytes from a 1024-aligned base) for TT token slots.
struct VerifyLayout {
  uint32_t a, b, kh, qh, dd, vrow, beta, kappa, su, bar, tslot, total;
};

__host__ __device__ inline VerifyLayout verify_layout(int TT) {
  VerifyLayout L{};
  const uint32_t tok = (uint32_t)TT * KD * 4u;
  uint32_t o = 0;
  L.a = o;
  o += 128u * 256u;  // state, 128 rows x 128 keys bf16
  L.b = o;           // B operand, 16 rows x 128 keys bf16; the prologue's g before it
  o += tok > 4096u ? tok : 4096u;
  L.kh = o;
  o += tok;
  L.qh = o;
  o += tok;
  L.dd = o;
  o += tok;
  L.vrow = o;
  o += tok;
  L.beta = o;
  o += KDA_MAX_T * 4u;
  L.kappa = o;
  o += KDA_MAX_T * 4u;
  L.su = o;  // per-warp slots of the rows' u
  o += 128u * 4u;
  L.bar = o;
  o += 16u;
  L.tslot = o;
  o += 16u;
  L.total = o;
  return L;
}

__host__ __device__ inline size_t verify_tc_smem_bytes(int TT) { return (size_t)verify_layout(TT).total + 1024; }

// x as three bf16 parts at rows r, r + 2, r + 4 of the B operand, column c.
__device__ __forceinline__ void store_split3_b(unsigned char* sb, int r, int c, float x) {
  const uint16_t x0 = float_to_bf16_bits(x);
  const float r1 = __fsub_rn(x, bf16_bits_to_float(x0));
  const uint16_t x1 = float_to_bf16_bits(r1);
  const uint16_t x2 = float_to_bf16_bits(__fsub_rn(r1, bf16_bits_to_float(x1)));
  *reinterpret_cast<uint16_t*>(sb + sw128_offset(16, r, c)) = x0;
  *reinterpret_cast<uint16_t*>(sb + sw128_offset(16, r + 2, c)) = x1;
  *reinterpret_cast<uint16_t*>(sb + sw128_offset(16, r + 4, c)) = x2;
}

template <bool TMA, int TT>
__global__ void __launch_bounds__(VT_THREADS, 4)
    kda_verify_tc_kernel(const __grid_constant__ CUtensorMap smap, const kda_params p, const int T) {
  static_assert(TT == 8 || TT == 16, "token slots");
  constexpr int NW = VT_THREADS / 32;
  constexpr int PT = TT / NW;  // prologue tokens per warp
  const int tid = threadIdx.x, warp = tid >> 5;
  const int h = blockIdx.x % p.H;
  const int b = blockIdx.x / p.H;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const VerifyLayout SL = verify_layout(TT);
  unsigned char* sA = sm + SL.a;
  unsigned char* sB = sm + SL.b;
  TokenSmem ts;
  ts.kh = reinterpret_cast<float*>(sm + SL.kh);
  ts.qh = reinterpret_cast<float*>(sm + SL.qh);
  ts.dd = reinterpret_cast<float*>(sm + SL.dd);
  ts.gg = reinterpret_cast<float*>(sB);  // g is not needed after the prologue
  ts.vrow = reinterpret_cast<float*>(sm + SL.vrow);
  ts.beta = reinterpret_cast<float*>(sm + SL.beta);
  ts.kappa = reinterpret_cast<float*>(sm + SL.kappa);
  ts.red = nullptr;
  uint64_t* barA = reinterpret_cast<uint64_t*>(sm + SL.bar);
  uint64_t* barD = barA + 1;
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL.tslot);

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t obase = (int64_t)b * p.out_b_stride + (int64_t)h * p.out_h_stride + tid;

  const int n = p.state_indices[b];
  TokenLoads<PT> first;  // issued alongside the index load
  prologue_issue<PT, NW>(p, b, h, T, 0, KD, first);
  if (n < 0 || n >= p.N) {
    for (int t = 0; t < T; ++t) outp[obase + (int64_t)t * p.out_t_stride] = 0;
    return;
  }
  uint16_t* gstate = static_cast<uint16_t*>(p.state) + (int64_t)n * p.state_slot_stride + (int64_t)h * KD * KD;
  if (tid == 0) {
    mbar_init(barA, 1);
    mbar_init(barD, 1);
    if constexpr (TMA) {
      mbar_expect_tx(barA, KD * KD * 2);
      tma_load_3d(sA, &smap, 0, h * KD, n, barA);
      tma_load_3d(sA + KD * 128, &smap, 64, h * KD, n, barA);
    }
  }
  if constexpr (!TMA) {  // plain loads into the same swizzled layout
    for (int r = 0; r < KD; ++r)
      *reinterpret_cast<uint16_t*>(sA + sw128_offset(KD, r, tid)) = gstate[(int64_t)r * KD + tid];
  }
  if (warp == 0) tmem_alloc(tslot, VT_TMEM_COLS);
  tc_fence_before();
  token_prologue<PT, NW>(p, b, h, T, 0, KD, ts, first);  // ends with a CTA barrier
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t row_tmem = tmem + ((uint32_t)(warp * 32) << 16);

  // B rows 6..15 stay zero (the prologue's g occupied them).
#pragma unroll
  for (int r = 6; r < 16; ++r) *reinterpret_cast<uint16_t*>(sB + sw128_offset(16, r, tid)) = 0;

  bool ok = true;
  if constexpr (TMA) ok = mbar_wait_bounded(barA, 0);
  ok = __syncthreads_and(ok) != 0;
  if (!ok && tid == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);

  // This thread's tile: rows r0 .. r0 + 15, keys 8 kg .. 8 kg + 7 (4 bf16 pairs per row).
  const int lane = tid & 31, kg = lane & 15;
  const int r0 = warp * 32 + (lane >> 4) * 16;
  uint32_t rw[16][4];
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const uint4 c = *reinterpret_cast<const uint4*>(sA + sw128_offset(KD, r0 + i, 8 * kg));
    rw[i][0] = c.x;
    rw[i][1] = c.y;
    rw[i][2] = c.z;
    rw[i][3] = c.w;
  }
  float* su = reinterpret_cast<float*>(sm + SL.su) + warp * 32;  // u of rows 32 warp .. + 31

  bool pendD = false;  // a product is in flight, issued with parity pend_par
  uint32_t pend_par = 0;
  for (int t = 0; t < T; ++t) {
    if (ok) {
      // B operand of token t: rows 0, 2, 4 = d * k_hat, rows 1, 3, 5 = d * q_hat.
      const float d = ts.dd[t * KD + tid];
      store_split3_b(sB, 0, tid, __fmul_rn(d, ts.kh[t * KD + tid]));
      store_split3_b(sB, 1, tid, __fmul_rn(d, ts.qh[t * KD + tid]));
      fence_proxy_async_smem();  // B and the tiles written back are read by the tensor core
    }
    tc_fence_before();
    ok = __syncthreads_and(ok) != 0;
    float o = 0.0f;
    if (ok) {
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, 16);
        const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_bf16(tmem, sw128_desc(a0 + (kk >> 2) * (KD * 128) + (kk & 3) * 32),
                      sw128_desc(b0 + (kk >> 2) * (16 * 128) + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
        tc_commit(barD);
      }
      pendD = true;
      pend_par = (uint32_t)(t & 1);
      ok = mbar_wait_bounded(barD, pend_par);  // every thread waits for the product itself
      if (!ok) {
        if (p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      } else {
        pendD = false;
        tc_fence_after();
        // Row tid's sums: x and y in three parts each, then u and o of the row.
        float c[8];
        tmem_ld8(row_tmem, c);
        const float x = __fadd_rn(__fadd_rn(c[0], c[2]), c[4]);
        const float y = __fadd_rn(__fadd_rn(c[1], c[3]), c[5]);
        const float u = __fmul_rn(ts.beta[t], __fsub_rn(ts.vrow[t * KD + tid], x));
        o = __fmul_rn(p.scale, __fmaf_rn(u, ts.kappa[t], y));
        su[lane] = u;
      }
    }
    __syncwarp();
    if (ok) {
      // The tile: s <- bf16(d * s + k_hat u), in registers and in the A operand.
      const float* dv = ts.dd + t * KD + 8 * kg;
      const float* kv = ts.kh + t * KD + 8 * kg;
      const float4 d0 = *reinterpret_cast<const float4*>(dv);
      const float4 d1 = *reinterpret_cast<const float4*>(dv + 4);
      const float4 k0 = *reinterpret_cast<const float4*>(kv);
      const float4 k1 = *reinterpret_cast<const float4*>(kv + 4);
      const f32x2 dp0 = pk2(d0.x, d0.y), dp1 = pk2(d0.z, d0.w), dp2 = pk2(d1.x, d1.y), dp3 = pk2(d1.z, d1.w);
      const f32x2 kp0 = pk2(k0.x, k0.y), kp1 = pk2(k0.z, k0.w), kp2 = pk2(k1.x, k1.y), kp3 = pk2(k1.z, k1.w);
      const float4* uq = reinterpret_cast<const float4*>(su + (lane & 16));
#pragma unroll
      for (int i4 = 0; i4 < 4; ++i4) {
        const float4 u4 = uq[i4];
        const float ur[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
        for (int i1 = 0; i1 < 4; ++i1) {
          const int i = 4 * i4 + i1;
          const f32x2 uu = pk2(ur[i1], ur[i1]);
          f32x2 a0 = mul2(dp0, bf16x2_to_f32x2(rw[i][0]));
          f32x2 a1 = mul2(dp1, bf16x2_to_f32x2(rw[i][1]));
          f32x2 a2 = mul2(dp2, bf16x2_to_f32x2(rw[i][2]));
          f32x2 a3 = mul2(dp3, bf16x2_to_f32x2(rw[i][3]));
          a0 = fma2(kp0, uu, a0);
          a1 = fma2(kp1, uu, a1);
          a2 = fma2(kp2, uu, a2);
          a3 = fma2(kp3, uu, a3);
          rw[i][0] = f32x2_to_bf16x2(a0);
          rw[i][1] = f32x2_to_bf16x2(a1);
          rw[i][2] = f32x2_to_bf16x2(a2);
          rw[i][3] = f32x2_to_bf16x2(a3);
          *reinterpret_cast<uint4*>(sA + sw128_offset(KD, r0 + i, 8 * kg)) =
              make_uint4(rw[i][0], rw[i][1], rw[i][2], rw[i][3]);
        }
      }
    }
    outp[obase + (int64_t)t * p.out_t_stride] = ok ? float_to_bf16_bits(o) : (uint16_t)0;
  }
  ok = __syncthreads_and(ok) != 0;
  if (!ok && tid == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);

  // The final rows: a tensor-map store of the A operand, or plain stores.
  if (ok) {
    fence_proxy_async_smem();
    __syncthreads();
    if constexpr (TMA) {
      if (tid == 0) {
        tma_store_3d(&smap, 0, h * KD, n, sA);
        tma_store_3d(&smap, 64, h * KD, n, sA + KD * 128);
        bulk_commit();
        bulk_wait_read_all();
      }
    } else {
      for (int r = 0; r < KD; ++r)
        gstate[(int64_t)r * KD + tid] = *reinterpret_cast<const uint16_t*>(sA + sw128_offset(KD, r, tid));
    }
  }
  // A product that did not finish in time gets one more bounded wait before
  // its tensor memory is released.
  if (pendD && tid == 0) mbar_wait_bounded(barD, pend_par);
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, VT_TMEM_COLS);
  }
}

template <bool TMA, int TT>
static cudaError_t launch_vtc(const CUtensorMap& map, const kda_params& p, int T, cudaStream_t s) {
  auto kern = kda_verify_tc_kernel<TMA, TT>;
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, verify_tc_smem_bytes(TT), smem_set);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> carveout_set{false};  // all of L1 as shared memory: four CTAs per SM
  if (!carveout_set.load(std::memory_order_acquire)) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    carveout_set.store(true, std::memory_order_release);
  }
  kern<<<(unsigned)((long long)p.B * p.H), VT_THREADS, verify_tc_smem_bytes(TT), s>>>(map, p, T);
  return cudaGetLastError();
}

cudaError_t launch_verify_tc(const kda_params& p, int T, bool bulk, cudaStream_t s) {
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (bulk) {
    const cudaError_t e = state_tensor_map(p, &map);
    if (e != cudaSuccess) return e;
    return T <= 8 ? launch_vtc<true, 8>(map, p, T, s) : launch_vtc<true, 16>(map, p, T, s);
  }
  return T <= 8 ? launch_vtc<false, 8>(map, p, T, s) : launch_vtc<false, 16>(map, p, T, s);
}

}  // namespace kda
