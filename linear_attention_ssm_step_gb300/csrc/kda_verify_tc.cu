// kda_verify_tc.cu - T-token verify with the dot products on the tensor cores
// (sm_103a).
//
// The step is that of "feat(kda): add packed-input CuTe decode kernel"
// (PR #4417), "T=1 fast path inside recurrent_kda", applied T times with the
// state rounded to bf16 after every token (a T-token verify equals T decode
// steps). Per token and value row v, with a = d * s_v:
//   x = a . k_hat = s_v . (d * k_hat),  y = a . q_hat = s_v . (d * q_hat),
//   u = beta (v - x),  s_v <- bf16(a + k_hat u),  o_v = scale (y + u kappa).
// Both dot products of all 128 rows form one [128 x 128] x [128 x N] product
// of the bf16 state (exact as stored) with the vectors d * k_hat and
// d * q_hat, each split into a high and a low bf16 part (exact to 2^-17
// relative): 8 tcgen05.mma of N = 16 per token, fp32 sums in tensor memory.
// The update and the rounding are the CUDA-core kernel's, per element; the
// dot products' sums run in another order and on the two-part vectors.
//
// One CTA of 128 threads per (batch row, head). Per thread: key channel tid in
// the per-channel work; value row tid's sums; and in the per-row work a tile
// of 16 value rows x 8 keys of the state (registers, bf16 pairs): lane l of
// warp w takes rows 32 w + 16 (l / 16) .. + 15 and keys 8 (l % 16) .. + 7, so
// a warp holds whole rows 32 w .. + 31, the rows whose sums it reads.
//   1. the token inputs (the T token rows of q, k, g_raw and v) arrive by four
//      tensor-map copies into the B region, issued before the slot index is
//      known (plain loads where a view is not 16-byte aligned); the state by two
//      tensor-map loads into the K-major, 128-byte-swizzled layout of the A
//      operand; the per-token prologue (the CUDA-core verify's quantities with
//      the fast gate) runs meanwhile and writes every token's B operand:
//      token t's four rows (high parts of d k_hat and d q_hat, then the low
//      parts) at rows 4 (t % 4) .. + 3 of 16-row slice t / 4;
//   2. per token: a CTA barrier (every row is back in the A operand); warp 0
//      issues 8 tcgen05.mma on the slice of the token; every thread waits for
//      the product, reads its row's sums and computes u and o; u goes to its
//      warp's shared-memory slot; each thread updates its tile and writes it
//      back. (Independent product chains per half or per warp of the rows,
//      each product reading all 128 rows, were measured slower: the tensor
//      core's queue grows with the number of products.)
//   3. the final rows leave by two tensor-map stores.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "kda_chunk.cuh"
#include "kda_device.cuh"
#include "kda_launch.h"
#include "kda_tc.cuh"

namespace kda {

constexpr int VT_THREADS = 128;
constexpr uint32_t VT_TMEM_COLS = 32;  // the sums: 16 columns
constexpr uint32_t VT_SLICE_BYTES = 16u * 256u;  // one B slice: 16 rows x 128 keys bf16

// Shared-memory carve-up (bytes from a 1024-aligned base) for TT token slots.
struct VerifyLayout {
  uint32_t a, b, kh, dd, vrow, beta, kappa, su, bar, tslot, total;
};

__host__ __device__ inline VerifyLayout verify_layout(int TT) {
  VerifyLayout L{};
  const uint32_t tok = (uint32_t)TT * KD * 4u;
  uint32_t o = 0;
  L.a = o;
  o += 128u * 256u;  // state, 128 rows x 128 keys bf16
  L.b = o;           // the staged token inputs (TT x 4 rows of 256 bytes), then the B slices
  o += (uint32_t)((TT + 3) / 4) * VT_SLICE_BYTES;  // = TT x 1024
  L.kh = o;
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
  L.bar = o;  // the state copy's mbarrier, the token inputs', the products'
  o += 32u;
  L.tslot = o;
  o += 16u;
  L.total = o;
  return L;
}

__host__ __device__ inline size_t verify_tc_smem_bytes(int TT) { return (size_t)verify_layout(TT).total + 1024; }

// x as two bf16 parts at rows r and r + 2 of a B slice, column c.
__device__ __forceinline__ void store_split2_b(unsigned char* sb, int r, int c, float x) {
  const uint16_t x0 = float_to_bf16_bits(x);
  const uint16_t x1 = float_to_bf16_bits(__fsub_rn(x, bf16_bits_to_float(x0)));
  *reinterpret_cast<uint16_t*>(sb + sw128_offset(16, r, c)) = x0;
  *reinterpret_cast<uint16_t*>(sb + sw128_offset(16, r + 2, c)) = x1;
}

// token_prologue's quantities from the same loads (k_hat, the decay d =
// exp(g), the v rows, kappa and beta; g and q_hat are not kept), and every
// token's B rows (d k_hat and d q_hat as high and low parts; zero past T)
// written straight into the B slices, with the chunk kernels' fast gate
// (FastGate: __expf and the approximate reciprocal) and rsqrt for the norms.
// Their relative errors, a few 1e-7, are far inside the verify's tolerances;
// configurations 0-3 keep the IEEE forms, whose bits the decode shares.
template <int PT, int NW>
__device__ __forceinline__ void token_prologue_fast(const kda_params& p, int T, const TokenSmem& ts,
                                                    const TokenLoads<PT>& L, unsigned char* sB) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const FastGate gate(p, L.alog);
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
    rq[s] = rsqrtf(__fadd_rn(sum_channels(qq[0], qq[1], qq[2], qq[3]), L2_EPS));
    rk[s] = rsqrtf(__fadd_rn(sum_channels(kk[0], kk[1], kk[2], kk[3]), L2_EPS));
    sqk[s] = sum_channels(qk[0], qk[1], qk[2], qk[3]);
  }
#pragma unroll
  for (int s = 0; s < PT; ++s) {
    const int t = warp + NW * s;
    unsigned char* slice = sB + (t >> 2) * VT_SLICE_BYTES;
    if (t < T) {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        const float d = __expf(gate.g(L.g[s][i], L.dtb[i]));
        const float kh = __fmul_rn(L.k[s][i], rk[s]);
        ts.dd[t * KD + c] = d;
        ts.kh[t * KD + c] = kh;
        ts.vrow[t * KD + c] = L.v[s][i];
        store_split2_b(slice, 4 * (t & 3), c, __fmul_rn(d, kh));
        store_split2_b(slice, 4 * (t & 3) + 1, c, __fmul_rn(d, __fmul_rn(L.q[s][i], rq[s])));
      }
      if (lane == 0) {
        ts.kappa[t] = __fmul_rn(__fmul_rn(sqk[s], rq[s]), rk[s]);
        ts.beta[t] = gate.beta(L.bl[s]);
      }
    } else {
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        store_split2_b(slice, 4 * (t & 3), lane + 32 * i, 0.0f);
        store_split2_b(slice, 4 * (t & 3) + 1, lane + 32 * i, 0.0f);
      }
    }
  }
  fence_proxy_async_smem();  // the B slices are read by the tensor core
  __syncthreads();
}

// The tensor maps of the token views (TOK): q, k, g_raw, v as {128, H, T, B}
// tensors in {128, 1, TT, 1} boxes.
struct VerifyTokenMaps {
  CUtensorMap m[4];
};

// TOK: the token inputs arrive by four tensor-map copies (every view 16-byte
// aligned): view j's TT token slots at j TT 256 bytes of the B region.
template <bool TMA, int TT, bool TOK>
__global__ void __launch_bounds__(VT_THREADS, 4)
    kda_verify_tc_kernel(const __grid_constant__ CUtensorMap smap, const __grid_constant__ VerifyTokenMaps tmaps,
                         const kda_params p, const int T) {
  static_assert(TT == 8 || TT == 16, "token slots");
  constexpr int NW = VT_THREADS / 32;
  constexpr int PT = TT / NW;  // prologue tokens per warp
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.H;
  const int b = blockIdx.x / p.H;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const VerifyLayout SL = verify_layout(TT);
  unsigned char* sA = sm + SL.a;
  unsigned char* sB = sm + SL.b;
  TokenSmem ts;
  ts.kh = reinterpret_cast<float*>(sm + SL.kh);
  ts.qh = nullptr;  // q_hat and g are not kept: q_hat goes straight into the B slices
  ts.dd = reinterpret_cast<float*>(sm + SL.dd);
  ts.gg = nullptr;
  ts.vrow = reinterpret_cast<float*>(sm + SL.vrow);
  ts.beta = reinterpret_cast<float*>(sm + SL.beta);
  ts.kappa = reinterpret_cast<float*>(sm + SL.kappa);
  ts.red = nullptr;
  uint64_t* barA = reinterpret_cast<uint64_t*>(sm + SL.bar);
  uint64_t* barT = barA + 1;  // the token inputs' tensor-map copies
  uint64_t* barD = barA + 2;  // the products
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL.tslot);

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t obase = (int64_t)b * p.out_b_stride + (int64_t)h * p.out_h_stride + tid;

  // Token inputs: row t of q, k, g_raw, v at byte (4 t + j) 256 of the B
  // region (bulk copies), or plain loads into registers.
  const uint16_t* stage = reinterpret_cast<const uint16_t*>(sB);
  TokenLoads<PT> first;
  if constexpr (TOK) {
    if (tid == 32) {  // warp 1, so that warp 0 starts the state copy at once
      mbar_init(barT, 1);
      mbar_expect_tx(barT, 4u * TT * 256u);
#pragma unroll
      for (int j = 0; j < 4; ++j) tma_load_4d(sB + j * TT * 256, &tmaps.m[j], 0, h, 0, b, barT);
    }
    gate_issue(p, h, first);
#pragma unroll
    for (int s2 = 0; s2 < PT; ++s2) {  // beta's logits: one value per token
      const int t = warp + NW * s2;
      first.bl[s2] = (t < T && lane == 0)
                         ? bf16_bits_to_float(static_cast<const uint16_t*>(p.beta_logit.ptr)[
                               (int64_t)b * p.beta_logit.b_stride + (int64_t)t * p.beta_logit.t_stride +
                               (int64_t)h * p.beta_logit.h_stride])
                         : 0.0f;
    }
  } else {
    prologue_issue<PT, NW>(p, b, h, T, 0, KD, first);  // issued alongside the index load
  }
  const int n = p.state_indices[b];
  if (n < 0 || n >= p.N) {
    for (int t = 0; t < T; ++t) outp[obase + (int64_t)t * p.out_t_stride] = 0;
    if (TOK && tid == 32) mbar_drain_bounded(barT, 0);  // the copies land before the CTA leaves
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
  bool tok_ok = true;
  if constexpr (TOK) {  // this warp's tokens into registers, as the plain loads give them
    __syncthreads();      // the mbarrier's initialisation
    tok_ok = mbar_wait_bounded(barT, 0);
#pragma unroll
    for (int s2 = 0; s2 < PT; ++s2) {
      const int t = warp + NW * s2;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        const bool in = t < T && tok_ok;
        first.q[s2][i] = in ? bf16_bits_to_float(stage[(0 * TT + t) * KD + c]) : 0.0f;
        first.k[s2][i] = in ? bf16_bits_to_float(stage[(1 * TT + t) * KD + c]) : 0.0f;
        first.g[s2][i] = in ? bf16_bits_to_float(stage[(2 * TT + t) * KD + c]) : 0.0f;
        first.v[s2][i] = in ? bf16_bits_to_float(stage[(3 * TT + t) * KD + c]) : 0.0f;
      }
    }
    __syncthreads();  // the prologue writes over the staged inputs
  }
  tc_fence_before();
  token_prologue_fast<PT, NW>(p, T, ts, first, sB);  // writes the B slices; ends with a CTA barrier
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t row_tmem = tmem + ((uint32_t)(warp * 32) << 16);  // row tid's sums

  bool ok = tok_ok;
  if constexpr (TMA) ok = mbar_wait_bounded(barA, 0) && ok;
  ok = __syncthreads_and(ok) != 0;  // also publishes the B slices
  if (!ok && tid == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);

  // This thread's tile: rows r0 .. r0 + 15, keys 8 kg .. 8 kg + 7 (4 bf16 pairs per row).
  const int kg = lane & 15;
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
    // The rows of token t are in the A operand (written and fenced by every
    // warp), and the last product's sums have been read.
    tc_fence_before();
    ok = __syncthreads_and(ok) != 0;
    float o = 0.0f;
    if (ok) {
      if (warp == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, 16);
        const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB) + (uint32_t)(t >> 2) * VT_SLICE_BYTES;
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)
          tc_mma_bf16_w(tmem, sw128_desc(a0 + (kk >> 2) * (KD * 128) + (kk & 3) * 32),
                        sw128_desc(b0 + (kk >> 2) * (16 * 128) + (kk & 3) * 32), idesc, kk > 0 ? 1u : 0u);
        tc_commit_w(barD);
      }
      pendD = true;
      pend_par = (uint32_t)(t & 1);
      // One warp polls the product's mbarrier; the others sleep at the CTA
      // barrier, leaving the issue slots to the SM's other CTAs.
      bool d_ok = true;
      if (warp == 0) d_ok = mbar_wait_bounded(barD, pend_par);
      ok = __syncthreads_or(!d_ok) == 0;
      if (!ok) {
        if (p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      } else {
        pendD = false;
        tc_fence_after();
        // Row tid's sums for token t: columns 4 (t % 4) .. + 3 (x high, y high, x low, y low).
        float c[8];
        tmem_ld8(row_tmem + 8u * (uint32_t)((t >> 1) & 1), c);
        const bool odd = (t & 1) != 0;
        const float x = __fadd_rn(odd ? c[4] : c[0], odd ? c[6] : c[2]);
        const float y = __fadd_rn(odd ? c[5] : c[1], odd ? c[7] : c[3]);
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
      fence_proxy_async_smem();  // the tile written back is read by the tensor core
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

template <bool TMA, int TT, bool TOK>
static cudaError_t launch_vtc(const CUtensorMap& map, const VerifyTokenMaps& tm, const kda_params& p, int T,
                              cudaStream_t s) {
  auto kern = kda_verify_tc_kernel<TMA, TT, TOK>;
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
  kern<<<(unsigned)((long long)p.B * p.H), VT_THREADS, verify_tc_smem_bytes(TT), s>>>(map, tm, p, T);
  return cudaGetLastError();
}

// Every row (b, t, h) of the view starts on a 16-byte boundary.
static bool rows_aligned16(const kda_view& vw) {
  return reinterpret_cast<uintptr_t>(vw.ptr) % 16 == 0 && vw.b_stride % 8 == 0 && vw.t_stride % 8 == 0 &&
         vw.h_stride % 8 == 0;
}

// The token views' tensor maps for TT token slots; false (plain loads) where
// a view is not 16-byte aligned or a map cannot be formed.
static bool verify_token_maps(const kda_params& p, int T, int TT, VerifyTokenMaps* tm) {
  const kda_view* vw[4] = {&p.q, &p.k, &p.g_raw, &p.v};
  for (int j = 0; j < 4; ++j)
    if (!rows_aligned16(*vw[j]) || token_tensor_map_bt(*vw[j], p.B, T, p.H, TT, &tm->m[j]) != cudaSuccess)
      return false;
  return true;
}

cudaError_t launch_verify_tc(const kda_params& p, int T, bool bulk, cudaStream_t s) {
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  VerifyTokenMaps tm;
  memset(&tm, 0, sizeof(tm));
  const int TT = T <= 8 ? 8 : 16;
  if (bulk) {
    const cudaError_t e = state_tensor_map(p, &map);
    if (e != cudaSuccess) return e;
    if (verify_token_maps(p, T, TT, &tm))
      return TT == 8 ? launch_vtc<true, 8, true>(map, tm, p, T, s) : launch_vtc<true, 16, true>(map, tm, p, T, s);
    return TT == 8 ? launch_vtc<true, 8, false>(map, tm, p, T, s) : launch_vtc<true, 16, false>(map, tm, p, T, s);
  }
  return TT == 8 ? launch_vtc<false, 8, false>(map, tm, p, T, s) : launch_vtc<false, 16, false>(map, tm, p, T, s);
}

}  // namespace kda
