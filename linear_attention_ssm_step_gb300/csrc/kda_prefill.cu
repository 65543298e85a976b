// kda_prefill.cu - varlen prefill of the KDA recurrence on the bf16 state pool
// (sm_103a), the reading of include/kda_prefill.h.
//
// Source: "feat(kda): add CuTe DSL recurrent prefill backend" (PR #4605):
// packed sequences by cu_seqlens, the initial state read from an indexed pool
// and the final state written back in place.
//
// One CTA of 32 NW threads per (sequence, head, tile of TV value rows). The
// value rows of a head are independent given the per-token vectors, so a
// sequence's head is split over 128 / TV CTAs, each repeating the per-token
// prologue for its rows.
//   1. Every thread reads cu_seqlens[i], cu_seqlens[i+1] and the slot; invalid
//      bounds set KDA_ERR_SEQLENS, an inactive slot zeroes the out rows.
//   2. Each warp starts one bulk copy of its TV/NW state rows (plain loads for
//      a misaligned pool), which flies under the first chunk's prologue.
//   3. Tokens go in chunks of 16: the chunk's prologue (q/k L2 norms, k.q,
//      gate, beta: the verify kernel's warp-per-token prologue, the same bits)
//      into shared memory, lane-major; then every token in order on the rows, held in
//      fp32 registers for the whole sequence (8 lanes per row, 4 rows per
//      warp access, the decode step's arithmetic without its rounding); the
//      chunk's outputs leave as bf16 rows.
//   4. The rows are rounded to bf16 once and leave by one bulk store per warp.
#include "kda_device.cuh"
#include "kda_launch.h"
#include "kda_prefill.h"

namespace kda {

constexpr int PF_CHUNK = KDA_MAX_T;  // tokens per prologue chunk

__host__ __device__ constexpr size_t prefill_smem_bytes(int TV) {
  return (size_t)TV * KD * 2                 // state tile
         + 128                               // mbarriers (up to 16 warps)
         + (size_t)PF_CHUNK * KD * 4 * 3     // kh, qh, dd (lane-major)
         + (size_t)PF_CHUNK * TV * 4 * 2     // vrow, orow
         + (size_t)PF_CHUNK * 4 * 2;         // beta, kappa
}

// The token vectors (k_hat, q_hat, d) are stored lane-major: lane j's 16 keys
// (8j..8j+7 and 64+8j..64+8j+7, four float4) sit in float4 slots j, 8+j, 16+j,
// 24+j, so each of a lane's four 16-byte loads covers 128 contiguous bytes
// across the 8 lanes of a row (no bank conflicts; the 4 rows of a warp access
// read the same bytes). Position of key channel c:
__device__ __forceinline__ int lane_major(int c) {
  return ((2 * (c >> 6) + ((c & 7) >> 2)) * 8 + ((c >> 3) & 7)) * 4 + (c & 3);
}

// load_pairs8 (kda_device.cuh) from a lane-major vector: the same pairs.
__device__ __forceinline__ void load_pairs8_lm(const float* v, int j, f32x2 (&out)[8]) {
  const float4* a = reinterpret_cast<const float4*>(v);
  const float4 a0 = a[j], a1 = a[8 + j], b0 = a[16 + j], b1 = a[24 + j];
  out[0] = pk2(a0.x, a0.y);
  out[1] = pk2(a0.z, a0.w);
  out[2] = pk2(a1.x, a1.y);
  out[3] = pk2(a1.z, a1.w);
  out[4] = pk2(b0.x, b0.y);
  out[5] = pk2(b0.z, b0.w);
  out[6] = pk2(b1.x, b1.y);
  out[7] = pk2(b1.z, b1.w);
}

// token_prologue (kda_device.cuh) with the same arithmetic, writing k_hat,
// q_hat and d lane-major and no g (the prefill keeps no ring).
template <int PT, int NW>
__device__ __forceinline__ void token_prologue_lm(const kda_params& p, int h, int T, int TV, const TokenSmem& ts,
                                                  const TokenLoads<PT>& L) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const Gate gate(p, L.alog, true);
  const float* dtb = L.dtb;
#pragma unroll
  for (int s = 0; s < PT; ++s) {
    const int t = warp + NW * s;
    if (t < T) {
      float qq[4], kk[4], qk[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        qq[i] = __fmul_rn(L.q[s][i], L.q[s][i]);
        kk[i] = __fmul_rn(L.k[s][i], L.k[s][i]);
        qk[i] = __fmul_rn(L.q[s][i], L.k[s][i]);
      }
      const float rq = inv_norm(sum_channels(qq[0], qq[1], qq[2], qq[3]));
      const float rk = inv_norm(sum_channels(kk[0], kk[1], kk[2], kk[3]));
      const float sqk = sum_channels(qk[0], qk[1], qk[2], qk[3]);
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i, pos = t * KD + lane_major(c);
        ts.dd[pos] = expf(gate.g(L.g[s][i], dtb[i]));
        ts.qh[pos] = __fmul_rn(L.q[s][i], rq);
        ts.kh[pos] = __fmul_rn(L.k[s][i], rk);
        if (c < TV) ts.vrow[t * TV + c] = L.v[s][i];
      }
      if (lane == 0) {
        ts.kappa[t] = __fmul_rn(__fmul_rn(sqk, rq), rk);
        ts.beta[t] = gate.beta(L.bl[s]);
      }
    }
  }
  __syncthreads();
}

// The decode step (row_step in kda_device.cuh) on a row held in fp32: the same
// operations in the same order, without rounding the row to bf16.
__device__ __forceinline__ float row_step_f32(f32x2 (&a)[8], const LaneVecs& lv, int j, float beta, float kappa,
                                              float vv, float scale) {
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = mul2(lv.dd[i], a[i]);
  float x, y, u, yr;
  partial_dots(a, lv, x, y);
  row_reduce(x, y, j, beta, vv, u, yr);
  const f32x2 uu = pk2(u, u);
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = fma2(lv.kh[i], uu, a[i]);
  return __fmul_rn(scale, __fmaf_rn(u, kappa, yr));
}

// p: the call's parameters with t_stride = b_stride in q, k, v, g_raw and
// beta_logit, so that token t of a chunk starting at row c0 is (b = c0, t).
template <int TV, bool BULK, int NW>
__global__ void __launch_bounds__(32 * NW) kda_prefill_kernel(const kda_params p, const int32_t* __restrict__ cu,
                                                              const int tiles) {
  constexpr int NT = 32 * NW;
  constexpr int RW = TV / NW;             // rows per warp
  constexpr int RQ = RW / ROWS_PER_WARP;  // 4-row groups per warp
  constexpr int PT = (PF_CHUNK + NW - 1) / NW;
  static_assert(RQ >= 1 && RW % ROWS_PER_WARP == 0, "every warp owns whole 4-row groups");
  static_assert(NW <= 16, "one mbarrier per warp in 128 bytes");
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x % tiles;
  const int sh = blockIdx.x / tiles;
  const int h = sh % p.H;
  const int seq = sh / p.H;
  const int v0 = tile * TV;

  uint16_t* st = reinterpret_cast<uint16_t*>(smem);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + TV * KD * 2);
  float* fbase = reinterpret_cast<float*>(smem + TV * KD * 2 + 128);
  TokenSmem ts;
  ts.kh = fbase;
  ts.qh = ts.kh + PF_CHUNK * KD;
  ts.dd = ts.qh + PF_CHUNK * KD;
  ts.gg = nullptr;  // no ring
  ts.vrow = ts.dd + PF_CHUNK * KD;
  float* orow = ts.vrow + PF_CHUNK * TV;
  ts.beta = orow + PF_CHUNK * TV;
  ts.kappa = ts.beta + PF_CHUNK;
  ts.red = nullptr;  // the warp-per-token prologue needs no block sums
  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t out_h = (int64_t)h * p.out_h_stride + v0;

  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int t0 = cu[seq], t1 = cu[seq + 1];
  const int n = p.state_indices[seq];
  if (t0 < 0 || t1 < t0 || t1 > p.B) {
    if (tid == 0 && tile == 0 && h == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_SEQLENS);
    return;
  }
  if (t0 == t1) return;
  if (n < 0 || n >= p.N) {
    for (int64_t i = tid; i < (int64_t)(t1 - t0) * TV; i += NT) {
      const int t = (int)(i / TV), r = (int)(i - (int64_t)t * TV);
      outp[(int64_t)(t0 + t) * p.out_b_stride + out_h + r] = 0;
    }
    return;
  }

  uint16_t* gst = static_cast<uint16_t*>(p.state) + (int64_t)n * p.state_slot_stride +
                  ((int64_t)h * KD + v0 + warp * RW) * KD;
  uint16_t* sst = st + warp * RW * KD;
  constexpr uint32_t CHUNK_BYTES = RW * KD * 2;
  if constexpr (BULK) {
    if (lane == 0) {
      mbar_init(&mbar[warp], 1);
      mbar_expect_tx(&mbar[warp], CHUNK_BYTES);
      bulk_g2s(sst, gst, CHUNK_BYTES, &mbar[warp]);
    }
  } else {
    for (int i = lane; i < RW * KD; i += 32) sst[i] = gst[i];
  }

  const int r = lane / LPR, j = lane % LPR;  // row within a 4-row group, lane within the row
  f32x2 a[RQ][8];
  bool ok = true;
  for (int c0 = t0; c0 < t1; c0 += PF_CHUNK) {
    const int T = min(PF_CHUNK, t1 - c0);
    TokenLoads<PT> L;
    prologue_issue<PT, NW>(p, c0, h, T, v0, TV, L);
    token_prologue_lm<PT, NW>(p, h, T, TV, ts, L);  // ends with __syncthreads
    if (c0 == t0) {  // the state rows, once: bf16 -> fp32 registers
      __syncwarp();
      if constexpr (BULK) ok = mbar_wait_bounded(&mbar[warp], 0);
      if (ok) {
#pragma unroll
        for (int q = 0; q < RQ; ++q) row_to_f32(load_row_bf16(sst + (ROWS_PER_WARP * q + r) * KD, j), a[q]);
      } else if (lane == 0) {
        if (p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
        if constexpr (BULK) mbar_drain_bounded(&mbar[warp], 0);
      }
    }
    if (ok) {
#pragma unroll 2
      for (int t = 0; t < T; ++t) {
        LaneVecs lv;
        load_pairs8_lm(ts.kh + t * KD, j, lv.kh);
        load_pairs8_lm(ts.qh + t * KD, j, lv.qh);
        load_pairs8_lm(ts.dd + t * KD, j, lv.dd);
        const float beta = ts.beta[t], kappa = ts.kappa[t];
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const int row = warp * RW + ROWS_PER_WARP * q + r;
          const float o = row_step_f32(a[q], lv, j, beta, kappa, ts.vrow[t * TV + row], p.scale);
          if (j == 0) orow[t * TV + row] = o;
        }
      }
    } else {
      for (int i = lane; i < T * RW; i += 32) {
        const int t = i / RW, rr = i - t * RW;
        orow[t * TV + warp * RW + rr] = 0.0f;
      }
    }
    __syncthreads();
    for (int i = tid; i < T * TV; i += NT) {
      const int t = i / TV, rr = i - t * TV;
      outp[(int64_t)(c0 + t) * p.out_b_stride + out_h + rr] = float_to_bf16_bits(orow[i]);
    }
    // The next chunk's prologue rewrites the token vectors, which every thread
    // finished reading before the barrier above; orow is rewritten only after
    // that prologue's own barrier.
  }

  if (ok) {
#pragma unroll
    for (int q = 0; q < RQ; ++q) store_row_bf16(sst + (ROWS_PER_WARP * q + r) * KD, j, row_to_bf16(a[q]));
    if constexpr (BULK) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_s2g(gst, sst, CHUNK_BYTES);
        bulk_commit();
        bulk_wait_read_all();
      }
    } else {
      __syncwarp();
      for (int i = lane; i < RW * KD; i += 32) gst[i] = sst[i];
    }
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int TV, int NW>
static cudaError_t launch_pf(const kda_params& p, const int32_t* cu, int num_seqs, bool bulk, cudaStream_t stream) {
  auto kern = bulk ? kda_prefill_kernel<TV, true, NW> : kda_prefill_kernel<TV, false, NW>;
  static std::atomic<bool> smem_set_bulk{false}, smem_set_plain{false};
  cudaError_t e = set_smem_limit_once(kern, prefill_smem_bytes(TV), bulk ? smem_set_bulk : smem_set_plain);
  if (e != cudaSuccess) return e;
  kda_params q = p;  // token t of a chunk is activation row c0 + t
  q.q.t_stride = q.q.b_stride;
  q.k.t_stride = q.k.b_stride;
  q.v.t_stride = q.v.b_stride;
  q.g_raw.t_stride = q.g_raw.b_stride;
  q.beta_logit.t_stride = q.beta_logit.b_stride;
  const int tiles = KD / TV;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)num_seqs * p.H * tiles));
  cfg.blockDim = dim3(32 * NW);
  cfg.dynamicSmemBytes = prefill_smem_bytes(TV);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, q, cu, tiles);
}

// 4 warps for tiles of 16 and 32 rows, 8 for 64 and 16 for whole heads, so
// that each warp holds at most two 4-row groups in registers.
cudaError_t launch_prefill(const kda_params& p, const int32_t* cu, int num_seqs, int tile_v, bool bulk,
                           cudaStream_t s) {
  switch (tile_v) {
    case 16: return launch_pf<16, 4>(p, cu, num_seqs, bulk, s);
    case 32: return launch_pf<32, 4>(p, cu, num_seqs, bulk, s);
    case 64: return launch_pf<64, 8>(p, cu, num_seqs, bulk, s);
    case 128: return launch_pf<128, 16>(p, cu, num_seqs, bulk, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
