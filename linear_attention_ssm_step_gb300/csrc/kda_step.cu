// kda_step.cu - T=1 decode and T-token verify kernels for sm_103a.
//
// One CTA (128 threads; 256 for verify tiles of 64 or 128 rows) per (batch
// row b, head h, tile of TV value rows).
//   1. All threads read state_indices[b]; an inactive row writes zero output
//      and touches nothing else ("feat(kda): add packed-input CuTe decode
//      kernel" (PR #4417), opening paragraph).
//   2. Lane 0 of each warp starts one bulk copy of the warp's TV/4 state rows
//      (TV/4 * 256 bytes, contiguous in HBM) into shared memory, completing on
//      the warp's mbarrier, before anything else, so the HBM read overlaps
//      the prologue.
//   3. The CTA computes every token's prologue (q/k L2 norms, k.q, gate
//      decay, beta) into shared memory, thread c owning key channel c.
//   4. Each warp waits for its rows, applies the T steps (8 lanes per row, 4
//      rows per warp access; rows streamed from shared memory when T = 1,
//      held in registers across tokens otherwise,
//      rounded to bf16 after every token so that T tokens equal T decode
//      calls bit for bit), writes the rows back to shared memory and starts
//      one bulk store of them to HBM.
//   5. The CTA writes the outputs (bf16) for its rows and tokens.
// A misaligned state pool runs the same kernel with plain loads and stores
// in step 2 and 4 (BULK = false); the arithmetic is the same.
#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {

__host__ __device__ constexpr size_t step_smem_bytes(int TV, int T) {
  return (size_t)TV * KD * 2          // state tile
         + 64                           // 4 mbarriers (padded)
         + (size_t)T * KD * 4 * 4       // kh, qh, dd, gg
         + (size_t)T * TV * 4 * 2       // vrow, orow
         + (size_t)KDA_MAX_T * 4 * 2    // beta, kappa
         + (size_t)3 * KD * 4;          // single-token reduction products
}

// NW warps per CTA; TT token slots of the prologue (T <= TT). T = 1 kernels
// (4 warps) are capped at 85 registers so that six 128-thread CTAs (the
// shared-memory limit of the 128-row tile) fit on an SM; 8-warp verify
// kernels at 128 registers, two CTAs (16 warps) per SM.
template <int TV, bool BULK, bool MULTI, int NW, int TT>
__global__ void __launch_bounds__(32 * NW, MULTI ? (NW == 8 ? 2 : 1) : 6)
    kda_step_kernel(const kda_params p, const int T, const int tiles) {
  static_assert(TV % 16 == 0 && TV >= 16 && TV <= KD, "tile must be a multiple of 16 rows");
  constexpr int NT = 32 * NW;             // threads
  constexpr int RW = TV / NW;             // rows per warp
  constexpr int RQ = RW / ROWS_PER_WARP;  // 4-row groups per warp
  static_assert(RQ >= 1 && RW % ROWS_PER_WARP == 0, "every warp owns whole 4-row groups");
  static_assert(MULTI || NW == NWARPS, "the single-token prologue uses 128 threads");
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x % tiles;
  const int bh = blockIdx.x / tiles;
  const int h = bh % p.H;
  const int b = bh / p.H;
  const int v0 = tile * TV;

  uint16_t* st = reinterpret_cast<uint16_t*>(smem);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + TV * KD * 2);
  float* fbase = reinterpret_cast<float*>(smem + TV * KD * 2 + 64);
  TokenSmem ts;
  ts.kh = fbase;
  ts.qh = ts.kh + T * KD;
  ts.dd = ts.qh + T * KD;
  ts.gg = ts.dd + T * KD;
  ts.vrow = ts.gg + T * KD;
  float* orow = ts.vrow + T * TV;
  ts.beta = orow + T * TV;
  ts.kappa = ts.beta + KDA_MAX_T;
  ts.red = ts.kappa + KDA_MAX_T;

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t out_base = (int64_t)b * p.out_b_stride + (int64_t)h * p.out_h_stride + v0;

  // Launched with programmatic dependent launch allowed: wait here, before the
  // first read of global memory, until the kernel ahead on the stream has
  // completed and its writes are visible (a no-op without one).
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = p.state_indices[b];
  // Token inputs, issued alongside the index load (unused by an inactive row):
  // one token over all threads for T = 1, else up to PT tokens per warp.
  constexpr int PT = (TT + NW - 1) / NW;
  TokenLoads<MULTI ? PT : 1> first;
  TokenLoads1 first1;
  if constexpr (MULTI)
    prologue_issue<PT, NW>(p, b, h, T, v0, TV, first);
  else
    prologue_issue1(p, b, h, v0, TV, first1);
  if (n < 0 || n >= p.N) {
    for (int i = tid; i < T * TV; i += NT) {
      const int t = i / TV, r = i - t * TV;
      outp[out_base + (int64_t)t * p.out_t_stride + r] = 0;
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

  if constexpr (MULTI)
    token_prologue<PT, NW>(p, b, h, T, v0, TV, ts, first);
  else
    token_prologue1(p, h, TV, ts, first1);

  bool ok = true;
  if constexpr (BULK) {
    __syncwarp();
    ok = mbar_wait_bounded(&mbar[warp], 0);
  } else {
    __syncwarp();
  }
  const int r = lane / LPR, j = lane % LPR;  // row within a 4-row group, lane within the row

  if (ok) {
    if constexpr (!MULTI) {
      LaneVecs lv;
      load_lane_vecs(ts, 0, j, lv);
      const float beta = ts.beta[0], kappa = ts.kappa[0];
#pragma unroll 2
      for (int q = 0; q < RQ; ++q) {
        const int row = warp * RW + ROWS_PER_WARP * q + r;
        RowBf16 s = load_row_bf16(st + row * KD, j);
        const float o = row_step(s, lv, j, beta, kappa, ts.vrow[row], p.scale);
        store_row_bf16(st + row * KD, j, s);
        if (j == 0) orow[row] = o;
      }
    } else {
      RowBf16 s[RQ];
#pragma unroll
      for (int q = 0; q < RQ; ++q) s[q] = load_row_bf16(st + (warp * RW + ROWS_PER_WARP * q + r) * KD, j);
      for (int t = 0; t < T; ++t) {
        LaneVecs lv;
        load_lane_vecs(ts, t, j, lv);
        const float beta = ts.beta[t], kappa = ts.kappa[t];
#pragma unroll
        for (int q = 0; q < RQ; ++q) {
          const int row = warp * RW + ROWS_PER_WARP * q + r;
          const float o = row_step(s[q], lv, j, beta, kappa, ts.vrow[t * TV + row], p.scale);
          if (j == 0) orow[t * TV + row] = o;
        }
      }
#pragma unroll
      for (int q = 0; q < RQ; ++q) store_row_bf16(st + (warp * RW + ROWS_PER_WARP * q + r) * KD, j, s[q]);
    }
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
  } else {
    if (lane == 0) {
      if (p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      if constexpr (BULK) mbar_drain_bounded(&mbar[warp], 0);
    }
    for (int i = lane; i < T * RW; i += 32) {
      const int t = i / RW, rr = i - t * RW;
      orow[t * TV + warp * RW + rr] = 0.0f;
    }
  }
  __syncthreads();
  for (int i = tid; i < T * TV; i += NT) {
    const int t = i / TV, rr = i - t * TV;
    outp[out_base + (int64_t)t * p.out_t_stride + rr] = float_to_bf16_bits(orow[i]);
  }
  // This CTA's writes are issued: the next kernel on the stream may start launching.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int TV, bool BULK, bool MULTI, int NW, int TT>
static cudaError_t launch_one(const kda_params& p, int T, cudaStream_t stream) {
  auto kern = kda_step_kernel<TV, BULK, MULTI, NW, TT>;
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, step_smem_bytes(TV, KDA_MAX_T), smem_set);
  if (e != cudaSuccess) return e;
  const int tiles = KD / TV;
  const long long blocks = (long long)p.B * p.H * tiles;
  // Programmatic dependent launch: the grid may be scheduled while the kernel
  // ahead on the stream finishes (its CTAs wait at griddepcontrol.wait).
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(32 * NW);
  cfg.dynamicSmemBytes = step_smem_bytes(TV, T);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, T, tiles);
}

// Verify tiles of 64 or 128 rows run 8 warps (16 warps per SM at two CTAs);
// smaller tiles keep 4.
template <int TV, bool BULK>
static cudaError_t launch_verify(const kda_params& p, int T, cudaStream_t s) {
  constexpr int NW = TV >= 64 ? 8 : 4;
  return T <= 8 ? launch_one<TV, BULK, true, NW, 8>(p, T, s) : launch_one<TV, BULK, true, NW, 16>(p, T, s);
}

template <int TV>
static cudaError_t launch_tv(const kda_params& p, int T, bool bulk, cudaStream_t s) {
  if (T == 1)
    return bulk ? launch_one<TV, true, false, NWARPS, 1>(p, T, s) : launch_one<TV, false, false, NWARPS, 1>(p, T, s);
  return bulk ? launch_verify<TV, true>(p, T, s) : launch_verify<TV, false>(p, T, s);
}

cudaError_t launch_step(const kda_params& p, int T, int tile_v, bool bulk, cudaStream_t s) {
  switch (tile_v) {
    case 16: return launch_tv<16>(p, T, bulk, s);
    case 32: return launch_tv<32>(p, T, bulk, s);
    case 64: return launch_tv<64>(p, T, bulk, s);
    case 128: return launch_tv<128>(p, T, bulk, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
