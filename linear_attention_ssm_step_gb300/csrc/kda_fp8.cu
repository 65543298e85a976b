// kda_fp8.cu - T=1 decode on an fp8 (E4M3) state pool for sm_103a.
//
// Source: "feat(kda): add packed-input CuTe decode kernel" (PR #4417),
// section "Nsight Compute": the bf16 decode already runs at the machine's
// ceiling for its access pattern, so the remaining headroom is fewer bytes
// per state element, for example an fp8 state. The format is this library's
// reading (include/kda_fp8.h): E4M3 codes, one power-of-two fp32 scale per
// state row, kda_decode's arithmetic on the exact values code * 2^e, and
// requantization decided in fp32 - m = max |s'| over the row's 128 keys, e =
// the smallest integer with m 2^-e <= 448, codes = round-to-nearest-even of
// s' 2^-e.
//
// One CTA of 128 threads per (batch row, HP heads, tile of TV value rows), as
// in the bf16 decode (whole-head tiles take two heads, HP = 2):
//   1. all threads read state_indices[b]; an inactive row writes zero output
//      and touches nothing else;
//   2. lane 0 of each warp starts two bulk copies on one mbarrier: the warp's
//      HP TV/4 rows of codes (128 bytes each, contiguous) and their scales;
//      the single-token prologue of each head runs meanwhile (the bf16
//      decode's, the same bits);
//   3. 8 lanes share a row, 4 rows per warp access; lane j holds keys
//      16j..16j+15 (16 code bytes), so a row's 8 lanes read its 128 bytes at
//      once. Codes become fp32 through the hardware conversions
//      cvt.rn.f16x2.e4m3x2 (exact) and f16 -> f32; the new row's maximum
//      goes over the row's 8 lanes; cvt.rn.satfinite.e4m3x2.f32 rounds the
//      scaled values;
//   4. the warp writes its rows and scales back with two bulk stores, the CTA
//      writes the outputs.
#include <cuda_fp16.h>

#include "kda_device.cuh"
#include "kda_fp8.h"
#include "kda_fp8_codec.cuh"
#include "kda_launch.h"

namespace kda {

constexpr int F8_ROW_BYTES = KD;  // 128 codes per state row

// Token vectors of one head (kh, qh, dd, gg), its v rows and outputs, beta and kappa.
__host__ __device__ constexpr size_t fp8_head_floats(int TV) { return 4 * KD + 2 * TV + 2 * KDA_MAX_T; }

__host__ __device__ constexpr size_t fp8_smem_bytes(int TV, int HP) {
  return (size_t)HP * TV * F8_ROW_BYTES        // codes
         + (size_t)HP * TV * 4                  // row scales
         + 64                                   // 4 mbarriers (padded)
         + (size_t)HP * fp8_head_floats(TV) * 4 // per-head token vectors
         + (size_t)3 * KD * 4;                  // single-token reduction products
}

// A lane's 16 consecutive keys 16j..16j+15 of one token's vectors, as 8 pairs.
__device__ __forceinline__ void load_pairs16(const float* v, int j, f32x2 (&out)[8]) {
  const float4* a = reinterpret_cast<const float4*>(v + 16 * j);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 f = a[i];
    out[2 * i] = pk2(f.x, f.y);
    out[2 * i + 1] = pk2(f.z, f.w);
  }
}

// One step on one fp8 state row, shared by its 8 lanes (see row_step for the
// arithmetic): dequantize, decay, the two dot products over the 8 lanes,
// update; then the row's new exponent and codes. codes and rscale are updated
// in place; returns the output of the row.
__device__ __forceinline__ float row_step_fp8(uint4& codes, float& rscale, const LaneVecs& lv, int j, float beta,
                                              float kappa, float vv, float oscale) {
  const uint32_t w[4] = {codes.x, codes.y, codes.z, codes.w};
  const f32x2 sc = pk2(rscale, rscale);
  f32x2 a[8];
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    a[2 * i] = e4m3x2_to_f32x2(w[i]);
    a[2 * i + 1] = e4m3x2_to_f32x2(w[i] >> 16);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) a[i] = mul2(lv.dd[i], mul2(a[i], sc));  // d * (code * 2^e)
  float x, y, u, yr;
  partial_dots(a, lv, x, y);
  row_reduce(x, y, j, beta, vv, u, yr);
  const f32x2 uu = pk2(u, u);
  float mx = 0.0f;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    a[i] = fma2(lv.kh[i], uu, a[i]);
    float lo, hi;
    upk2(a[i], lo, hi);
    mx = fmaxf(mx, fmaxf(fabsf(lo), fabsf(hi)));
  }
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
  mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
  const int e = row_exponent(mx);
  uint32_t c[4];
  if (__all_sync(0xffffffffu, e >= -127)) {  // 2^-e is one fp32 value (every row of the warp access)
    const f32x2 ia = pk2(pow2f(-e), pow2f(-e));
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = f32x2_to_e4m3x2(mul2(a[2 * i], ia)) | (f32x2_to_e4m3x2(mul2(a[2 * i + 1], ia)) << 16);
  } else {  // rows below the normal range (e down to -134): 2^-e in two exact factors
    const int ea = min(-e, 127);
    const f32x2 ia = pk2(pow2f(ea), pow2f(ea)), ib = pk2(pow2f(-e - ea), pow2f(-e - ea));
#pragma unroll
    for (int i = 0; i < 4; ++i)
      c[i] = f32x2_to_e4m3x2(mul2(mul2(a[2 * i], ia), ib)) |
             (f32x2_to_e4m3x2(mul2(mul2(a[2 * i + 1], ia), ib)) << 16);
  }
  codes = make_uint4(c[0], c[1], c[2], c[3]);
  rscale = pow2f(e);
  return __fmul_rn(oscale, __fmaf_rn(u, kappa, yr));
}

// Five CTAs per SM: 102 registers, no spills (six would cap them at 80 and spill).
// A CTA covers HP heads of TV rows each: with whole-head tiles, two heads (the
// rows of heads h and h + 1 are contiguous in a slot), so that each warp has
// 64 rows (8 KB) in flight, as many bytes as the bf16 decode's 32 rows.
template <int TV, int HP, bool BULK>
__global__ void __launch_bounds__(NTHREADS, 5)
    kda_decode_fp8_kernel(const kda_params p, const kda_fp8_pool f, const int tiles) {
  static_assert(TV % 16 == 0 && TV >= 16 && TV <= KD, "tile must be a multiple of 16 rows");
  static_assert(HP == 1 || (HP == 2 && TV == KD), "two heads per CTA only with whole-head tiles");
  constexpr int ROWS = HP * TV;            // rows per CTA
  constexpr int RW = ROWS / NWARPS;        // rows per warp, all of one head
  constexpr int RQ = RW / ROWS_PER_WARP;   // 4-row groups per warp
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int groups = p.H / HP;
  const int tile = blockIdx.x % tiles;
  const int hb = blockIdx.x / tiles;
  const int h0 = (hb % groups) * HP;
  const int b = hb / groups;
  const int v0 = tile * TV;

  uint8_t* st = smem;
  float* ssc = reinterpret_cast<float*>(smem + ROWS * F8_ROW_BYTES);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + ROWS * F8_ROW_BYTES + ROWS * 4);
  float* fbase = reinterpret_cast<float*>(smem + ROWS * F8_ROW_BYTES + ROWS * 4 + 64);
  float* red = fbase + HP * fp8_head_floats(TV);
  auto head_smem = [&](int hh, float*& orow) {
    TokenSmem t;
    t.kh = fbase + hh * fp8_head_floats(TV);
    t.qh = t.kh + KD;
    t.dd = t.qh + KD;
    t.gg = t.dd + KD;
    t.vrow = t.gg + KD;
    orow = t.vrow + TV;
    t.beta = orow + TV;
    t.kappa = t.beta + KDA_MAX_T;
    t.red = red;
    return t;
  };
  float* orow0;
  float* orow1;
  const TokenSmem ts0 = head_smem(0, orow0);
  const TokenSmem ts1 = head_smem(HP - 1, orow1);

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t out_base = (int64_t)b * p.out_b_stride + (int64_t)h0 * p.out_h_stride + v0;

  // Programmatic dependent launch, as the bf16 decode: wait for the kernel
  // ahead on the stream before the first read of global memory.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = p.state_indices[b];
  TokenLoads1 first0, first1;  // issued alongside the index load
  prologue_issue1(p, b, h0, v0, TV, first0);
  if (HP == 2) prologue_issue1(p, b, h0 + 1, v0, TV, first1);
  if (n < 0 || n >= p.N) {
    for (int i = tid; i < ROWS; i += NTHREADS) outp[out_base + (int64_t)(i / TV) * p.out_h_stride + i % TV] = 0;
    return;
  }

  const int64_t row0 = (int64_t)h0 * KD + v0 + warp * RW;  // first state row of this warp in the slot
  uint8_t* gst = static_cast<uint8_t*>(p.state) + (int64_t)n * p.state_slot_stride + row0 * F8_ROW_BYTES;
  float* gsc = f.scale + (int64_t)n * f.scale_slot_stride + row0;
  uint8_t* sst = st + warp * RW * F8_ROW_BYTES;
  float* ssw = ssc + warp * RW;
  constexpr uint32_t CODE_BYTES = RW * F8_ROW_BYTES, SCALE_BYTES = RW * 4;

  if constexpr (BULK) {
    if (lane == 0) {
      mbar_init(&mbar[warp], 1);
      mbar_expect_tx(&mbar[warp], CODE_BYTES + SCALE_BYTES);
      bulk_g2s(sst, gst, CODE_BYTES, &mbar[warp]);
      bulk_g2s(ssw, gsc, SCALE_BYTES, &mbar[warp]);
    }
  } else {
    for (int i = lane; i < (int)CODE_BYTES; i += 32) sst[i] = gst[i];
    for (int i = lane; i < RW; i += 32) ssw[i] = gsc[i];
  }

  token_prologue1(p, h0, TV, ts0, first0);
  if (HP == 2) token_prologue1(p, h0 + 1, TV, ts1, first1);

  bool ok = true;
  __syncwarp();
  if constexpr (BULK) ok = mbar_wait_bounded(&mbar[warp], 0);
  const int r = lane / LPR, j = lane % LPR;  // row within a 4-row group, lane within the row
  const int hw = (warp * RW) / TV;           // this warp's head within the CTA
  const TokenSmem& ts = hw ? ts1 : ts0;
  float* orow = hw ? orow1 : orow0;
  const int hrow0 = warp * RW - hw * TV;     // the warp's first row within its head's tile

  if (ok) {
    LaneVecs lv;
    load_pairs16(ts.kh, j, lv.kh);
    load_pairs16(ts.qh, j, lv.qh);
    load_pairs16(ts.dd, j, lv.dd);
    const float beta = ts.beta[0], kappa = ts.kappa[0];
#pragma unroll 2
    for (int q = 0; q < RQ; ++q) {
      const int row = ROWS_PER_WARP * q + r;  // within the warp's rows
      uint4* cell = reinterpret_cast<uint4*>(sst + row * F8_ROW_BYTES + 16 * j);
      uint4 c = *cell;
      float rs = ssw[row];
      const float o = row_step_fp8(c, rs, lv, j, beta, kappa, ts.vrow[hrow0 + row], p.scale);
      *cell = c;
      if (j == 0) {
        ssw[row] = rs;
        orow[hrow0 + row] = o;
      }
    }
    if constexpr (BULK) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_s2g(gst, sst, CODE_BYTES);
        bulk_s2g(gsc, ssw, SCALE_BYTES);
        bulk_commit();
        bulk_wait_read_all();
      }
    } else {
      __syncwarp();
      for (int i = lane; i < (int)CODE_BYTES; i += 32) gst[i] = sst[i];
      for (int i = lane; i < RW; i += 32) gsc[i] = ssw[i];
    }
  } else {
    if (lane == 0) {
      if (p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      if constexpr (BULK) mbar_drain_bounded(&mbar[warp], 0);
    }
    for (int i = lane; i < RW; i += 32) orow[hrow0 + i] = 0.0f;
  }
  __syncthreads();
  for (int i = tid; i < ROWS; i += NTHREADS) {
    const float o = i < TV ? orow0[i] : orow1[i - TV];
    outp[out_base + (int64_t)(i / TV) * p.out_h_stride + i % TV] = float_to_bf16_bits(o);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// T-token verify on the fp8 pool: one CTA of 128 threads per (batch row,
// head, tile of TV value rows). The T-token prologue of the bf16 verify, then
// each warp holds its rows' codes and scales in registers across the tokens,
// and every token dequantizes, steps and requantizes each row exactly as one
// kda_decode_fp8 call does (row_step_fp8), so that T tokens equal T decode
// calls bit for bit.
__host__ __device__ constexpr size_t fp8_verify_smem_bytes(int TV, int T) {
  return (size_t)TV * F8_ROW_BYTES                    // codes
         + (size_t)TV * 4                             // row scales
         + 64                                         // 4 mbarriers (padded)
         + ((size_t)T * KD * 4                        // kh, qh, dd, gg
            + (size_t)T * TV * 2                      // vrow, orow
            + (size_t)KDA_MAX_T * 2 + 3 * KD) * 4;    // beta, kappa, reduction products
}

template <int TV, bool BULK>
__global__ void __launch_bounds__(NTHREADS, 3)
    kda_verify_fp8_kernel(const kda_params p, const kda_fp8_pool f, const int T, const int tiles) {
  static_assert(TV % 16 == 0 && TV >= 16 && TV <= KD, "tile must be a multiple of 16 rows");
  constexpr int RW = TV / NWARPS;          // rows per warp
  constexpr int RQ = RW / ROWS_PER_WARP;   // 4-row groups per warp
  constexpr int PT = (KDA_MAX_T + NWARPS - 1) / NWARPS;
  extern __shared__ __align__(128) unsigned char smem[];

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x % tiles;
  const int bh = blockIdx.x / tiles;
  const int h = bh % p.H;
  const int b = bh / p.H;
  const int v0 = tile * TV;

  uint8_t* st = smem;
  float* ssc = reinterpret_cast<float*>(smem + TV * F8_ROW_BYTES);
  uint64_t* mbar = reinterpret_cast<uint64_t*>(smem + TV * F8_ROW_BYTES + TV * 4);
  float* fbase = reinterpret_cast<float*>(smem + TV * F8_ROW_BYTES + TV * 4 + 64);
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

  asm volatile("griddepcontrol.wait;" ::: "memory");
  const int n = p.state_indices[b];
  TokenLoads<PT> first;
  prologue_issue<PT, NWARPS>(p, b, h, T, v0, TV, first);
  if (n < 0 || n >= p.N) {
    for (int i = tid; i < T * TV; i += NTHREADS) {
      const int t = i / TV, r = i - t * TV;
      outp[out_base + (int64_t)t * p.out_t_stride + r] = 0;
    }
    return;
  }

  const int64_t row0 = (int64_t)h * KD + v0 + warp * RW;
  uint8_t* gst = static_cast<uint8_t*>(p.state) + (int64_t)n * p.state_slot_stride + row0 * F8_ROW_BYTES;
  float* gsc = f.scale + (int64_t)n * f.scale_slot_stride + row0;
  uint8_t* sst = st + warp * RW * F8_ROW_BYTES;
  float* ssw = ssc + warp * RW;
  constexpr uint32_t CODE_BYTES = RW * F8_ROW_BYTES, SCALE_BYTES = RW * 4;

  if constexpr (BULK) {
    if (lane == 0) {
      mbar_init(&mbar[warp], 1);
      mbar_expect_tx(&mbar[warp], CODE_BYTES + SCALE_BYTES);
      bulk_g2s(sst, gst, CODE_BYTES, &mbar[warp]);
      bulk_g2s(ssw, gsc, SCALE_BYTES, &mbar[warp]);
    }
  } else {
    for (int i = lane; i < (int)CODE_BYTES; i += 32) sst[i] = gst[i];
    for (int i = lane; i < RW; i += 32) ssw[i] = gsc[i];
  }

  token_prologue<PT, NWARPS>(p, b, h, T, v0, TV, ts, first);  // ends with a CTA barrier

  bool ok = true;
  __syncwarp();
  if constexpr (BULK) ok = mbar_wait_bounded(&mbar[warp], 0);
  const int r = lane / LPR, j = lane % LPR;  // row within a 4-row group, lane within the row

  if (ok) {
    uint4 c[RQ];
    float rs[RQ];
#pragma unroll
    for (int q = 0; q < RQ; ++q) {
      const int row = ROWS_PER_WARP * q + r;
      c[q] = *reinterpret_cast<const uint4*>(sst + row * F8_ROW_BYTES + 16 * j);
      rs[q] = ssw[row];
    }
#pragma unroll 1
    for (int t = 0; t < T; ++t) {
      LaneVecs lv;
      load_pairs16(ts.kh + t * KD, j, lv.kh);
      load_pairs16(ts.qh + t * KD, j, lv.qh);
      load_pairs16(ts.dd + t * KD, j, lv.dd);
      const float beta = ts.beta[t], kappa = ts.kappa[t];
#pragma unroll
      for (int q = 0; q < RQ; ++q) {
        const int row = warp * RW + ROWS_PER_WARP * q + r;  // within the tile
        const float o = row_step_fp8(c[q], rs[q], lv, j, beta, kappa, ts.vrow[t * TV + row], p.scale);
        if (j == 0) orow[t * TV + row] = o;
      }
    }
#pragma unroll
    for (int q = 0; q < RQ; ++q) {
      const int row = ROWS_PER_WARP * q + r;
      *reinterpret_cast<uint4*>(sst + row * F8_ROW_BYTES + 16 * j) = c[q];
      if (j == 0) ssw[row] = rs[q];
    }
    if constexpr (BULK) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_s2g(gst, sst, CODE_BYTES);
        bulk_s2g(gsc, ssw, SCALE_BYTES);
        bulk_commit();
        bulk_wait_read_all();
      }
    } else {
      __syncwarp();
      for (int i = lane; i < (int)CODE_BYTES; i += 32) gst[i] = sst[i];
      for (int i = lane; i < RW; i += 32) gsc[i] = ssw[i];
    }
  } else {
    if (lane == 0) {
      if (p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      if constexpr (BULK) mbar_drain_bounded(&mbar[warp], 0);
    }
    for (int i = lane; i < RW * T; i += 32) orow[(i / RW) * TV + warp * RW + i % RW] = 0.0f;
  }
  __syncthreads();
  for (int i = tid; i < T * TV; i += NTHREADS) {
    const int t = i / TV, rr = i - t * TV;
    outp[out_base + (int64_t)t * p.out_t_stride + rr] = float_to_bf16_bits(orow[i]);
  }
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

template <int TV, bool BULK>
static cudaError_t launch_vf8(const kda_params& p, const kda_fp8_pool& f, int T, cudaStream_t s) {
  auto kern = kda_verify_fp8_kernel<TV, BULK>;
  const size_t smem = fp8_verify_smem_bytes(TV, KDA_MAX_T);  // sized for any T, so one attribute call suffices
  static std::atomic<bool> smem_set{false};
  cudaError_t e = set_smem_limit_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  const int tiles = KD / TV;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)((long long)p.B * p.H * tiles));
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = fp8_verify_smem_bytes(TV, T);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p, f, T, tiles);
}

cudaError_t launch_verify_fp8(const kda_params& p, const kda_fp8_pool& f, int T, int tile_v, bool bulk,
                              cudaStream_t s) {
  switch (tile_v) {
    case 16: return bulk ? launch_vf8<16, true>(p, f, T, s) : launch_vf8<16, false>(p, f, T, s);
    case 32: return bulk ? launch_vf8<32, true>(p, f, T, s) : launch_vf8<32, false>(p, f, T, s);
    case 64: return bulk ? launch_vf8<64, true>(p, f, T, s) : launch_vf8<64, false>(p, f, T, s);
    case 128: return bulk ? launch_vf8<128, true>(p, f, T, s) : launch_vf8<128, false>(p, f, T, s);
    default: return cudaErrorInvalidValue;
  }
}

template <int TV, int HP, bool BULK>
static cudaError_t launch_f8(const kda_params& p, const kda_fp8_pool& f, cudaStream_t s) {
  const int tiles = KD / TV;
  const long long blocks = (long long)p.B * (p.H / HP) * tiles;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)blocks);
  cfg.blockDim = dim3(NTHREADS);
  cfg.dynamicSmemBytes = fp8_smem_bytes(TV, HP);
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kda_decode_fp8_kernel<TV, HP, BULK>, p, f, tiles);
}

template <int TV>
static cudaError_t launch_f8_tv(const kda_params& p, const kda_fp8_pool& f, bool bulk, cudaStream_t s) {
  return bulk ? launch_f8<TV, 1, true>(p, f, s) : launch_f8<TV, 1, false>(p, f, s);
}

cudaError_t launch_decode_fp8(const kda_params& p, const kda_fp8_pool& f, int tile_v, bool bulk, cudaStream_t s) {
  switch (tile_v) {
    case 16: return launch_f8_tv<16>(p, f, bulk, s);
    case 32: return launch_f8_tv<32>(p, f, bulk, s);
    case 64: return launch_f8_tv<64>(p, f, bulk, s);
    case 128:
      if (p.H % 2 == 0) return bulk ? launch_f8<128, 2, true>(p, f, s) : launch_f8<128, 2, false>(p, f, s);
      return launch_f8_tv<128>(p, f, bulk, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
