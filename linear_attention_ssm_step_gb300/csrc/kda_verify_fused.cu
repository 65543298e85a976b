// kda_verify_fused.cu - T-token verify on the CUDA cores with each token's
// dot products fused into the previous token's update pass (sm_103a).
//
// The step is that of "feat(kda): add packed-input CuTe decode kernel"
// (PR #4417), "T=1 fast path inside recurrent_kda", applied T times with the
// state rounded to bf16 after every token (a T-token verify equals T decode
// steps). Per token t and value row v, with a = d_t * s_v:
//   x = a . k_hat_t = s_v . (d_t * k_hat_t),   y = s_v . (d_t * q_hat_t),
//   u = beta_t (v - x),   s_v <- bf16(a + k_hat_t u),   o_v = scale (y + u kappa_t).
// The rounding makes every token an element-wise pass over the state; this
// kernel does the next token's two dot products in the same pass, on the
// freshly rounded values: s_v . (d_{t+1} * k_hat_{t+1}) and
// s_v . (d_{t+1} * q_hat_{t+1}), so that the only exchange between tokens is a
// reduction across the lanes that share a row, inside one warp.
//
// One CTA of 256 threads per (batch row, head). Lane l of warp w owns a tile of
// 8 value rows x 8 keys of the state, held in registers as bf16 pairs: rows
// 16 w + 8 (l / 16) .. + 7, keys 8 (l % 16) .. + 7; the 16 lanes of a half-warp
// hold 8 whole rows. Per token:
//   1. each lane's partial sums of its 8 rows (x and y, 16 values) reduce over
//      the half-warp's 16 lanes by a transposed butterfly (15 shuffles), after
//      which lane j < 8 holds x of row j and lane 8 + j holds y of row j;
//   2. lane j computes u of row j, lane 8 + j gets it by a shuffle and writes
//      o; the 8 values of u pass to the half-warp through shared memory;
//   3. each lane updates its tile, s <- bf16(d_t s + k_hat_t u), and sums the
//      rounded values against the next token's two vectors.
// Nothing waits on other warps after the prologue; the state arrives and
// leaves by 16-byte loads and stores (2-byte ones for a misaligned pool).
#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {

constexpr int VF_THREADS = 256;
constexpr int VF_WARPS = VF_THREADS / 32;

// Shared-memory carve-up (bytes) for TT token slots: the prologue's vectors,
// the next-token weights d * k_hat and d * q_hat, and each half-warp's u.
__host__ __device__ constexpr size_t vf_smem_bytes(int TT) {
  return (size_t)TT * KD * 4 * 7            // kh, qh, dd, gg, vrow, wk, wq
         + (size_t)KDA_MAX_T * 4 * 2        // beta, kappa
         + (size_t)VF_WARPS * 16 * 4;       // u of each half-warp's 8 rows
}

// Transposed butterfly over the 16 lanes of a half-warp: v[i] (i < 16) summed
// over the lanes; lane j of the half-warp returns the sum of value j. The
// order of the additions is fixed, so the result is deterministic.
__device__ __forceinline__ float halfwarp_transpose_sum(float (&v)[16], int j) {
#pragma unroll
  for (int lvl = 3; lvl >= 0; --lvl) {
    const int off = 1 << lvl;  // 8, 4, 2, 1
    const bool up = (j & off) != 0;
#pragma unroll
    for (int i = 0; i < off; ++i) {
      const float keep = up ? v[off + i] : v[i];
      const float send = up ? v[i] : v[off + i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, off));
    }
  }
  return v[0];
}

template <bool BULK, int TT>
__global__ void __launch_bounds__(VF_THREADS, 2)
    kda_verify_fused_kernel(const kda_params p, const int T) {
  static_assert(TT == 8 || TT == 16, "token slots");
  constexpr int PT = TT / VF_WARPS;  // prologue tokens per warp
  extern __shared__ __align__(16) unsigned char smem[];
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int h = blockIdx.x % p.H;
  const int b = blockIdx.x / p.H;

  float* fb = reinterpret_cast<float*>(smem);
  TokenSmem ts;
  ts.kh = fb;
  ts.qh = ts.kh + TT * KD;
  ts.dd = ts.qh + TT * KD;
  ts.gg = ts.dd + TT * KD;
  ts.vrow = ts.gg + TT * KD;
  float* wk = ts.vrow + TT * KD;
  float* wq = wk + TT * KD;
  ts.beta = wq + TT * KD;
  ts.kappa = ts.beta + KDA_MAX_T;
  ts.red = nullptr;
  float* su = ts.kappa + KDA_MAX_T + warp * 16 + (lane >> 4) * 8;  // u of this half-warp's 8 rows

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int kg = lane & 15;                       // key group: keys 8 kg .. 8 kg + 7
  const int r0 = warp * 16 + (lane >> 4) * 8;     // first of this lane's 8 rows
  const int64_t obase = (int64_t)b * p.out_b_stride + (int64_t)h * p.out_h_stride + r0 + (kg & 7);

  const int n = p.state_indices[b];
  TokenLoads<PT> first;  // issued alongside the index load
  prologue_issue<PT, VF_WARPS>(p, b, h, T, 0, KD, first);
  if (n < 0 || n >= p.N) {
    if (kg >= 8)
      for (int t = 0; t < T; ++t) outp[obase + (int64_t)t * p.out_t_stride] = 0;
    return;
  }

  // The tile, straight from the pool: 8 rows x 8 keys (16 bytes per row).
  uint16_t* grow = static_cast<uint16_t*>(p.state) + (int64_t)n * p.state_slot_stride +
                   ((int64_t)h * KD + r0) * KD + 8 * kg;
  uint32_t st[8][4];
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if constexpr (BULK) {
      const uint4 c = *reinterpret_cast<const uint4*>(grow + r * KD);
      st[r][0] = c.x;
      st[r][1] = c.y;
      st[r][2] = c.z;
      st[r][3] = c.w;
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q)
        st[r][q] = (uint32_t)grow[r * KD + 2 * q] | ((uint32_t)grow[r * KD + 2 * q + 1] << 16);
    }
  }

  token_prologue<PT, VF_WARPS>(p, b, h, T, 0, KD, ts, first);  // ends with a CTA barrier
  for (int i = tid; i < T * KD; i += VF_THREADS) {
    const float d = ts.dd[i];
    wk[i] = __fmul_rn(d, ts.kh[i]);
    wq[i] = __fmul_rn(d, ts.qh[i]);
  }
  __syncthreads();

  // Partial sums of token 0: x and y of each of the 8 rows over this lane's 8 keys.
  f32x2 ax[8], ay[8];
  {
    f32x2 wkp[4], wqp[4];
    const float4* w0 = reinterpret_cast<const float4*>(wk + 8 * kg);
    const float4* w1 = reinterpret_cast<const float4*>(wq + 8 * kg);
    const float4 a0 = w0[0], a1 = w0[1], b0 = w1[0], b1 = w1[1];
    wkp[0] = pk2(a0.x, a0.y); wkp[1] = pk2(a0.z, a0.w); wkp[2] = pk2(a1.x, a1.y); wkp[3] = pk2(a1.z, a1.w);
    wqp[0] = pk2(b0.x, b0.y); wqp[1] = pk2(b0.z, b0.w); wqp[2] = pk2(b1.x, b1.y); wqp[3] = pk2(b1.z, b1.w);
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      f32x2 s0 = bf16x2_to_f32x2(st[r][0]);
      ax[r] = mul2(wkp[0], s0);
      ay[r] = mul2(wqp[0], s0);
#pragma unroll
      for (int q = 1; q < 4; ++q) {
        const f32x2 s = bf16x2_to_f32x2(st[r][q]);
        ax[r] = fma2(wkp[q], s, ax[r]);
        ay[r] = fma2(wqp[q], s, ay[r]);
      }
    }
  }

  for (int t = 0; t < T; ++t) {
    // 1-2. The rows' sums, u and o.
    float v16[16];
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      float lo, hi;
      upk2(ax[r], lo, hi);
      v16[r] = __fadd_rn(lo, hi);
      upk2(ay[r], lo, hi);
      v16[8 + r] = __fadd_rn(lo, hi);
    }
    const float sum = halfwarp_transpose_sum(v16, kg);  // x of row kg (kg < 8), y of row kg - 8
    const int row = r0 + (kg & 7);
    float u = 0.0f;
    if (kg < 8) {
      u = __fmul_rn(ts.beta[t], __fsub_rn(ts.vrow[t * KD + row], sum));
      su[kg] = u;
    }
    u = __shfl_xor_sync(0xffffffffu, u, 8);  // lane 8 + j gets row j's u
    if (kg >= 8) {
      const float o = __fmul_rn(p.scale, __fmaf_rn(u, ts.kappa[t], sum));
      outp[obase + (int64_t)t * p.out_t_stride] = float_to_bf16_bits(o);
    }
    __syncwarp();
    float ur[8];
    {
      const float4 u0 = reinterpret_cast<const float4*>(su)[0], u1 = reinterpret_cast<const float4*>(su)[1];
      ur[0] = u0.x; ur[1] = u0.y; ur[2] = u0.z; ur[3] = u0.w;
      ur[4] = u1.x; ur[5] = u1.y; ur[6] = u1.z; ur[7] = u1.w;
    }

    // 3. The update, s <- bf16(d_t s + k_hat_t u), and the next token's partial sums.
    f32x2 dp[4], kp[4], wkp[4], wqp[4];
    {
      const float4* d4 = reinterpret_cast<const float4*>(ts.dd + t * KD + 8 * kg);
      const float4* k4 = reinterpret_cast<const float4*>(ts.kh + t * KD + 8 * kg);
      const float4 d0 = d4[0], d1 = d4[1], k0 = k4[0], k1 = k4[1];
      dp[0] = pk2(d0.x, d0.y); dp[1] = pk2(d0.z, d0.w); dp[2] = pk2(d1.x, d1.y); dp[3] = pk2(d1.z, d1.w);
      kp[0] = pk2(k0.x, k0.y); kp[1] = pk2(k0.z, k0.w); kp[2] = pk2(k1.x, k1.y); kp[3] = pk2(k1.z, k1.w);
    }
    const bool more = t + 1 < T;
    if (more) {
      const float4* w0 = reinterpret_cast<const float4*>(wk + (t + 1) * KD + 8 * kg);
      const float4* w1 = reinterpret_cast<const float4*>(wq + (t + 1) * KD + 8 * kg);
      const float4 a0 = w0[0], a1 = w0[1], b0 = w1[0], b1 = w1[1];
      wkp[0] = pk2(a0.x, a0.y); wkp[1] = pk2(a0.z, a0.w); wkp[2] = pk2(a1.x, a1.y); wkp[3] = pk2(a1.z, a1.w);
      wqp[0] = pk2(b0.x, b0.y); wqp[1] = pk2(b0.z, b0.w); wqp[2] = pk2(b1.x, b1.y); wqp[3] = pk2(b1.z, b1.w);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) wkp[q] = wqp[q] = pk2(0.0f, 0.0f);
    }
#pragma unroll
    for (int r = 0; r < 8; ++r) {
      const f32x2 uu = pk2(ur[r], ur[r]);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        f32x2 a = mul2(dp[q], bf16x2_to_f32x2(st[r][q]));
        a = fma2(kp[q], uu, a);
        st[r][q] = f32x2_to_bf16x2(a);
        const f32x2 s = bf16x2_to_f32x2(st[r][q]);
        ax[r] = q == 0 ? mul2(wkp[0], s) : fma2(wkp[q], s, ax[r]);
        ay[r] = q == 0 ? mul2(wqp[0], s) : fma2(wqp[q], s, ay[r]);
      }
    }
    __syncwarp();  // every lane has read su before the next token writes it
  }

  // The final tile back into the pool.
#pragma unroll
  for (int r = 0; r < 8; ++r) {
    if constexpr (BULK) {
      *reinterpret_cast<uint4*>(grow + r * KD) = make_uint4(st[r][0], st[r][1], st[r][2], st[r][3]);
    } else {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        grow[r * KD + 2 * q] = (uint16_t)(st[r][q] & 0xffffu);
        grow[r * KD + 2 * q + 1] = (uint16_t)(st[r][q] >> 16);
      }
    }
  }
}

template <bool BULK, int TT>
static cudaError_t launch_vf(const kda_params& p, int T, cudaStream_t s) {
  auto kern = kda_verify_fused_kernel<BULK, TT>;
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, vf_smem_bytes(TT), smem_set);
  if (e != cudaSuccess) return e;
  kern<<<(unsigned)((long long)p.B * p.H), VF_THREADS, vf_smem_bytes(TT), s>>>(p, T);
  return cudaGetLastError();
}

cudaError_t launch_verify_fused(const kda_params& p, int T, bool bulk, cudaStream_t s) {
  if (bulk) return T <= 8 ? launch_vf<true, 8>(p, T, s) : launch_vf<true, 16>(p, T, s);
  return T <= 8 ? launch_vf<false, 8>(p, T, s) : launch_vf<false, 16>(p, T, s);
}

}  // namespace kda
