// kda_ring.cu - ring-cache verify with replay and fold for sm_103a.
//
// Source: "feat(kda): ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)"
// (PR #4864), sections "What it does", "API" and "Caching": instead of writing
// the state back every verify, append (k_hat, u, G) to a per-slot ring, compute
// outputs from the checkpoint plus the ring with per-channel weights
// exp(G_P - G_j), and fold the ring into the checkpoint once hist_len reaches
// flush_min.
//
// One CTA (128 threads) per (batch row, head, tile of TV = 16, 32 or 64 value rows):
//   1. slot lookup, hist_len check (outside [0, W]: error bit, skip);
//   2. bulk copy of the checkpoint rows into shared memory (per warp);
//   3. per-token prologue, then per channel: k~ = bf16(k_hat),
//      G_P = fp32(G_{P-1} + g), decay exp(G_P - G_{P-1}), k~ . q_hat;
//   4. rows go to registers as fp32 and are replayed through the history in
//      chunks of HC entries staged in shared memory:
//      s <- exp(G_j - G_{j-1}) s + k_j u_j[v];
//   5. fold (hist_len >= flush_min): rows are rounded to bf16, bulk-stored to
//      the checkpoint and continue from the rounded values;
//   6. the T tokens: a = D s; x = a . k~; y = a . q_hat; u~ = bf16(beta (v - x));
//      s <- a + k~ u~; o = scale (y + u~ (k~ . q_hat)); outputs and this
//      tile's rows of u~ written (rows no other CTA reads).
// A second, stream-ordered kernel (one CTA per batch row) appends k~ and G_P
// and resets hist_len after a fold. Both are shared by every tile and head of
// a slot: after a fold the new entries overwrite ring positions 0..T-1 that
// other CTAs of the first kernel may still be replaying, and a reset
// hist_len must not be seen by a CTA that has not read it yet. The second
// kernel recomputes k~ and G with the same arithmetic, so the bits match.
#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {

constexpr int HC = 8;  // history entries staged per chunk

__host__ __device__ constexpr size_t ring_smem_bytes(int TV, int T) {
  return (size_t)TV * KD * 2                   // checkpoint tile (bf16)
         + 64                                    // mbarriers
         + (size_t)T * KD * 4 * 4                // kh (k~), qh, dd (decay), gg (g)
         + (size_t)T * TV * 4 * 3                // vrow, orow, urow
         + (size_t)KDA_MAX_T * 4 * 2             // beta, kappa
         + (size_t)KDA_MAX_T * NWARPS * 3 * 4    // reduction partials
         + (size_t)HC * KD * 4 * 2               // history k, decay
         + (size_t)HC * TV * 4;                  // history u rows
}

__device__ __forceinline__ float round_bf16(float x) { return bf16_bits_to_float(float_to_bf16_bits(x)); }

template <int TV, bool BULK>
__global__ void __launch_bounds__(NTHREADS)
    kda_ring_kernel(const kda_params p, const kda_ring_params rp, const int T, const int tiles) {
  static_assert(TV % 16 == 0 && TV >= 16 && TV <= 64, "ring tile must be 16, 32 or 64 rows");
  constexpr int RW = TV / NWARPS;         // rows per warp
  constexpr int RQ = RW / ROWS_PER_WARP;  // 4-row groups per warp
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
  float* urow = orow + T * TV;
  ts.beta = urow + T * TV;
  ts.kappa = ts.beta + KDA_MAX_T;
  ts.red = ts.kappa + KDA_MAX_T;
  float* hk = ts.red + KDA_MAX_T * NWARPS * 3;  // [HC][128]
  float* hd = hk + HC * KD;                     // [HC][128]
  float* hu = hd + HC * KD;                     // [HC][TV]

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t out_base = (int64_t)b * p.out_b_stride + (int64_t)h * p.out_h_stride + v0;

  const int n = p.state_indices[b];
  TokenLoads first;  // issued alongside the index load; unused by an inactive row
  prologue_issue(p, b, h, 0, T, v0, TV, first);
  if (n < 0 || n >= p.N) {
    for (int i = tid; i < T * TV; i += NTHREADS) {
      const int t = i / TV, r = i - t * TV;
      outp[out_base + (int64_t)t * p.out_t_stride + r] = 0;
    }
    return;
  }

  // The checkpoint copy starts before hist_len is known: reading it is harmless
  // even when the history turns out to be invalid.
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
  }
  const int hist = rp.hist_len[n];
  if (hist < 0 || hist > rp.W) {
    if (tid == 0 && tile == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_HIST_LEN);
    if constexpr (BULK) {
      __syncwarp();
      if (!mbar_wait_bounded(&mbar[warp], 0) && lane == 0 && p.error_word != nullptr)
        atomicOr(p.error_word, KDA_ERR_TIMEOUT);  // the copy must land before the CTA leaves
    }
    for (int i = tid; i < T * TV; i += NTHREADS) {
      const int t = i / TV, r = i - t * TV;
      outp[out_base + (int64_t)t * p.out_t_stride + r] = 0;
    }
    return;
  }
  if constexpr (!BULK) {
    for (int i = lane; i < RW * KD; i += 32) sst[i] = gst[i];
  }
  const bool fold = hist >= rp.flush_min;
  const int base = fold ? 0 : hist;

  // Ring slices of this (slot, head).
  uint16_t* kc = static_cast<uint16_t*>(rp.k_cache) + (int64_t)n * rp.k_slot_stride + (int64_t)h * rp.W * KD;
  uint16_t* uc = static_cast<uint16_t*>(rp.u_cache) + (int64_t)n * rp.u_slot_stride + (int64_t)h * rp.W * KD;
  float* gc = static_cast<float*>(rp.g_cache) + (int64_t)n * rp.g_slot_stride + (int64_t)h * rp.W * KD;

  token_prologue(p, b, h, T, v0, TV, ts, first);  // ends with a CTA barrier

  // Per channel: k~, G, the decay exp(G_P - G_{P-1}) and the partial sums of k~ . q_hat.
  {
    const int c = tid;
    float G_prev = (!fold && hist > 0) ? gc[(int64_t)(hist - 1) * KD + c] : 0.0f;
    float kq[KDA_MAX_T];
    for (int t = 0; t < T; ++t) {
      const float kt = round_bf16(ts.kh[t * KD + c]);
      const float G = __fadd_rn(G_prev, ts.gg[t * KD + c]);
      ts.dd[t * KD + c] = expf(__fsub_rn(G, G_prev));
      ts.kh[t * KD + c] = kt;
      kq[t] = __fmul_rn(kt, ts.qh[t * KD + c]);
      G_prev = G;
    }
    for (int t = 0; t < T; ++t) {
      const float s = warp_sum(kq[t]);
      if (lane == 0) ts.red[(t * NWARPS + warp) * 3] = s;
    }
  }
  __syncthreads();
  if (tid < T) {
    const float* r = ts.red + tid * NWARPS * 3;
    float s = r[0];
#pragma unroll
    for (int w = 1; w < NWARPS; ++w) s = __fadd_rn(s, r[w * 3]);
    ts.kappa[tid] = s;
  }

  bool ok = true;
  __syncwarp();
  if constexpr (BULK) ok = mbar_wait_bounded(&mbar[warp], 0);
  if (!ok && lane == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
  // The tile is written only if every warp's copy arrived; a CTA that gave up
  // writes zero output and leaves the checkpoint and ring alone. The barrier
  // also publishes kappa.
  ok = __syncthreads_and(ok) != 0;

  const int r = lane / LPR, j = lane % LPR;  // row within a 4-row group, lane within the row
  f32x2 s[RQ][8];  // the lane's 16 keys of each of its rows, fp32
#pragma unroll
  for (int q = 0; q < RQ; ++q) row_to_f32(load_row_bf16(st + (warp * RW + ROWS_PER_WARP * q + r) * KD, j), s[q]);

  // Replay the live history in chunks: s <- exp(G_j - G_{j-1}) s + k_j u_j[v].
  for (int j0 = 0; j0 < hist; j0 += HC) {
    const int nj = min(HC, hist - j0);
    __syncthreads();  // previous chunk consumed
    {
      const int c = tid;
      for (int jj = 0; jj < nj; ++jj) {
        const int jx = j0 + jj;
        hk[jj * KD + c] = bf16_bits_to_float(kc[(int64_t)jx * KD + c]);
        const float Gj = gc[(int64_t)jx * KD + c];
        const float Gm = jx > 0 ? gc[(int64_t)(jx - 1) * KD + c] : 0.0f;
        hd[jj * KD + c] = expf(__fsub_rn(Gj, Gm));
        if (c < TV) hu[jj * TV + c] = bf16_bits_to_float(uc[(int64_t)jx * KD + v0 + c]);
      }
    }
    __syncthreads();
    for (int jj = 0; jj < nj; ++jj) {
      f32x2 kr[8], dr[8];
      load_pairs8(hk + jj * KD, j, kr);
      load_pairs8(hd + jj * KD, j, dr);
#pragma unroll
      for (int q = 0; q < RQ; ++q) {
        const float uv = hu[jj * TV + warp * RW + ROWS_PER_WARP * q + r];
        const f32x2 uu = pk2(uv, uv);
#pragma unroll
        for (int i = 0; i < 8; ++i) s[q][i] = fma2(kr[i], uu, mul2(dr[i], s[q][i]));
      }
    }
  }

  if (fold && ok) {
#pragma unroll
    for (int q = 0; q < RQ; ++q) {
      const RowBf16 w = row_to_bf16(s[q]);
      store_row_bf16(st + (warp * RW + ROWS_PER_WARP * q + r) * KD, j, w);
      row_to_f32(w, s[q]);
    }
    if constexpr (BULK) {
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        bulk_s2g(gst, sst, CHUNK_BYTES);
        bulk_commit();
      }
    } else {
      __syncwarp();
      for (int i = lane; i < RW * KD; i += 32) gst[i] = sst[i];
    }
  }

  // The new tokens, state kept in fp32: a = D s; u~ = bf16(beta (v - a . k~));
  // s <- a + k~ u~; o = scale (a . q_hat + u~ (k~ . q_hat)).
  for (int t = 0; t < T; ++t) {
    LaneVecs lv;
    load_lane_vecs(ts, t, j, lv);
    const float beta = ts.beta[t], kappa = ts.kappa[t];
#pragma unroll
    for (int q = 0; q < RQ; ++q) {
      const int row = warp * RW + ROWS_PER_WARP * q + r;
      f32x2 a[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) a[i] = mul2(lv.dd[i], s[q][i]);
      float x, y, u, yr;
      partial_dots(a, lv, x, y);
      row_reduce(x, y, j, beta, ts.vrow[t * TV + row], u, yr);
      u = round_bf16(u);
      const f32x2 uu = pk2(u, u);
#pragma unroll
      for (int i = 0; i < 8; ++i) s[q][i] = fma2(lv.kh[i], uu, a[i]);
      if (j == 0) {
        urow[t * TV + row] = u;
        orow[t * TV + row] = ok ? __fmul_rn(p.scale, __fmaf_rn(u, kappa, yr)) : 0.0f;
      }
    }
  }
  if (fold && ok && BULK && lane == 0) bulk_wait_read_all();
  __syncthreads();
  for (int i = tid; i < T * TV; i += NTHREADS) {
    const int t = i / TV, rr = i - t * TV;
    outp[out_base + (int64_t)t * p.out_t_stride + rr] = float_to_bf16_bits(orow[i]);
    if (ok) uc[(int64_t)(base + t) * KD + v0 + rr] = float_to_bf16_bits(urow[i]);
  }
}

// Sum over the 128 key channels in the order token_prologue uses (thread c =
// 32 w + l sums within its warp by butterfly, then warps 0..3 in order). Lane
// l holds channels l, 32 + l, 64 + l, 96 + l.
__device__ __forceinline__ float sum128_like_cta(const float (&x)[4]) {
  float s = warp_sum(x[0]);
#pragma unroll
  for (int w = 1; w < 4; ++w) s = __fadd_rn(s, warp_sum(x[w]));
  return s;
}

// After the ring kernel, one CTA per batch row: append k~ and G_P at ring
// positions base..base+T-1 for every head, then reset hist_len[n] after a
// fold when restart_hist_on_flush. Warp w handles heads w, w+4, ...; lane l
// handles channels l + 32 i. The arithmetic of k~ and G repeats
// token_prologue and the ring kernel's channel pass operation for operation.
__global__ void __launch_bounds__(NTHREADS)
    kda_ring_append_kernel(const kda_params p, const kda_ring_params rp, const int T) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.state_indices[b];
  if (n < 0 || n >= p.N) return;
  const int hist = rp.hist_len[n];
  if (hist < 0 || hist > rp.W) return;
  const bool fold = hist >= rp.flush_min;
  const int base = fold ? 0 : hist;
  for (int h = warp; h < p.H; h += NWARPS) {
    uint16_t* kc = static_cast<uint16_t*>(rp.k_cache) + (int64_t)n * rp.k_slot_stride + (int64_t)h * rp.W * KD;
    float* gc = static_cast<float*>(rp.g_cache) + (int64_t)n * rp.g_slot_stride + (int64_t)h * rp.W * KD;
    const float a_h = expf(p.A_log[h]);
    float G_prev[4], dtb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      dtb[i] = p.dt_bias[(int64_t)h * KD + c];
      G_prev[i] = (!fold && hist > 0) ? gc[(int64_t)(hist - 1) * KD + c] : 0.0f;
    }
    for (int t = 0; t < T; ++t) {
      float kc4[4], sq[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        kc4[i] = load_bf16(p.k, b, t, h, lane + 32 * i);
        sq[i] = __fmul_rn(kc4[i], kc4[i]);
      }
      const float rk = __frcp_rn(__fsqrt_rn(__fadd_rn(sum128_like_cta(sq), L2_EPS)));
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int c = lane + 32 * i;
        const float gr = load_bf16(p.g_raw, b, t, h, c);
        const float z = __fmul_rn(a_h, __fadd_rn(gr, dtb[i]));
        const float sig = __frcp_rn(__fadd_rn(1.0f, expf(-z)));
        const float g = __fmul_rn(p.lower_bound, sig);
        const float G = __fadd_rn(G_prev[i], g);
        kc[(int64_t)(base + t) * KD + c] = float_to_bf16_bits(__fmul_rn(kc4[i], rk));
        gc[(int64_t)(base + t) * KD + c] = G;
        G_prev[i] = G;
      }
    }
  }
  if (fold && rp.restart_hist_on_flush) {
    __syncthreads();
    if (threadIdx.x == 0) rp.hist_len[n] = 0;
  }
}

template <int TV, bool BULK>
static cudaError_t launch_ring_one(const kda_params& p, int T, const kda_ring_params& r, cudaStream_t s) {
  auto kern = kda_ring_kernel<TV, BULK>;
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, ring_smem_bytes(TV, KDA_MAX_T), smem_set);
  if (e != cudaSuccess) return e;
  const int tiles = KD / TV;
  const long long blocks = (long long)p.B * p.H * tiles;
  kern<<<(unsigned)blocks, NTHREADS, ring_smem_bytes(TV, T), s>>>(p, r, T, tiles);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  kda_ring_append_kernel<<<(unsigned)p.B, NTHREADS, 0, s>>>(p, r, T);
  return cudaGetLastError();
}

cudaError_t launch_ring(const kda_params& p, int T, const kda_ring_params& r, int tile_v, bool bulk,
                        cudaStream_t s) {
  if (tile_v > 64) tile_v = 64;
  switch (tile_v) {
    case 16: return bulk ? launch_ring_one<16, true>(p, T, r, s) : launch_ring_one<16, false>(p, T, r, s);
    case 32: return bulk ? launch_ring_one<32, true>(p, T, r, s) : launch_ring_one<32, false>(p, T, r, s);
    case 64: return bulk ? launch_ring_one<64, true>(p, T, r, s) : launch_ring_one<64, false>(p, T, r, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
