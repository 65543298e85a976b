// kda_ring.cu - ring-cache verify with replay and fold for sm_103a.
//
// Source: "feat(kda): ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)"
// (PR #4864), sections "What it does", "API" and "Caching": instead of writing
// the state back every verify, append (k_hat, u, G) to a per-slot ring, compute
// outputs from the checkpoint plus the ring with per-channel weights
// exp(G_P - G_j), and fold the ring into the checkpoint once hist_len reaches
// flush_min.
//
// The step it computes, per (row, head): with base state S_b and token decays
// d_t = exp(G_t - G_{t-1}),
//   u~_t = bf16(beta_t (v_t - (D_t S_{t-1})^T k~_t)),  S_t = D_t S_{t-1} + k~_t u~_t^T,
//   o_t  = scale S_t^T q_hat_t.
// Unrolled over the tokens (the WY form of these pages' replay), with
// P_t = d_0 * ... * d_t and w_tj = P_t / P_j = d_{j+1} * ... * d_t:
//   (D_t S_{t-1})^T k~_t = S_b^T (P_t k~_t) + sum_{j<t}  u~_j (w_tj k~_j) . k~_t
//   S_t^T q_hat_t        = S_b^T (P_t q_hat_t) + sum_{j<=t} u~_j (w_tj k~_j) . q_hat_t
// so each state row is read once for 2T dot products, and the token-to-token
// dependence shrinks to a T-step scalar recurrence per row over the T x T
// coefficients cc[t][j] = (w_tj k~_j) . k~_t and ec[t][j] = (w_tj k~_j) . q_hat_t.
// The base state is the checkpoint replayed through the h live entries, in
// closed form with the pages' replay weights:
//   S_h = diag(exp(G_{h-1})) S_0 + sum_{j<h} (exp(G_{h-1} - G_j) k~_j) u~_j^T;
// a fold (h >= flush_min) rounds S_h to bf16, stores it as the new checkpoint
// and uses the rounded state as the base (G restarts at 0); otherwise S_h
// stays in fp32 and G continues from G_{h-1}.
//
// One CTA per (batch row, head, tile of TV = 16, 32, 64 or 128 rows), 4 warps
// (8 for the whole-head tile):
//   1. slot lookup, checkpoint bulk copy, hist_len check (outside [0, W]:
//      error bit, skip);
//   2. per-token prologue; per channel: k~, G, d_t, P_t, the query vectors
//      P_t k~_t and P_t q_hat_t, exp(G_{h-1}), the history keys;
//   3. the coefficient matrices, one warp per column j;
//   4. per 4-row group pair: base rows (replay, fold), the 2T dot products,
//      a reduce-scatter that leaves token t's two sums on lane t % 8 of the
//      row, and the T-step recurrence for u~_t and o_t;
//   5. outputs and this tile's rows of u~ (rows no other CTA reads).
// A second, stream-ordered kernel (one CTA per batch row) appends k~ and G
// and resets hist_len after a fold. Both are shared by every tile and head of
// a slot: after a fold the new entries overwrite ring positions 0..T-1 that
// other CTAs of the first kernel may still be replaying, and a reset
// hist_len must not be seen by a CTA that has not read it yet. The second
// kernel recomputes k~ and G with the same arithmetic, so the bits match.
#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {

__host__ __device__ constexpr size_t ring_smem_bytes(int TV, int T, int W) {
  return (size_t)TV * KD * 2                        // checkpoint tile (bf16)
         + 64                                         // mbarriers
         + (size_t)T * KD * 4 * 4                     // kh (k~), qh, dd (d_t), gg (g, then P_t k~_t)
         + (size_t)T * KD * 4                         // qq = P_t q_hat_t
         + (size_t)T * TV * 4 * 3                     // vrow, orow, urow
         + (size_t)KDA_MAX_T * 4 * 2                  // beta, kappa
         + (size_t)KDA_MAX_T * KDA_MAX_T * 4 * 2      // cc, ec
         + (size_t)KD * 4                             // exp(G_{h-1})
         + (size_t)W * KD * 4                         // history G, then history keys (in place)
         + (size_t)W * KD * 2                         // history k~ (bf16, as stored)
         + (size_t)W * TV * 2                         // history u~ of this tile's rows (bf16)
         + 16;                                        // history mbarrier
}

__device__ __forceinline__ float round_bf16(float x) { return bf16_bits_to_float(float_to_bf16_bits(x)); }

// Dot product of a lane's 16 keys of a row with the lane's 16 keys of a vector.
__device__ __forceinline__ float dot16(const f32x2 (&vec)[8], const f32x2 (&row)[8]) {
  f32x2 xa = mul2(vec[0], row[0]), xb = mul2(vec[1], row[1]);
#pragma unroll
  for (int i = 2; i < 8; i += 2) {
    xa = fma2(vec[i], row[i], xa);
    xb = fma2(vec[i + 1], row[i + 1], xb);
  }
  float x0, x1, x2, x3;
  upk2(xa, x0, x1);
  upk2(xb, x2, x3);
  return __fadd_rn(__fadd_rn(x0, x2), __fadd_rn(x1, x3));
}

// Slot of token t's sum ("which" = 0: with k~, 1: with q_hat) among the 2 TT
// values a lane holds before the reduce-scatter; after it, lane j of the row
// holds slots [j * 2TT/8, (j + 1) * 2TT/8), that is tokens j and j + 8.
template <int TT>
__device__ __forceinline__ constexpr int wy_slot(int t, int which) {
  return TT == 8 ? 2 * t + which : 4 * (t & 7) + 2 * (t >> 3) + which;
}

// Reduce-scatter of NV per-lane values over the 8 lanes of a row: at the
// level with lane mask m, a lane keeps the half of its current values picked
// by bit m of its row lane and sends the other half to lane ^ m, who keeps it.
template <int NV>
__device__ __forceinline__ void reduce_scatter8(float (&v)[NV], int j) {
#pragma unroll
  for (int m = 4, c = NV; m >= 1; m >>= 1, c >>= 1) {
    const bool hi = (j & m) != 0;
#pragma unroll
    for (int i = 0; i < c / 2; ++i) {
      const float keep = hi ? v[c / 2 + i] : v[i];
      const float send = hi ? v[i] : v[c / 2 + i];
      v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
    }
  }
}

// Reduce-scatter of NV (16 or 32) per-lane values over a whole warp: halving
// levels (as in reduce_scatter8) while a lane holds more than one value, then
// plain butterfly levels. Afterwards v[0] holds the warp-wide sum of value
// lane >> (5 - log2 NV); each value is summed in one fixed order.
template <int NV>
__device__ __forceinline__ void reduce_scatter32(float (&v)[NV], int lane) {
  static_assert(NV == 16 || NV == 32, "16 or 32 values");
  int c = NV;
#pragma unroll
  for (int m = 16; m >= 1; m >>= 1) {
    if (c > 1) {
      const bool hi = (lane & m) != 0;
#pragma unroll
      for (int i = 0; i < NV / 2; ++i) {
        if (i < c / 2) {
          const float keep = hi ? v[c / 2 + i] : v[i];
          const float send = hi ? v[i] : v[c / 2 + i];
          v[i] = __fadd_rn(keep, __shfl_xor_sync(0xffffffffu, send, m));
        }
      }
      c >>= 1;
    } else {
      v[0] = __fadd_rn(v[0], __shfl_xor_sync(0xffffffffu, v[0], m));
    }
  }
}

template <int TV, bool BULK, int TT, int NW>
__global__ void __launch_bounds__(32 * NW)
    kda_ring_kernel(const kda_params p, const kda_ring_params rp, const int T, const int tiles) {
  static_assert(TV % 16 == 0 && TV >= 16 && TV <= 128, "ring tile must be 16, 32, 64 or 128 rows");
  static_assert(TT == 8 || TT == 16, "token slots");
  static_assert(NW == 4 || NW == 8, "4 or 8 warps");
  static_assert(TV % (4 * NW) == 0, "every warp owns whole 4-row groups");
  constexpr int NT = 32 * NW;             // threads
  constexpr int RW = TV / NW;             // rows per warp
  constexpr int RQ = RW / ROWS_PER_WARP;  // 4-row groups per warp
  constexpr int RG = RQ < 2 ? RQ : 2;     // groups processed together
  constexpr int NV = 2 * TT;              // sums per row before the reduce-scatter
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
  float* qk = ts.gg;  // each thread overwrites its channel's g_t with P_t k~_t in the channel pass
  float* qq = ts.gg + T * KD;
  ts.vrow = qq + T * KD;
  float* orow = ts.vrow + T * TV;
  float* urow = orow + T * TV;
  ts.beta = urow + T * TV;
  ts.kappa = ts.beta + KDA_MAX_T;
  float* cc = ts.kappa + KDA_MAX_T;             // [t][j], j < t
  float* ec = cc + KDA_MAX_T * KDA_MAX_T;       // [t][j], j <= t
  float* cdec = ec + KDA_MAX_T * KDA_MAX_T;     // [128] exp(G_{h-1})
  float* hk = cdec + KD;                        // [W][128] G_j as copied, then exp(G_{h-1} - G_j) k~_j
  uint16_t* hkb = reinterpret_cast<uint16_t*>(hk + rp.W * KD);  // [W][128] k~_j (bf16)
  uint16_t* hub = hkb + rp.W * KD;                               // [W][TV] u~_j[v0..v0+TV) (bf16)
  uint64_t* hbar = reinterpret_cast<uint64_t*>(hub + rp.W * TV);  // history copies

  uint16_t* outp = static_cast<uint16_t*>(p.out);
  const int64_t out_base = (int64_t)b * p.out_b_stride + (int64_t)h * p.out_h_stride + v0;

  const int n = p.state_indices[b];
  constexpr int PT = TT / NW;  // tokens per warp in the prologue
  TokenLoads<PT> first;        // issued alongside the index load; unused by an inactive row
  prologue_issue<PT, NW>(p, b, h, T, v0, TV, first);
  if (n < 0 || n >= p.N) {
    for (int i = tid; i < T * TV; i += NT) {
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
    for (int i = tid; i < T * TV; i += NT) {
      const int t = i / TV, r = i - t * TV;
      outp[out_base + (int64_t)t * p.out_t_stride + r] = 0;
    }
    return;
  }
  const bool fold = hist >= rp.flush_min;
  const int base = fold ? 0 : hist;

  // Ring slices of this (slot, head).
  uint16_t* kc = static_cast<uint16_t*>(rp.k_cache) + (int64_t)n * rp.k_slot_stride + (int64_t)h * rp.W * KD;
  uint16_t* uc = static_cast<uint16_t*>(rp.u_cache) + (int64_t)n * rp.u_slot_stride + (int64_t)h * rp.W * KD;
  float* gc = static_cast<float*>(rp.g_cache) + (int64_t)n * rp.g_slot_stride + (int64_t)h * rp.W * KD;

  // The live history arrives by bulk copies started now, so that its latency
  // overlaps the prologue: k~ and G of entries 0..hist-1 are contiguous, this
  // tile's u~ rows are one short copy per entry. The ring pointers and slot
  // strides are 16-byte aligned (checked on the host), v0 is a multiple of 16.
  if (hist > 0 && tid == 0) {
    mbar_init(hbar, 1);
    mbar_expect_tx(hbar, (uint32_t)hist * (KD * 2 + KD * 4 + TV * 2));
    bulk_g2s(hkb, kc, (uint32_t)hist * KD * 2, hbar);
    bulk_g2s(hk, gc, (uint32_t)hist * KD * 4, hbar);
    for (int jx = 0; jx < hist; ++jx) bulk_g2s(hub + jx * TV, uc + (int64_t)jx * KD + v0, TV * 2, hbar);
  }
  if constexpr (!BULK) {
    for (int i = lane; i < RW * KD; i += 32) sst[i] = gst[i];
  }

  token_prologue<PT, NW>(p, b, h, T, v0, TV, ts, first);  // ends with a CTA barrier (publishes hbar's init)

  bool hist_ok = true;
  if (hist > 0) hist_ok = mbar_wait_bounded(hbar, 0);
  if (!hist_ok && tid == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);

  // Channel pass, thread c (and c + 128 with 8 warps) = key channel c.
  {
    const int c = tid & (KD - 1), part = tid / KD;
    const float Gl = hist > 0 ? hk[(hist - 1) * KD + c] : 0.0f;  // G_{h-1}
    if (part == 0) cdec[c] = hist > 0 ? expf(Gl) : 1.0f;
    if (NT > KD) __syncthreads();  // every thread has read G_{h-1} before entry h-1 is overwritten
    for (int jx = part; jx < hist; jx += NT / KD) {  // in place: G_j -> exp(G_{h-1} - G_j) k~_j
      const float kj = bf16_bits_to_float(hkb[jx * KD + c]);
      hk[jx * KD + c] = __fmul_rn(expf(__fsub_rn(Gl, hk[jx * KD + c])), kj);
    }
    float G_prev = fold ? 0.0f : Gl;
    float P = 1.0f;
    for (int t = 0; t < (part == 0 ? T : 0); ++t) {
      const float kt = round_bf16(ts.kh[t * KD + c]);
      const float G = __fadd_rn(G_prev, ts.gg[t * KD + c]);
      const float d = expf(__fsub_rn(G, G_prev));
      P = __fmul_rn(P, d);
      ts.kh[t * KD + c] = kt;
      ts.dd[t * KD + c] = d;
      qk[t * KD + c] = __fmul_rn(P, kt);
      qq[t * KD + c] = __fmul_rn(P, ts.qh[t * KD + c]);
      G_prev = G;
    }
  }
  __syncthreads();

  // Coefficients, warp w for columns j = w, w + 4, ...; lane l sums channels
  // l + 32 i; w_tj is a running product of the token decays. A column's 2 TT
  // partial sums (cc and ec for every t) are reduced together, see
  // reduce_scatter32.
  for (int j = warp; j < T; j += NW) {
    float kj[4], wgt[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      kj[i] = ts.kh[j * KD + lane + 32 * i];
      wgt[i] = 1.0f;
    }
    float vals[2 * TT];
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      float sc = 0.0f, se = 0.0f;
      if (t >= j && t < T) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = lane + 32 * i;
          if (t > j) wgt[i] = __fmul_rn(wgt[i], ts.dd[t * KD + c]);
          const float pj = __fmul_rn(wgt[i], kj[i]);
          sc = __fmaf_rn(pj, ts.kh[t * KD + c], sc);
          se = __fmaf_rn(pj, ts.qh[t * KD + c], se);
        }
      }
      vals[2 * t] = sc;
      vals[2 * t + 1] = se;
    }
    reduce_scatter32<2 * TT>(vals, lane);
    constexpr int SHIFT = (2 * TT == 16) ? 1 : 0;  // lanes per result
    if ((lane & ((1 << SHIFT) - 1)) == 0) {
      const int idx = lane >> SHIFT, t = idx >> 1;
      if (t >= j && t < T) {
        if (idx & 1)
          ec[t * KDA_MAX_T + j] = vals[0];
        else if (t > j)
          cc[t * KDA_MAX_T + j] = vals[0];
      }
    }
  }

  bool ok = true;
  __syncwarp();
  if constexpr (BULK) ok = mbar_wait_bounded(&mbar[warp], 0);
  if (!ok && lane == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
  // The tile is written only if every warp's copy arrived; a CTA that gave up
  // writes zero output and leaves the checkpoint and ring alone. The barrier
  // also publishes the coefficients.
  ok = __syncthreads_and(ok && hist_ok) != 0;

  const int r = lane / LPR, j = lane % LPR;  // row within a 4-row group, lane within the row
  for (int g = 0; g < RQ; g += RG) {
    f32x2 s[RG][8];
    int rows[RG];
#pragma unroll
    for (int q = 0; q < RG; ++q) {
      rows[q] = warp * RW + ROWS_PER_WARP * (g + q) + r;
      row_to_f32(load_row_bf16(st + rows[q] * KD, j), s[q]);
    }
    // base = exp(G_{h-1}) S_0 + sum_j (exp(G_{h-1} - G_j) k~_j) u~_j[row]
    if (hist > 0) {
      f32x2 cv[8];
      load_pairs8(cdec, j, cv);
#pragma unroll
      for (int q = 0; q < RG; ++q)
#pragma unroll
        for (int i = 0; i < 8; ++i) s[q][i] = mul2(cv[i], s[q][i]);
      for (int jx = 0; jx < hist; ++jx) {
        f32x2 kr[8];
        load_pairs8(hk + jx * KD, j, kr);
#pragma unroll
        for (int q = 0; q < RG; ++q) {
          const float uv = bf16_bits_to_float(hub[jx * TV + rows[q]]);
          const f32x2 uu = pk2(uv, uv);
#pragma unroll
          for (int i = 0; i < 8; ++i) s[q][i] = fma2(kr[i], uu, s[q][i]);
        }
      }
    }
    if (fold) {
#pragma unroll
      for (int q = 0; q < RG; ++q) {
        const RowBf16 w = row_to_bf16(s[q]);
        if (ok) store_row_bf16(st + rows[q] * KD, j, w);
        row_to_f32(w, s[q]);
      }
    }
    // 2T dot products of each base row: S_b^T (P_t k~_t) and S_b^T (P_t q_hat_t).
    float acc[RG][NV];
#pragma unroll
    for (int q = 0; q < RG; ++q)
#pragma unroll
      for (int i = 0; i < NV; ++i) acc[q][i] = 0.0f;
#pragma unroll
    for (int t = 0; t < TT; ++t) {
      if (t < T) {
        f32x2 vk[8], vq[8];
        load_pairs8(qk + t * KD, j, vk);
        load_pairs8(qq + t * KD, j, vq);
#pragma unroll
        for (int q = 0; q < RG; ++q) {
          acc[q][wy_slot<TT>(t, 0)] = dot16(vk, s[q]);
          acc[q][wy_slot<TT>(t, 1)] = dot16(vq, s[q]);
        }
      }
    }
    // The T-step recurrence; lane j of the row owns tokens j and j + 8.
#pragma unroll
    for (int q = 0; q < RG; ++q) {
      reduce_scatter8<NV>(acc[q], j);
      const int row = rows[q];
      float cu[2] = {0.0f, 0.0f}, co[2] = {0.0f, 0.0f}, uo[2] = {0.0f, 0.0f};
      for (int sx = 0; sx < T; ++sx) {
        const int half = sx >> 3;
        float mine = 0.0f;
        if (j == (sx & 7)) {
          // token sx's sum with k~ sits in slot 0 (first token) or 2 (second) of its owner lane
          const float A = half ? acc[q][TT == 16 ? 2 : 0] : acc[q][0];
          const float cuh = half ? cu[1] : cu[0];
          mine = round_bf16(__fmul_rn(ts.beta[sx], __fsub_rn(ts.vrow[sx * TV + row], __fadd_rn(A, cuh))));
        }
        const float us = __shfl_sync(0xffffffffu, mine, (lane & ~(LPR - 1)) | (sx & 7));
#pragma unroll
        for (int hh = 0; hh < TT / 8; ++hh) {
          const int tok = j + 8 * hh;
          if (tok < T) {
            if (tok > sx) cu[hh] = __fmaf_rn(cc[tok * KDA_MAX_T + sx], us, cu[hh]);
            if (tok >= sx) co[hh] = __fmaf_rn(ec[tok * KDA_MAX_T + sx], us, co[hh]);
            if (tok == sx) uo[hh] = us;
          }
        }
      }
#pragma unroll
      for (int hh = 0; hh < TT / 8; ++hh) {
        const int tok = j + 8 * hh;
        if (tok < T) {
          urow[tok * TV + row] = uo[hh];
          orow[tok * TV + row] = ok ? __fmul_rn(p.scale, __fadd_rn(acc[q][2 * hh + 1], co[hh])) : 0.0f;
        }
      }
    }
  }

  if (fold && ok) {
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
  __syncthreads();
  for (int i = tid; i < T * TV; i += NT) {
    const int t = i / TV, rr = i - t * TV;
    outp[out_base + (int64_t)t * p.out_t_stride + rr] = float_to_bf16_bits(orow[i]);
    if (ok) uc[(int64_t)(base + t) * KD + v0 + rr] = float_to_bf16_bits(urow[i]);
  }
}

// After the ring kernel, one CTA per batch row: append k~ and G_P at ring
// positions base..base+T-1 for every head, then reset hist_len[n] after a
// fold when restart_hist_on_flush. One warp per head (the CTA has
// APPEND_WARPS warps and loops when H is larger); lane l handles channels
// l + 32 i, and each head's inputs for up to 8 tokens are loaded in one
// batch, so the CTA waits for memory a few times rather than once per token.
// k~ and G come from the same helpers and summation order as token_prologue
// and the ring kernel's channel pass, so the bits match.
constexpr int APPEND_WARPS = 16;

__global__ void __launch_bounds__(32 * APPEND_WARPS)
    kda_ring_append_kernel(const kda_params p, const kda_ring_params rp, const int T) {
  const int b = blockIdx.x;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n = p.state_indices[b];
  if (n < 0 || n >= p.N) return;
  const int hist = rp.hist_len[n];
  if (hist < 0 || hist > rp.W) return;
  const bool fold = hist >= rp.flush_min;
  const int base = fold ? 0 : hist;
  for (int h = warp; h < p.H; h += blockDim.x >> 5) {
    uint16_t* kc = static_cast<uint16_t*>(rp.k_cache) + (int64_t)n * rp.k_slot_stride + (int64_t)h * rp.W * KD;
    float* gc = static_cast<float*>(rp.g_cache) + (int64_t)n * rp.g_slot_stride + (int64_t)h * rp.W * KD;
    const Gate gate(p, h);
    float G_prev[4], dtb[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const int c = lane + 32 * i;
      dtb[i] = gate.dt_bias(p, h, c);
      G_prev[i] = (!fold && hist > 0) ? gc[(int64_t)(hist - 1) * KD + c] : 0.0f;
    }
    for (int t0 = 0; t0 < T; t0 += 8) {
      float kv[8][4], gv[8][4];
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          kv[tt][i] = gv[tt][i] = 0.0f;
          if (t0 + tt < T) {
            kv[tt][i] = load_bf16(p.k, b, t0 + tt, h, lane + 32 * i);
            gv[tt][i] = load_bf16(p.g_raw, b, t0 + tt, h, lane + 32 * i);
          }
        }
      }
#pragma unroll
      for (int tt = 0; tt < 8; ++tt) {
        const int t = t0 + tt;
        if (t >= T) break;
        float sq[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) sq[i] = __fmul_rn(kv[tt][i], kv[tt][i]);
        const float rk = inv_norm(sum_channels(sq[0], sq[1], sq[2], sq[3]));
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int c = lane + 32 * i;
          const float g = gate.g(gv[tt][i], dtb[i]);
          const float G = __fadd_rn(G_prev[i], g);
          kc[(int64_t)(base + t) * KD + c] = float_to_bf16_bits(__fmul_rn(kv[tt][i], rk));
          gc[(int64_t)(base + t) * KD + c] = G;
          G_prev[i] = G;
        }
      }
    }
  }
  if (fold && rp.restart_hist_on_flush) {
    __syncthreads();  // every warp has read hist_len
    if (threadIdx.x == 0) rp.hist_len[n] = 0;
  }
}

template <int TV, bool BULK, int TT>
static cudaError_t launch_ring_one(const kda_params& p, int T, const kda_ring_params& r, cudaStream_t s) {
  constexpr int NW = TV == 128 ? 8 : 4;  // a whole-head tile gets 8 warps
  auto kern = kda_ring_kernel<TV, BULK, TT, NW>;
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, ring_smem_bytes(TV, KDA_MAX_T, 64), smem_set);
  if (e != cudaSuccess) return e;
  const int tiles = KD / TV;
  const long long blocks = (long long)p.B * p.H * tiles;
  kern<<<(unsigned)blocks, 32 * NW, ring_smem_bytes(TV, T, r.W), s>>>(p, r, T, tiles);
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  const int append_warps = p.H < APPEND_WARPS ? p.H : APPEND_WARPS;
  kda_ring_append_kernel<<<(unsigned)p.B, 32 * append_warps, 0, s>>>(p, r, T);
  return cudaGetLastError();
}

template <int TV>
static cudaError_t launch_ring_tv(const kda_params& p, int T, const kda_ring_params& r, bool bulk, cudaStream_t s) {
  if (T <= 8) return bulk ? launch_ring_one<TV, true, 8>(p, T, r, s) : launch_ring_one<TV, false, 8>(p, T, r, s);
  return bulk ? launch_ring_one<TV, true, 16>(p, T, r, s) : launch_ring_one<TV, false, 16>(p, T, r, s);
}

cudaError_t launch_ring(const kda_params& p, int T, const kda_ring_params& r, int tile_v, bool bulk,
                        cudaStream_t s) {
  switch (tile_v) {
    case 16: return launch_ring_tv<16>(p, T, r, bulk, s);
    case 32: return launch_ring_tv<32>(p, T, r, bulk, s);
    case 64: return launch_ring_tv<64>(p, T, r, bulk, s);
    case 128: return launch_ring_tv<128>(p, T, r, bulk, s);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace kda
