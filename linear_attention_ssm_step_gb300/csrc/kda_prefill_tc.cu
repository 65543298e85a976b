// kda_prefill_tc.cu - varlen prefill in chunks of 16 tokens with the chunk
// math on the tensor cores (sm_103a), the reading of include/kda_prefill.h.
//
// Source: "feat(kda): add CuTe DSL recurrent prefill backend" (PR #4605):
// packed sequences by cu_seqlens, the initial state read from an indexed pool
// and the final state written back in place; the backend it describes splits
// each sequence into chunks of 16 tokens (BT16) whose per-chunk math runs as
// dense products, separately from the state-carrying recurrence between
// chunks (Description, and the embedded #4675 commit text).
//
// The arithmetic is the decode step, token after token, on an fp32 state
// rounded to bf16 once at the end (kda_prefill.h). Within a chunk of C tokens
// starting from state S_0 (keys x values), with token decays d_t = exp(g_t),
// P_t = d_0 ... d_t and w_tj = d_{j+1} ... d_t (the ring kernel's WY form):
//   (D_t S_{t-1})^T k_t = S_0^T (P_t k_t) + sum_{j<t}  u_j (w_tj k_j) . k_t
//   S_t^T q_t           = S_0^T (P_t q_t) + sum_{j<=t} u_j (w_tj k_j) . q_t
//   S_C                 = P_{C-1} S_0 + sum_j (w_{C-1,j} k_j) u_j^T
// (k, q the L2-normalised key and query), so per chunk the state enters
// through two products on the tensor cores:
//   X/Y:    [128 value rows x 128 keys] x [128 keys x 2C] - every row's 2C dot
//           products with the decayed keys and queries; S_0 (fp32) as two bf16
//           parts (hi, lo), the vectors as two bf16 parts, all four products
//           accumulated in fp32 (the state and vectors exact to about 2^-17);
//   update: [128 value rows x C] x [C x 128 keys] - sum_j u_j (w_{C-1,j} k_j)
//           with u and the decayed keys as three bf16 parts each, the six
//           products of order <= 2 (exact to about 2^-24), accumulated onto
//           P_{C-1} S_0 in tensor memory;
// and between them only a C-step scalar recurrence per value row over the
// C x C coefficients (cc and ec, block sums of per-channel products):
//   u_t = beta_t (v_t - X_t - sum_{j<t} cc[t][j] u_j),   o_t = Y_t + sum_{j<=t} ec[t][j] u_j.
//
// One CTA of 128 threads, persistent over (sequence, head) items; thread i is
// key channel i in the per-channel work and value row i in the per-row work.
// The fp32 state of the item lives in tensor memory (128 columns) for the
// whole sequence. Per chunk:
//   1. token inputs (loaded during the previous chunk), L2 norms, gates, P_t,
//      the B operand of the X/Y product, the coefficients, P_{C-1};
//   2. row i: S into the two bf16 parts of the A operand, and S <- P_{C-1} S
//      in tensor memory (first chunk: the slot's bf16 state, which arrived by
//      tensor-map loads straight into the first part);
//   3. X/Y product (one thread issues 8 or 16 tcgen05.mma, N = 64); the next
//      chunk's token inputs are fetched meanwhile: where every token view is
//      16-byte aligned (TOK) by four tensor-map copies (16 rows of one head of
//      q, k, g_raw and v each) into the transpose tiles, which the chunk has
//      finished with, else by per-lane loads into registers;
//   4. row i: the recurrence, the outputs of the chunk's tokens;
//   5. U (row i) and the decayed keys W (channel i) as bf16 parts, then the
//      update product accumulates onto S; it runs while the next chunk's
//      step 1 does.
// At the end the state is rounded to bf16 once and row i is stored in the slot.
#include <cuda.h>

#include <algorithm>
#include <cstring>

#include "kda_chunk.cuh"
#include "kda_device.cuh"
#include "kda_launch.h"
#include "kda_prefill.h"
#include "kda_tc.cuh"

namespace kda {

constexpr int PC = KDA_MAX_T;  // tokens per chunk
constexpr int PC_NB = 2 * PC;  // dot products per row and chunk: P_t k_t (even columns), P_t q_t (odd)
constexpr int PC_THREADS = 128;
constexpr uint32_t PC_TMEM_COLS = 256;     // S: columns 0..127; the X/Y sums: 128..191
constexpr uint32_t PC_XY = 128;
constexpr uint32_t PC_PART = 128u * 256u;  // one bf16 part of S as the A operand (128 rows x 128 keys)
constexpr uint32_t PC_UW_PART = 4096u;     // one bf16 part of U or W: 128 rows x 16 tokens, 32-byte swizzle

// Shared-memory carve-up (bytes from a 1024-aligned base).
struct PcLayout {
  uint32_t a, b, red, fcp, rn, plast, beta, xpose, bar, tslot, total;
};

__host__ __device__ inline PcLayout pc_layout() {
  PcLayout L{};
  uint32_t o = 0;
  L.a = o;  // S as two bf16 parts (X/Y product); later in the chunk U and W parts (update product)
  o += 2u * PC_PART;
  L.b = o;  // X/Y B operand: rows 0..31 high parts, 32..63 low parts, 128 keys, 128-byte swizzle
  o += 2u * PC_NB * 256u;
  L.red = o;  // per-warp partial sums: norms, then the coefficients
  o += (1u + PC * PC / 32u) * 512u;
  L.fcp = o;  // coefficient sums, as pairs (M[a][b], M[b][a])
  o += PC * PC * 8u;
  L.rn = o;  // inverse norms
  o += PC_NB * 4u;
  L.plast = o;  // P_{C-1} per key channel
  o += 128u * 4u;
  L.beta = o;
  o += PC * 4u;
  L.xpose = o;  // per-warp transpose tiles of the block sums
  o += 4u * XPOSE_WARP_BYTES;
  L.bar = o;
  o += 32u;
  L.tslot = o;
  o += 16u;
  L.total = o;
  return L;
}

__host__ __device__ inline size_t pc_smem_bytes() { return (size_t)pc_layout().total + 1024; }

// The tensor maps of the token views (TOK): q, k, g_raw, v.
struct TokenMaps {
  CUtensorMap m[4];
};

// The scalar inputs load_tokens also fetches: beta's logits (thread t < T),
// A_log and dt_bias of channel tid (raw gate).
template <int TT>
__device__ __forceinline__ void load_token_scalars(const kda_params& p, int b, int h, int T, TokenRegs<TT>& L) {
  const int tid = threadIdx.x;
  if (tid < T) L.blogit = load_bits(p.beta_logit, b, tid, h, 0);
  if (p.gate_mode == KDA_GATE_RAW) {
    L.alog = p.A_log[h];
    L.dtb = p.dt_bias[(int64_t)h * KD + tid];
  }
}

// Channel tid's values of the staged chunk (zero past T), as load_tokens gives
// them: view j's 16 rows at j * 4096 bytes of the stage.
template <int TT>
__device__ __forceinline__ void tokens_from_stage(const unsigned char* stage, int T, TokenRegs<TT>& L) {
  const uint16_t* st = reinterpret_cast<const uint16_t*>(stage);
  const int tid = threadIdx.x;
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    const bool in = t < T;
    L.qv[t] = in ? st[0 * 2048 + t * KD + tid] : (uint16_t)0;
    L.kv[t] = in ? st[1 * 2048 + t * KD + tid] : (uint16_t)0;
    L.gv[t] = in ? st[2 * 2048 + t * KD + tid] : (uint16_t)0;
    L.vv[t] = in ? st[3 * 2048 + t * KD + tid] : (uint16_t)0;
  }
}

// p: the call's parameters with t_stride = b_stride in q, k, v, g_raw and
// beta_logit, so that token t of a chunk starting at row c0 is (b = c0, t).
template <bool TMA, bool TOK>
__global__ void __launch_bounds__(PC_THREADS, 2)
    kda_prefill_tc_kernel(const __grid_constant__ CUtensorMap smap, const __grid_constant__ TokenMaps tmaps,
                          const kda_params p, const int32_t* __restrict__ cu, const int num_seqs) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int total = num_seqs * p.H;

  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const PcLayout SL = pc_layout();
  unsigned char* sA = sm + SL.a;
  unsigned char* sU = sA;                    // U parts, after the X/Y product has read S
  unsigned char* sW = sA + 3u * PC_UW_PART;  // W parts, likewise
  unsigned char* sB = sm + SL.b;
  float* red = reinterpret_cast<float*>(sm + SL.red);
  float* fcp = reinterpret_cast<float*>(sm + SL.fcp);
  float* rn = reinterpret_cast<float*>(sm + SL.rn);
  float* splast = reinterpret_cast<float*>(sm + SL.plast);
  float* sbeta = reinterpret_cast<float*>(sm + SL.beta);
  float* xtile = reinterpret_cast<float*>(sm + SL.xpose + warp * XPOSE_WARP_BYTES);
  uint64_t* barA = reinterpret_cast<uint64_t*>(sm + SL.bar);  // the slot's state copy
  uint64_t* barD = barA + 1;                                   // X/Y product
  uint64_t* barU = barA + 2;                                   // update product
  uint64_t* barT = barA + 3;                                   // a chunk's token inputs (TOK)
  // ... staged in the transpose tiles, from their first 128-byte boundary
  unsigned char* stage = sm + ((SL.xpose + 127u) & ~127u);
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL.tslot);
  uint16_t* outp = static_cast<uint16_t*>(p.out);

  if (tid == 0) {
    mbar_init(barA, 1);
    mbar_init(barD, 1);
    mbar_init(barU, 1);
    mbar_init(barT, 1);
  }
  if (warp == 0) tmem_alloc(tslot, PC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t row_tmem = tmem + ((uint32_t)(warp * 32) << 16);  // lane tid, column 0
  uint32_t phA = 0, phD = 0, phU = 0;                                // mbarrier phases
  bool pendA = false, pendD = false, pendU = false;                  // a copy or a product is in flight
  uint32_t phT = 0;
  bool pendT = false;  // a chunk's token copies are in flight (TOK)
  bool broken = false;  // a bounded wait gave up: nothing more is issued

  // The first chunk's token inputs of an item, loaded during the previous
  // item's last chunk when that item had one (pre_it: the item they are for).
  TokenRegs<PC> L;
  int pre_it = -1;
  // TOK: the staged chunk has landed (a CTA-uniform answer; false if the
  // bounded wait gave up).
  auto wait_stage = [&]() -> bool {
    const bool w = __syncthreads_and(mbar_wait_bounded(barT, phT)) != 0;
    if (w) {
      phT ^= 1u;
      pendT = false;
    }
    return w;
  };
  // TOK: stage the chunk of 16 rows from activation row b, head h, after any
  // staged chunk still in flight (an item that was skipped) has landed.
  auto stage_next = [&](int b, int h) -> bool {
    if (pendT && !wait_stage()) return false;
    if (tid == 0) {
      mbar_expect_tx(barT, 4u * 4096u);
#pragma unroll
      for (int j = 0; j < 4; ++j) tma_load_3d(stage + j * 4096, &tmaps.m[j], 0, h, b, barT);
    }
    pendT = true;
    return true;
  };
  for (int it = blockIdx.x; it < total; it += gridDim.x) {
    const int seq = it / p.H, h = it - seq * p.H;
    const int t0 = cu[seq], t1 = cu[seq + 1];
    const int n = p.state_indices[seq];
    if (t0 < 0 || t1 < t0 || t1 > p.B) {
      if (tid == 0 && h == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_SEQLENS);
      continue;
    }
    const int64_t ob = (int64_t)h * p.out_h_stride + tid;  // output element of row tid, + token row * out_b_stride
    if (n < 0 || n >= p.N || broken) {  // inactive (or skipped after a wait gave up): zero outputs
      for (int t = t0; t < t1; ++t) outp[(int64_t)t * p.out_b_stride + ob] = 0;
      continue;
    }
    if (t0 == t1) continue;
    uint16_t* gstate = static_cast<uint16_t*>(p.state) + (int64_t)n * p.state_slot_stride + (int64_t)h * KD * KD;

    // The slot's bf16 state into the first part of the A operand (exact as stored).
    if constexpr (TMA) {
      if (tid == 0) {
        mbar_expect_tx(barA, KD * KD * 2);
        tma_load_3d(sA, &smap, 0, h * KD, n, barA);
        tma_load_3d(sA + KD * 128, &smap, 64, h * KD, n, barA);
      }
      pendA = true;
    } else {
      for (int r = 0; r < KD; ++r)
        *reinterpret_cast<uint16_t*>(sA + sw128_offset(KD, r, tid)) = gstate[(int64_t)r * KD + tid];
    }

    bool first = true, ok = true;
    if (pre_it != it) {
      zero_tokens(L);
      if constexpr (TOK) {
        fence_proxy_async_smem();  // the last item's generic uses of the tiles come before the copies
        __syncthreads();
        ok = stage_next(t0, h);
        load_token_scalars(p, t0, h, min(PC, t1 - t0), L);
      } else {
        load_tokens(p, t0, h, min(PC, t1 - t0), L);
      }
    }
    pre_it = -1;
    for (int c0 = t0; c0 < t1 && ok; c0 += PC) {
      const int Tc = min(PC, t1 - c0);
      if constexpr (TOK) {  // the chunk's staged tokens into registers; the tiles are written next
        if (!wait_stage()) {
          ok = false;
          break;
        }
        tokens_from_stage(stage, Tc, L);
        __syncthreads();
      }

      // 1. L2 norms: block sums of q_t^2 (value t) and k_t^2 (value PC + t).
#pragma unroll
      for (int t = 0; t < PC; ++t) {
        const float q = bf16_bits_to_float(L.qv[t]), k = bf16_bits_to_float(L.kv[t]);
        tile_put(xtile, lane, t, __fmul_rn(q, q));
        tile_put(xtile, lane, PC + t, __fmul_rn(k, k));
      }
      __syncwarp();
      {
        const float s = tile_row_sum(xtile, lane);
        __syncwarp();
        red[warp * 32 + lane] = s;
      }
      __syncthreads();
      if (tid < PC_NB) rn[tid] = inv_norm(block_sum(red, 0, tid));
      __syncthreads();

      // Per channel tid: the normalised vectors, the gate (tokens past the
      // chunk's end: decay 1, beta 0, zero vectors), P_t and the B operand.
      const FastGate gate(p, L.alog);
      if (tid < PC) sbeta[tid] = tid < Tc ? gate.beta(bf16_bits_to_float(L.blogit)) : 0.0f;
      float qh[PC], kh[PC], dd[PC];
#pragma unroll
      for (int t = 0; t < PC; ++t) {
        qh[t] = __fmul_rn(bf16_bits_to_float(L.qv[t]), rn[t]);
        kh[t] = __fmul_rn(bf16_bits_to_float(L.kv[t]), rn[PC + t]);
        dd[t] = t < Tc ? __expf(gate.g(bf16_bits_to_float(L.gv[t]), L.dtb)) : 1.0f;
      }
      {
        float P = 1.0f;
        const Sw128Col col = sw128_col(2 * PC_NB, tid);
#pragma unroll
        for (int t = 0; t < PC; ++t) {
          P = __fmul_rn(P, dd[t]);
          float xk, xq;
          upk2(mul2(pk2(P, P), pk2(kh[t], qh[t])), xk, xq);
          store_split_at(sB, sB + PC_NB * 128, sw128_at(col, 2 * t), xk);
          store_split_at(sB, sB + PC_NB * 128, sw128_at(col, 2 * t + 1), xq);
        }
        splast[tid] = P;
      }

      // Coefficients M[a][b] (flat a PC + b): a > b holds cc[a][b] = (w_ab k_b) . k_a,
      // a <= b holds ec[b][a] = (w_ba k_a) . q_b, w a running product of the decays.
#pragma unroll
      for (int a0 = 0; a0 < PC; a0 += 32 / PC) {
        float vals[32];
#pragma unroll
        for (int r = 0; r < 32 / PC; ++r) {
          const int a = a0 + r;
#pragma unroll
          for (int b2 = 0; b2 < PC; ++b2) vals[r * PC + b2] = 0.0f;
          float w = 1.0f;  // w_{a,b} for b = a-1, a-2, ...: d_a d_{a-1} ... d_{b+1}
#pragma unroll
          for (int b2 = PC - 1; b2 >= 0; --b2) {
            if (b2 < a) {
              w = __fmul_rn(w, dd[b2 + 1]);
              vals[r * PC + b2] = __fmul_rn(__fmul_rn(w, kh[b2]), kh[a]);
            }
          }
          float w2 = 1.0f;  // w_{b,a} for b = a, a+1, ...: d_{a+1} ... d_b
#pragma unroll
          for (int b2 = 0; b2 < PC; ++b2) {
            if (b2 >= a) {
              if (b2 > a) w2 = __fmul_rn(w2, dd[b2]);
              vals[r * PC + b2] = __fmul_rn(__fmul_rn(w2, kh[a]), qh[b2]);
            }
          }
        }
        red[((1 + a0 * PC / 32) * 4 + warp) * 32 + lane] = warp_sum32(vals, xtile, lane);
      }
      // The update's decayed keys of channel tid: W_j = (d_{j+1} ... d_{PC-1}) k_j.
      float Wk[PC];
      {
        float wl = 1.0f;
#pragma unroll
        for (int j = PC - 1; j >= 0; --j) {
          Wk[j] = __fmul_rn(wl, kh[j]);
          wl = __fmul_rn(wl, dd[j]);
        }
      }
      __syncthreads();  // partial sums, the B operand, P_{C-1}, beta
      for (int i = tid; i < PC * PC; i += PC_THREADS) {
        const float v = block_sum(red, 1 + (i >> 5), i & 31);
        fcp[2 * i] = v;
        fcp[2 * ((i % PC) * PC + i / PC) + 1] = v;
      }

      // 2. The previous update has finished with S and the A region; on the
      // first chunk the slot's state has arrived.
      {
        bool w_ok = true;
        if (pendU) w_ok = mbar_wait_bounded(barU, phU);
        if (TMA && first && w_ok) w_ok = mbar_wait_bounded(barA, phA);
        ok = __syncthreads_and(w_ok) != 0;
      }
      if (!ok) break;
      if (pendU) {
        phU ^= 1u;
        pendU = false;
      }
      if (TMA && first) {
        phA ^= 1u;
        pendA = false;
      }
      tc_fence_after();
      // Row tid: S into the bf16 parts of the A operand, S <- P_{C-1} S in tensor memory.
#pragma unroll 1
      for (int cb = 0; cb < 4; ++cb) {
        float s[32];
        if (first) {  // the slot's bf16 row, from the A operand
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            const uint4 raw = *reinterpret_cast<const uint4*>(sA + sw128_offset(KD, tid, cb * 32 + 8 * c));
            unpack_bf16x2(raw.x, s[8 * c], s[8 * c + 1]);
            unpack_bf16x2(raw.y, s[8 * c + 2], s[8 * c + 3]);
            unpack_bf16x2(raw.z, s[8 * c + 4], s[8 * c + 5]);
            unpack_bf16x2(raw.w, s[8 * c + 6], s[8 * c + 7]);
          }
        } else {
          tmem_ld32(row_tmem + cb * 32, s);
#pragma unroll
          for (int c = 0; c < 4; ++c) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
              const float s0 = s[8 * c + 2 * q], s1 = s[8 * c + 2 * q + 1];
              hw[q] = pack_bf16x2(s0, s1);
              float h0, h1;
              unpack_bf16x2(hw[q], h0, h1);
              lw[q] = pack_bf16x2(__fsub_rn(s0, h0), __fsub_rn(s1, h1));
            }
            const uint32_t off = sw128_offset(KD, tid, cb * 32 + 8 * c);
            *reinterpret_cast<uint4*>(sA + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(sA + PC_PART + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
#pragma unroll
        for (int c = 0; c < 8; ++c) {
          const float4 pl = *reinterpret_cast<const float4*>(splast + cb * 32 + 4 * c);
          f32x2 a = mul2(pk2(pl.x, pl.y), pk2(s[4 * c], s[4 * c + 1]));
          f32x2 b = mul2(pk2(pl.z, pl.w), pk2(s[4 * c + 2], s[4 * c + 3]));
          upk2(a, s[4 * c], s[4 * c + 1]);
          upk2(b, s[4 * c + 2], s[4 * c + 3]);
        }
        tmem_st32(row_tmem + cb * 32, s);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // the A operand is read by the tensor core
      tc_fence_before();
      __syncthreads();

      // 3. The X/Y product: D[row][col] = sum_k S[row][k] B[col][k], K in 8 steps of
      // 16, per part of S; columns 32.. hold the low parts' share.
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, 2 * PC_NB);
        const uint32_t a0 = smem_addr(sA), b0 = smem_addr(sB);
        const int parts = first ? 1 : 2;
        for (int part = 0; part < parts; ++part)
#pragma unroll
          for (int kk = 0; kk < 8; ++kk)
            tc_mma_bf16(tmem + PC_XY, sw128_desc(a0 + part * PC_PART + (kk >> 2) * (KD * 128) + (kk & 3) * 32),
                        sw128_desc(b0 + (kk >> 2) * (2 * PC_NB * 128) + (kk & 3) * 32), idesc,
                        (part > 0 || kk > 0) ? 1u : 0u);
        tc_commit(barD);
      }
      pendD = true;
      uint16_t vcur[PC];
#pragma unroll
      for (int t = 0; t < PC; ++t) vcur[t] = L.vv[t];
      // The next chunk's token inputs fly while this chunk finishes (TOK: the
      // tiles' last reads, the coefficient sums, came before the product's
      // barrier and its proxy fence).
      bool s_ok = true;
      if (c0 + PC < t1) {
        zero_tokens(L);
        if constexpr (TOK) {
          s_ok = stage_next(c0 + PC, h);
          load_token_scalars(p, c0 + PC, h, min(PC, t1 - c0 - PC), L);
        } else {
          load_tokens(p, c0 + PC, h, min(PC, t1 - c0 - PC), L);
        }
      } else if (it + (int)gridDim.x < total) {  // the last chunk: the next item's first chunk
        const int nit = it + gridDim.x;
        const int nseq = nit / p.H, nh = nit - nseq * p.H;
        const int n0 = cu[nseq], n1 = cu[nseq + 1];
        if (n0 >= 0 && n1 > n0 && n1 <= p.B) {  // a sequence with tokens (loaded even if inactive: unused then)
          zero_tokens(L);
          if constexpr (TOK) {
            s_ok = stage_next(n0, nh);
            load_token_scalars(p, n0, nh, min(PC, n1 - n0), L);
          } else {
            load_tokens(p, n0, nh, min(PC, n1 - n0), L);
          }
          pre_it = nit;
        }
      }
      ok = __syncthreads_and(mbar_wait_bounded(barD, phD) && s_ok) != 0;
      if (!ok) break;
      phD ^= 1u;
      pendD = false;
      tc_fence_after();
      f32x2 X[PC];  // (S_0^T (P_t k_t), S_0^T (P_t q_t)) of row tid
#pragma unroll
      for (int c = 0; c < PC_NB; c += 16) {
        float xh[16], xl[16];
        tmem_ld16(row_tmem + PC_XY + c, xh);
        tmem_ld16(row_tmem + PC_XY + PC_NB + c, xl);
#pragma unroll
        for (int i = 0; i < 8; ++i) X[c / 2 + i] = add2(pk2(xh[2 * i], xh[2 * i + 1]), pk2(xl[2 * i], xl[2 * i + 1]));
      }

      // 4. Row tid: the recurrence over the chunk's tokens, and their outputs.
      float uval[PC];
      {
        f32x2 uu[PC];
#pragma unroll
        for (int t = 0; t < PC; ++t) {
          f32x2 ce[PC];  // (cc[t][s], ec[t][s]): cc for s < t, ec for s <= t (only those are loaded)
#pragma unroll
          for (int s2 = 0; s2 <= t / 2; ++s2) {
            const float4 c = reinterpret_cast<const float4*>(fcp + 2 * t * PC)[s2];
            ce[2 * s2] = pk2(c.x, c.y);
            ce[2 * s2 + 1] = pk2(c.z, c.w);
          }
          f32x2 acc_e = pk2(0.0f, 0.0f), acc_o = pk2(0.0f, 0.0f);  // two chains: half the latency
#pragma unroll
          for (int s2 = 0; s2 < t; ++s2) {
            if (s2 & 1)
              acc_o = fma2(ce[s2], uu[s2], acc_o);
            else
              acc_e = fma2(ce[s2], uu[s2], acc_e);
          }
          float acc, acco, xk, xq, ctt, ect;
          upk2(add2(acc_e, acc_o), acc, acco);
          upk2(X[t], xk, xq);
          upk2(ce[t], ctt, ect);
          (void)ctt;
          const float ut = __fmul_rn(sbeta[t], __fsub_rn(bf16_bits_to_float(vcur[t]), __fadd_rn(xk, acc)));
          uu[t] = pk2(ut, ut);
          uval[t] = ut;
          acco = __fmaf_rn(ect, ut, acco);
          const float o = __fmul_rn(p.scale, __fadd_rn(xq, acco));
          if (t < Tc) outp[(int64_t)(c0 + t) * p.out_b_stride + ob] = float_to_bf16_bits(o);
        }
      }

      // 5. U (row tid) and W (channel tid) as three bf16 parts; the update product
      // accumulates sum_j u_j W_j onto P_{C-1} S_0 in tensor memory.
      store_row_split3(sU, PC_UW_PART, tid, uval);
      store_row_split3(sW, PC_UW_PART, tid, Wk);
      fence_proxy_async_smem();
      tc_fence_before();
      __syncthreads();
      if (tid == 0) {
        tc_fence_after();
        constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
        const uint32_t u0 = smem_addr(sU), w0 = smem_addr(sW);
        // the products of order <= 2 of the parts: (0, 0) (1, 0) (2, 0) (0, 1) (1, 1) (0, 2)
#pragma unroll
        for (int q = 0; q < 6; ++q) {
          const uint32_t pa = q < 3 ? (uint32_t)q : (q == 4 ? 1u : 0u);
          const uint32_t pb = q < 3 ? 0u : (q == 5 ? 2u : 1u);
          tc_mma_bf16(tmem, sw32_desc(u0 + pa * PC_UW_PART), sw32_desc(w0 + pb * PC_UW_PART), idesc, 1u);
        }
        tc_commit(barU);
      }
      pendU = true;
      first = false;
    }

    if (ok) {  // the final state, rounded to bf16 once; row tid into the slot
      ok = __syncthreads_and(mbar_wait_bounded(barU, phU)) != 0;
      if (ok) {
        phU ^= 1u;
        pendU = false;
        tc_fence_after();
        uint16_t* grow = gstate + (int64_t)tid * KD;
#pragma unroll 1
        for (int cb = 0; cb < 4; ++cb) {
          float s[32];
          tmem_ld32(row_tmem + cb * 32, s);
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) w[q] = pack_bf16x2(s[2 * q], s[2 * q + 1]);
          if constexpr (TMA) {  // 16-byte aligned pool
            uint4* dst = reinterpret_cast<uint4*>(grow + cb * 32);
#pragma unroll
            for (int c = 0; c < 4; ++c) dst[c] = make_uint4(w[4 * c], w[4 * c + 1], w[4 * c + 2], w[4 * c + 3]);
          } else {
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              grow[cb * 32 + 2 * q] = (uint16_t)(w[q] & 0xffffu);
              grow[cb * 32 + 2 * q + 1] = (uint16_t)(w[q] >> 16);
            }
          }
        }
      }
    }
    if (!ok) {  // a bounded wait gave up: the sequence is skipped, and every later one
      broken = true;
      if (tid == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      for (int t = t0; t < t1; ++t) outp[(int64_t)t * p.out_b_stride + ob] = 0;
    }
    tc_fence_before();
    __syncthreads();  // this item's tensor-memory and shared-memory use is done
    tc_fence_after();
  }

  // Anything still in flight after a wait that gave up gets one more bounded
  // wait before the tensor memory is released and the CTA leaves.
  if (tid == 0) {
    if (pendA) mbar_wait_bounded(barA, phA);
    if (pendD) mbar_wait_bounded(barD, phD);
    if (pendU) mbar_wait_bounded(barU, phU);
    if (pendT) mbar_wait_bounded(barT, phT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, PC_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

template <bool TMA, bool TOK>
static cudaError_t launch_pftc(const CUtensorMap& map, const TokenMaps& tm, const kda_params& p, const int32_t* cu,
                               int num_seqs, cudaStream_t s) {
  auto kern = kda_prefill_tc_kernel<TMA, TOK>;
  const size_t smem = pc_smem_bytes();
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> carveout_set{false};  // all of L1 as shared memory: two CTAs per SM
  if (!carveout_set.load(std::memory_order_acquire)) {
    if ((e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout,
                                  (int)cudaSharedmemCarveoutMaxShared)) != cudaSuccess)
      return e;
    carveout_set.store(true, std::memory_order_release);
  }
  // Persistent grid: as many CTAs as fit at once (shared memory, registers and
  // the SM's 512 tensor-memory columns), at most one per (sequence, head).
  int dev = 0, sms = 0, smem_sm = 0, reserved = 0, regs_sm = 0, blocks_sm = 0;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&smem_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&regs_sm, cudaDevAttrMaxRegistersPerMultiprocessor, dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&blocks_sm, cudaDevAttrMaxBlocksPerMultiprocessor, dev)) != cudaSuccess) return e;
  cudaFuncAttributes fa;
  if ((e = cudaFuncGetAttributes(&fa, kern)) != cudaSuccess) return e;
  const int warp_regs = (fa.numRegs * 32 + 255) / 256 * 256;
  int per_sm = smem_sm / (int)(smem + reserved);
  per_sm = std::min(per_sm, regs_sm / (warp_regs * (PC_THREADS / 32)));
  per_sm = std::min(per_sm, 512 / (int)PC_TMEM_COLS);
  per_sm = std::min(per_sm, blocks_sm);
  if (per_sm < 1) return cudaErrorInvalidConfiguration;
  const long long items = (long long)num_seqs * p.H;
  const long long grid = std::min(items, (long long)sms * per_sm);
  kda_params q = p;  // token t of a chunk is activation row c0 + t
  q.q.t_stride = q.q.b_stride;
  q.k.t_stride = q.k.b_stride;
  q.v.t_stride = q.v.b_stride;
  q.g_raw.t_stride = q.g_raw.b_stride;
  q.beta_logit.t_stride = q.beta_logit.b_stride;
  kern<<<(unsigned)grid, PC_THREADS, smem, s>>>(map, tm, q, cu, num_seqs);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const kda_params& p, const int32_t* cu, int num_seqs, bool bulk, cudaStream_t s) {
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (bulk) {
    const cudaError_t e = state_tensor_map(p, &map);
    if (e != cudaSuccess) return e;
    TokenMaps tm;
    memset(&tm, 0, sizeof(tm));
    // The token views by tensor maps ({128, H, rows} in 16-row boxes) where
    // every row is 16-byte aligned and the maps can be formed, else plain loads.
    bool tok = prefill_rows_aligned16(p);
    const kda_view* vw[4] = {&p.q, &p.k, &p.g_raw, &p.v};
    for (int j = 0; j < 4 && tok; ++j) tok = token_tensor_map(*vw[j], p.B, p.H, &tm.m[j]) == cudaSuccess;
    if (tok) return launch_pftc<true, true>(map, tm, p, cu, num_seqs, s);
    return launch_pftc<true, false>(map, tm, p, cu, num_seqs, s);
  }
  TokenMaps tm;
  memset(&tm, 0, sizeof(tm));
  return launch_pftc<false, false>(map, tm, p, cu, num_seqs, s);
}

}  // namespace kda
