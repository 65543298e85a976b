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
//      chunk's token loads are issued meanwhile;
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
constexpr int PC_WG = 2;       // warp groups: each takes half of a chunk's tokens, state columns, coefficients
constexpr int PC_TW = PC / PC_WG;  // tokens per warp group
constexpr int PC_THREADS = 128 * PC_WG;
constexpr uint32_t PC_TMEM_COLS = 256;     // S: columns 0..127; the X/Y sums: 128..191
constexpr uint32_t PC_XY = 128;
constexpr uint32_t PC_PART = 128u * 256u;  // one bf16 part of S as the A operand (128 rows x 128 keys)
constexpr uint32_t PC_UW_PART = 4096u;     // one bf16 part of U or W: 128 rows x 16 tokens, 32-byte swizzle

// Shared-memory carve-up (bytes from a 1024-aligned base).
struct PcLayout {
  uint32_t a, b, red, fcp, rn, plast, beta, xkh, xqh, xdd, xv, su, xpose, bar, tslot, total;
};

__host__ __device__ inline PcLayout pc_layout() {
  PcLayout L{};
  uint32_t o = 0;
  L.a = o;  // S as two bf16 parts (X/Y product); later in the chunk U and W parts (update product)
  o += 2u * PC_PART;
  L.b = o;  // X/Y B operand: rows 0..31 high parts, 32..63 low parts, 128 keys, 128-byte swizzle
  o += 2u * PC_NB * 256u;
  L.red = o;  // per-warp partial sums: each warp group's norms, then the coefficients
  o += (PC_WG + PC * PC / 32u) * 512u;
  L.fcp = o;  // coefficient sums, as pairs (M[a][b], M[b][a])
  o += PC * PC * 8u;
  L.rn = o;  // inverse norms: q of token t at t, k at PC + t
  o += PC_NB * 4u;
  L.plast = o;  // P_{C-1} per key channel
  o += 128u * 4u;
  L.beta = o;
  o += PC * 4u;
  L.xkh = o;  // the chunk's k_hat, q_hat, decay and v, token-major [PC][128]: each warp group
  o += PC * 512u;  // writes its tokens, both read all
  L.xqh = o;
  o += PC * 512u;
  L.xdd = o;
  o += PC * 512u;
  L.xv = o;
  o += PC * 512u;
  L.su = o;  // the rows' u, token-major [PC][128], from the u chain to the outputs
  o += PC * 512u;
  L.xpose = o;  // per-warp transpose tiles of the block sums
  o += (PC_THREADS / 32u) * XPOSE_WARP_BYTES;
  L.bar = o;
  o += 32u;
  L.tslot = o;
  o += 16u;
  L.total = o;
  return L;
}

__host__ __device__ inline size_t pc_smem_bytes() { return (size_t)pc_layout().total + 1024; }

// p: the call's parameters with t_stride = b_stride in q, k, v, g_raw and
// beta_logit, so that token t of a chunk starting at row c0 is (b = c0, t).
//
// Thread tid is warp group wg = tid / 128 and index c = tid % 128: key channel
// c in the per-channel work, value row c in the per-row work (warps w and
// w + 4 read the same tensor-memory lanes). Warp group wg takes tokens
// 8 wg .. 8 wg + 7 of a chunk (inputs, norms, gates, B-operand rows), rows
// 8 wg .. of the coefficient matrix, columns 64 wg .. 64 wg + 63 of the state
// (its split and decay), entries 8 wg .. of the update's decayed keys; in the
// recurrence warp group 0 runs the u chain and warp group 1 the outputs.
template <bool TMA>
__global__ void __launch_bounds__(PC_THREADS, 1)
    kda_prefill_tc_kernel(const __grid_constant__ CUtensorMap smap, const kda_params p, const int32_t* __restrict__ cu,
                          const int num_seqs) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int wg = tid >> 7, c = tid & 127, wq = warp & 3;
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
  float* xkh = reinterpret_cast<float*>(sm + SL.xkh);
  float* xqh = reinterpret_cast<float*>(sm + SL.xqh);
  float* xdd = reinterpret_cast<float*>(sm + SL.xdd);
  float* xv = reinterpret_cast<float*>(sm + SL.xv);
  float* su = reinterpret_cast<float*>(sm + SL.su);
  float* xtile = reinterpret_cast<float*>(sm + SL.xpose + warp * XPOSE_WARP_BYTES);
  uint64_t* barA = reinterpret_cast<uint64_t*>(sm + SL.bar);  // the slot's state copy
  uint64_t* barD = barA + 1;                                   // X/Y product
  uint64_t* barU = barA + 2;                                   // update product
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL.tslot);
  uint16_t* outp = static_cast<uint16_t*>(p.out);

  if (tid == 0) {
    mbar_init(barA, 1);
    mbar_init(barD, 1);
    mbar_init(barU, 1);
  }
  if (warp == 0) tmem_alloc(tslot, PC_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t row_tmem = tmem + ((uint32_t)(wq * 32) << 16);  // lane c, column 0
  uint32_t phA = 0, phD = 0, phU = 0;                              // mbarrier phases
  bool pendA = false, pendD = false, pendU = false;                // a copy or a product is in flight
  bool broken = false;  // a bounded wait gave up: nothing more is issued

  for (int it = blockIdx.x; it < total; it += gridDim.x) {
    const int seq = it / p.H, h = it - seq * p.H;
    const int t0 = cu[seq], t1 = cu[seq + 1];
    const int n = p.state_indices[seq];
    if (t0 < 0 || t1 < t0 || t1 > p.B) {
      if (tid == 0 && h == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_SEQLENS);
      continue;
    }
    const int64_t ob = (int64_t)h * p.out_h_stride + c;  // output element of row c, + token row * out_b_stride
    if (n < 0 || n >= p.N || broken) {  // inactive (or skipped after a wait gave up): zero outputs
      for (int t = t0 + wg; t < t1; t += PC_WG) outp[(int64_t)t * p.out_b_stride + ob] = 0;
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
      for (int r = wg; r < KD; r += PC_WG)
        *reinterpret_cast<uint16_t*>(sA + sw128_offset(KD, r, c)) = gstate[(int64_t)r * KD + c];
    }

    // This warp group's tokens of the first chunk.
    TokenRegs<PC_TW> L;
    zero_tokens(L);
    load_tokens_at(p, t0 + wg * PC_TW, h, min(PC_TW, t1 - t0 - wg * PC_TW), L, c);
    bool first = true, ok = true;
    for (int c0 = t0; c0 < t1; c0 += PC) {
      const int Tc = min(PC, t1 - c0);
      const int tb = wg * PC_TW;  // this warp group's first token

      // 1. L2 norms of this warp group's tokens: block sums of q^2 (value i) and
      // k^2 (value PC_TW + i) over the group's four warps.
#pragma unroll
      for (int i = 0; i < PC_TW; ++i) {
        const float q = bf16_bits_to_float(L.qv[i]), k = bf16_bits_to_float(L.kv[i]);
        tile_put(xtile, lane, i, __fmul_rn(q, q));
        tile_put(xtile, lane, PC_TW + i, __fmul_rn(k, k));
      }
      __syncwarp();
      {
        const float s = tile_row_sum(xtile, lane & (2 * PC_TW - 1));
        __syncwarp();
        red[(wg * 4 + wq) * 32 + lane] = s;
      }
      __syncthreads();
      if (c < 2 * PC_TW) {
        const float inv = inv_norm(block_sum(red, wg, c));
        rn[c < PC_TW ? tb + c : PC + tb + c - PC_TW] = inv;
      }
      __syncthreads();

      // 2. Per channel c, this group's tokens: the normalised vectors, the gate
      // (tokens past the chunk's end: decay 1, beta 0, zero vectors), shared
      // through shared memory with the other group; v of row c likewise.
      {
        const FastGate gate(p, L.alog);
        if (c < PC_TW) sbeta[tb + c] = tb + c < Tc ? gate.beta(bf16_bits_to_float(L.blogit)) : 0.0f;
#pragma unroll
        for (int i = 0; i < PC_TW; ++i) {
          const int t = tb + i;
          xqh[t * KD + c] = __fmul_rn(bf16_bits_to_float(L.qv[i]), rn[t]);
          xkh[t * KD + c] = __fmul_rn(bf16_bits_to_float(L.kv[i]), rn[PC + t]);
          xdd[t * KD + c] = t < Tc ? __expf(gate.g(bf16_bits_to_float(L.gv[i]), L.dtb)) : 1.0f;
          xv[t * KD + c] = bf16_bits_to_float(L.vv[i]);
        }
      }
      __syncthreads();
      float qh[PC], kh[PC], dd[PC];
#pragma unroll
      for (int t = 0; t < PC; ++t) {
        qh[t] = xqh[t * KD + c];
        kh[t] = xkh[t * KD + c];
        dd[t] = xdd[t * KD + c];
      }
      {  // P_t, and this group's rows of the B operand
        float P = 1.0f;
#pragma unroll
        for (int t = 0; t < PC; ++t) {
          P = __fmul_rn(P, dd[t]);
          if (t >= tb && t < tb + PC_TW) {
            float xk, xq;
            upk2(mul2(pk2(P, P), pk2(kh[t], qh[t])), xk, xq);
            store_split<2 * PC_NB>(sB, sB + PC_NB * 128, 2 * t, c, xk);
            store_split<2 * PC_NB>(sB, sB + PC_NB * 128, 2 * t + 1, c, xq);
          }
        }
        if (wg == 0) splast[c] = P;
      }

      // Coefficients M[a][b] (flat a PC + b) for this group's rows a: a > b holds
      // cc[a][b] = (w_ab k_b) . k_a, a <= b holds ec[b][a] = (w_ba k_a) . q_b, w a
      // running product of the decays.
#pragma unroll
      for (int a0 = 0; a0 < PC; a0 += 32 / PC) {
        if (a0 / PC_TW != wg) continue;  // rows of the other warp group (a uniform branch; a0 stays static)
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
        red[((PC_WG + a0 * PC / 32) * 4 + wq) * 32 + lane] = warp_sum32(vals, xtile, lane);
      }
      // The update's decayed keys of channel c for this group's entries:
      // W_j = (d_{j+1} ... d_{PC-1}) k_j.
      float Wk[PC_TW];
      {
        float W16[PC];
        float wl = 1.0f;
#pragma unroll
        for (int j = PC - 1; j >= 0; --j) {
          W16[j] = __fmul_rn(wl, kh[j]);
          wl = __fmul_rn(wl, dd[j]);
        }
#pragma unroll
        for (int j = 0; j < PC_TW; ++j) Wk[j] = wg == 0 ? W16[j] : W16[PC_TW + j];
      }
      __syncthreads();  // partial sums, the B operand, P_{C-1}, beta
      {
        const int i = tid;  // PC * PC = 256 coefficients, one per thread
        const float v = block_sum(red, PC_WG + (i >> 5), i & 31);
        fcp[2 * i] = v;
        fcp[2 * ((i % PC) * PC + i / PC) + 1] = v;
      }

      // 3. The previous update has finished with S and the A region; on the
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
      // Row c, this group's 64 columns: S into the bf16 parts of the A operand,
      // S <- P_{C-1} S in tensor memory.
#pragma unroll 1
      for (int cb = 2 * wg; cb < 2 * wg + 2; ++cb) {
        float s[32];
        if (first) {  // the slot's bf16 row, from the A operand
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const uint4 raw = *reinterpret_cast<const uint4*>(sA + sw128_offset(KD, c, cb * 32 + 8 * q));
            unpack_bf16x2(raw.x, s[8 * q], s[8 * q + 1]);
            unpack_bf16x2(raw.y, s[8 * q + 2], s[8 * q + 3]);
            unpack_bf16x2(raw.z, s[8 * q + 4], s[8 * q + 5]);
            unpack_bf16x2(raw.w, s[8 * q + 6], s[8 * q + 7]);
          }
        } else {
          tmem_ld32(row_tmem + cb * 32, s);
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            uint32_t hw[4], lw[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              const float s0 = s[8 * q + 2 * e], s1 = s[8 * q + 2 * e + 1];
              hw[e] = pack_bf16x2(s0, s1);
              float h0, h1;
              unpack_bf16x2(hw[e], h0, h1);
              lw[e] = pack_bf16x2(__fsub_rn(s0, h0), __fsub_rn(s1, h1));
            }
            const uint32_t off = sw128_offset(KD, c, cb * 32 + 8 * q);
            *reinterpret_cast<uint4*>(sA + off) = make_uint4(hw[0], hw[1], hw[2], hw[3]);
            *reinterpret_cast<uint4*>(sA + PC_PART + off) = make_uint4(lw[0], lw[1], lw[2], lw[3]);
          }
        }
#pragma unroll
        for (int q = 0; q < 8; ++q) {
          const float4 pl = *reinterpret_cast<const float4*>(splast + cb * 32 + 4 * q);
          f32x2 x0 = mul2(pk2(pl.x, pl.y), pk2(s[4 * q], s[4 * q + 1]));
          f32x2 x1 = mul2(pk2(pl.z, pl.w), pk2(s[4 * q + 2], s[4 * q + 3]));
          upk2(x0, s[4 * q], s[4 * q + 1]);
          upk2(x1, s[4 * q + 2], s[4 * q + 3]);
        }
        tmem_st32(row_tmem + cb * 32, s);
      }
      tmem_st_wait();
      fence_proxy_async_smem();  // the A operand is read by the tensor core
      tc_fence_before();
      __syncthreads();

      // 4. The X/Y product: D[row][col] = sum_k S[row][k] B[col][k], K in 8 steps of
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
      if (c0 + PC < t1) {  // the next chunk's token inputs fly while this chunk finishes
        zero_tokens(L);
        const int nb = c0 + PC + tb;
        load_tokens_at(p, nb, h, min(PC_TW, t1 - nb), L, c);
      }
      ok = __syncthreads_and(mbar_wait_bounded(barD, phD)) != 0;
      if (!ok) break;
      phD ^= 1u;
      pendD = false;
      tc_fence_after();
      f32x2 X[PC];  // (S_0^T (P_t k_t), S_0^T (P_t q_t)) of row c
#pragma unroll
      for (int q = 0; q < PC_NB; q += 16) {
        float xh[16], xl[16];
        tmem_ld16(row_tmem + PC_XY + q, xh);
        tmem_ld16(row_tmem + PC_XY + PC_NB + q, xl);
#pragma unroll
        for (int i = 0; i < 8; ++i) X[q / 2 + i] = add2(pk2(xh[2 * i], xh[2 * i + 1]), pk2(xl[2 * i], xl[2 * i + 1]));
      }

      // 5. Row c: warp group 0 runs the u chain and shares u; warp group 1 then
      // forms the outputs. U (group 0) and this group's W entries as bf16 parts.
      if (wg == 0) {
        float uval[PC];
#pragma unroll
        for (int t = 0; t < PC; ++t) {
          float acc_e = 0.0f, acc_o = 0.0f;
#pragma unroll
          for (int s2 = 0; s2 < t; ++s2) {
            const float cc = fcp[2 * (t * PC + s2)];
            if (s2 & 1)
              acc_o = __fmaf_rn(cc, uval[s2], acc_o);
            else
              acc_e = __fmaf_rn(cc, uval[s2], acc_e);
          }
          float xk, xq;
          upk2(X[t], xk, xq);
          (void)xq;
          uval[t] = __fmul_rn(sbeta[t], __fsub_rn(xv[t * KD + c], __fadd_rn(xk, __fadd_rn(acc_e, acc_o))));
          su[t * KD + c] = uval[t];
        }
        store_row_split3(sU, PC_UW_PART, c, uval);
      }
      __syncthreads();  // u of every row
      if (wg == 1) {
        float uval[PC];
#pragma unroll
        for (int t = 0; t < PC; ++t) uval[t] = su[t * KD + c];
#pragma unroll
        for (int t = 0; t < PC; ++t) {
          if (t < Tc) {
            float xk, xq;
            upk2(X[t], xk, xq);
            (void)xk;
            float acc_e = 0.0f, acc_o = 0.0f;
#pragma unroll
            for (int s2 = 0; s2 <= t; ++s2) {
              const float ec = fcp[2 * (t * PC + s2) + 1];
              if (s2 & 1)
                acc_o = __fmaf_rn(ec, uval[s2], acc_o);
              else
                acc_e = __fmaf_rn(ec, uval[s2], acc_e);
            }
            const float o = __fmul_rn(p.scale, __fadd_rn(xq, __fadd_rn(acc_e, acc_o)));
            outp[(int64_t)(c0 + t) * p.out_b_stride + ob] = float_to_bf16_bits(o);
          }
        }
      }
      // W entries 8 wg .. 8 wg + 7 of row (key) c: one 16-byte chunk per part.
      {
        uint32_t w0[4], w1[4], w2[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float a = Wk[2 * q], b = Wk[2 * q + 1];
          w0[q] = pack_bf16x2(a, b);
          float a0, b0;
          unpack_bf16x2(w0[q], a0, b0);
          const float ra = __fsub_rn(a, a0), rb = __fsub_rn(b, b0);
          w1[q] = pack_bf16x2(ra, rb);
          float a1, b1;
          unpack_bf16x2(w1[q], a1, b1);
          w2[q] = pack_bf16x2(__fsub_rn(ra, a1), __fsub_rn(rb, b1));
        }
        const uint32_t off = sw32_offset(128, c, 8 * wg);
        *reinterpret_cast<uint4*>(sW + off) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
        *reinterpret_cast<uint4*>(sW + PC_UW_PART + off) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
        *reinterpret_cast<uint4*>(sW + 2 * PC_UW_PART + off) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
      }
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

    if (ok) {  // the final state, rounded to bf16 once; row c, this group's columns, into the slot
      ok = __syncthreads_and(mbar_wait_bounded(barU, phU)) != 0;
      if (ok) {
        phU ^= 1u;
        pendU = false;
        tc_fence_after();
        uint16_t* grow = gstate + (int64_t)c * KD;
#pragma unroll 1
        for (int cb = 2 * wg; cb < 2 * wg + 2; ++cb) {
          float s[32];
          tmem_ld32(row_tmem + cb * 32, s);
          uint32_t w[16];
#pragma unroll
          for (int q = 0; q < 16; ++q) w[q] = pack_bf16x2(s[2 * q], s[2 * q + 1]);
          if constexpr (TMA) {  // 16-byte aligned pool
            uint4* dst = reinterpret_cast<uint4*>(grow + cb * 32);
#pragma unroll
            for (int q = 0; q < 4; ++q) dst[q] = make_uint4(w[4 * q], w[4 * q + 1], w[4 * q + 2], w[4 * q + 3]);
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
      for (int t = t0 + wg; t < t1; t += PC_WG) outp[(int64_t)t * p.out_b_stride + ob] = 0;
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
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, PC_TMEM_COLS);
  }
}

// ---------------------------------------------------------------- host side

template <bool TMA>
static cudaError_t launch_pftc(const CUtensorMap& map, const kda_params& p, const int32_t* cu, int num_seqs,
                               cudaStream_t s) {
  auto kern = kda_prefill_tc_kernel<TMA>;
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
  kern<<<(unsigned)grid, PC_THREADS, smem, s>>>(map, q, cu, num_seqs);
  return cudaGetLastError();
}

cudaError_t launch_prefill_tc(const kda_params& p, const int32_t* cu, int num_seqs, bool bulk, cudaStream_t s) {
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (bulk) {
    const cudaError_t e = state_tensor_map(p, &map);
    if (e != cudaSuccess) return e;
    return launch_pftc<true>(map, p, cu, num_seqs, s);
  }
  return launch_pftc<false>(map, p, cu, num_seqs, s);
}

}  // namespace kda
