// kda_prefill_chain.cu - varlen prefill in two stages (sm_103a), the reading
// of include/kda_prefill.h: a preparation kernel that turns every 16-token
// chunk of every (sequence, head) into the operands of the state-carrying
// step, in parallel over all chunks, and a chain kernel that carries each
// (sequence, head) through its chunks with the fp32 state in tensor memory.
//
// Source: "feat(kda): add CuTe DSL recurrent prefill backend" (PR #4605): the
// embedded #4675 commit text (Description) builds the long-sequence prefill
// as a two-stage BT16 portfolio, a preparation stage followed by a
// recurrence-chain stage, and the review threads give the call a
// caller-owned workspace that holds what the stages share.
//
// Arithmetic. Within a chunk of C <= 16 tokens starting from state S_0 (keys x
// values), with P_t = d_0 ... d_t, w_ts = d_{s+1} ... d_t and the L2-normalised
// k and q (the notation of kda_prefill_tc.cu):
//   u_t = beta_t (v_t - S_0^T (P_t k_t) - sum_{s<t} cc[t][s] u_s)
//   o_t = scale (S_0^T (P_t q_t) + sum_{s<=t} ec[t][s] u_s)
//   S_C = diag(P_{C-1}) S_0 + sum_s (w_{C-1,s} k_s) u_s^T
// with cc[t][s] = (w_ts k_s) . k_t and ec[t][s] = (w_ts k_s) . q_t. u is affine
// in S_0, u_t = U_t - S_0^T W_t, where (forward substitution over the chunk's
// tokens, independent of S_0)
//   U_t = beta_t (v_t - sum_{s<t} cc[t][s] U_s),    W_t = beta_t (P_t k_t - sum_{s<t} cc[t][s] W_s),
// and then o_t = scale (S_0^T Q_t + O_t) with
//   Q_t = P_t q_t - sum_{s<=t} ec[t][s] W_s,         O_t = sum_{s<=t} ec[t][s] U_s.
// The preparation kernel writes, per (chunk, head), one chunk image: -W and Q
// as two bf16 parts (the B operand of the chain's first product), the decayed
// keys K~_s = w_{C-1,s} k_s as three bf16 parts (the B operand of its second),
// U and O in fp32 and P_{C-1}. The chain, per chunk, for value row i:
//   1. S_0 row i (tensor memory) -> two bf16 parts (the A operand), and
//      S <- diag(P_{C-1}) S_0 in tensor memory;
//   2. D = S_0^T [-W | Q] on the tensor cores (the products hi.hi, lo.hi
//      and hi.lo of the parts, the state and the vectors exact to about
//      2^-17: per K step one N = 64 product of the state's high part with
//      both parts of the vectors, whose rows lie together in the image, and
//      one N = 32 product of its low part with their high part; the hi.lo
//      sums, in their own columns, are added when D is read);
//   3. u_t = U_t + D_t, as three bf16 parts;
//   4. S += sum_t K~_t u_t^T on the tensor cores (the six products of order
//      <= 2 of the parts, exact to about 2^-24), while o_t = scale (D_{16+t} + O_t)
//      is formed and stored.
// Tokens past a chunk's end enter with decay 1, beta 0 and zero vectors, so
// their rows of every operand are zero.
//
// Workspace: chunk images (slot, head), slot = the number of chunks of the
// sequences before this one whose bounds are in order and inside [0, B], plus
// the chunk's index in its sequence; ceil(B / 16) + num_seqs slots bound them
// for any sequences whose token ranges do not overlap.
#include <cuda.h>

#include <algorithm>
#include <cstring>
#include <mutex>

#include "kda_chunk.cuh"
#include "kda_device.cuh"
#include "kda_launch.h"
#include "kda_prefill.h"
#include "kda_tc.cuh"

namespace kda {

constexpr int CH = KDA_MAX_T;  // tokens per chunk
constexpr int CH_THREADS = 128;

// One chunk image (bytes). XB: 64 rows x 128 keys, K-major, 128-byte swizzle
// (sw128_offset with R = 64): rows 0..15 the high parts of -W_t, 16..31 of
// Q_t, 32..63 the low parts in the same order. KW: three parts of 128 key
// rows x 16 tokens, 32-byte swizzle. U, O: fp32 [16 tokens][128 value rows].
// PL: P_{C-1} per key channel. The offsets keep every operand 1024-byte
// aligned relative to the image.
constexpr uint32_t IMG_XB = 0u;
constexpr uint32_t IMG_XB_LO = 32u * 128u;  // low-part rows, 32 rows after the high ones in each 64-key half
constexpr uint32_t IMG_KW = 16384u;
constexpr uint32_t IMG_KW_PART = 4096u;
constexpr uint32_t IMG_U = 28672u;
constexpr uint32_t IMG_O = 36864u;
constexpr uint32_t IMG_PL = 45056u;
constexpr uint32_t IMG_STAGED = IMG_U;  // XB and KW: staged in shared memory, stored by one bulk copy
static_assert(IMG_PL + 512u == kPrefillChunkImageBytes, "chunk image layout");

// The first chunk image of sequence `seq`: the chunk counts of the sequences
// before it whose bounds are in order and inside [0, B]. Every thread of the
// CTA (at most 256 threads) calls it; `scratch` holds one int per warp.
__device__ int chunk_base(const int32_t* __restrict__ cu, int seq, int B, int* scratch) {
  int s = 0;
  for (int k = threadIdx.x; k < seq; k += blockDim.x) {
    const int a = cu[k], b = cu[k + 1];
    if (a >= 0 && b >= a && b <= B) s += (b - a + CH - 1) / CH;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
  if ((threadIdx.x & 31) == 0) scratch[threadIdx.x >> 5] = s;
  __syncthreads();
  int r = 0;
  for (int w = 0; w < (int)(blockDim.x >> 5); ++w) r += scratch[w];
  __syncthreads();  // scratch is free again
  return r;
}

// ---------------------------------------------------------------- preparation

// Token inputs staged in shared memory (16-byte aligned views): q, k, v and
// g_raw of a chunk, [tensor][token][128 channels] bf16, two buffers.
constexpr uint32_t PP_TOK_BYTES = 4u * CH * KD * 2u;

struct PpLayout {
  uint32_t stage, tok, red, fcp, rn, beta, xpose, scratch, total;
};

__host__ __device__ inline PpLayout pp_layout(bool vec) {
  PpLayout L{};
  uint32_t o = 0;
  L.stage = o;  // XB and KW of the chunk being written
  o += IMG_STAGED;
  L.tok = o;
  if (vec) o += 2u * PP_TOK_BYTES;
  L.red = o;  // per-warp partial sums: norms, then the coefficients
  o += (1u + CH * CH / 32u) * 512u;
  L.fcp = o;  // (cc[t][s], ec[t][s]) at pair t * 16 + s
  o += CH * CH * 8u;
  L.rn = o;
  o += 2u * CH * 4u;
  L.beta = o;
  o += CH * 4u;
  L.xpose = o;
  o += 4u * XPOSE_WARP_BYTES;
  L.scratch = o;
  o += 16u;
  L.total = o;
  return L;
}

__host__ __device__ inline size_t pp_smem_bytes(bool vec) { return (size_t)pp_layout(vec).total + 1024; }
// One preparation group's shared memory inside the single-launch kernel (1024-byte multiple).
constexpr uint32_t PP_GROUP_STRIDE = 90112u;

// 16 bytes global -> shared without registers (cp.async); src_bytes 0 fills zeros and reads nothing.
__device__ __forceinline__ void cp_async16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_addr(dst)), "l"(src), "r"(src_bytes)
               : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait_prev() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// q, k, v and g_raw of the chunk of Tc tokens at row c0 (head h) into `buf`,
// 16 bytes per copy, zeros past Tc: piece i = (tensor, token, 8 channels).
// gtid: the thread's index in its 128-thread group.
__device__ __forceinline__ void issue_token_copies(const kda_params& p, int c0, int h, int Tc, unsigned char* buf,
                                                   int gtid) {
#pragma unroll
  for (int m = 0; m < 8; ++m) {
    const int i = gtid + CH_THREADS * m;  // tensor m / 2, token (i / 16) % 16, channels 8 (i % 16) ..
    const int t = (i >> 4) & (CH - 1), c8 = i & 15;
    const kda_view& vw = m < 2 ? p.q : m < 4 ? p.k : m < 6 ? p.v : p.g_raw;
    const int tt = t < Tc ? t : 0;
    const uint16_t* src = static_cast<const uint16_t*>(vw.ptr) + (int64_t)(c0 + tt) * vw.b_stride +
                          (int64_t)h * vw.h_stride + 8 * c8;
    cp_async16(buf + (uint32_t)i * 16u, src, t < Tc ? 16u : 0u);
  }
}

// A chunk to prepare: token rows c0 .. c0 + Tc - 1 of head h into chunk image `img`.
struct PrepItem {
  int c0, Tc, h;
  long long img;
  bool ok;  // false: no more items
};

// Chunk image `img` is complete and visible to every SM: the bulk stores of
// this thread have completed (wait), the group's plain stores are ordered
// before this thread by a group barrier, and the flag is set with release.
__device__ __forceinline__ void publish_image(uint32_t* flags, long long img) {
  bulk_wait_all();
  asm volatile("fence.proxy.async.global;" ::: "memory");
  __threadfence();
  asm volatile("st.release.gpu.global.u32 [%0], %1;" ::"l"(flags + img), "r"(1u) : "memory");
}

// One 128-thread group prepares next(0), next(1), ... in order, until an item
// with ok == false: thread gtid is key channel gtid and value row gtid; `bar`
// is the group's barrier (0 when the group is the whole CTA); `sm` its
// 1024-aligned shared memory (pp_layout(VEC)). VEC: q, k, v and g_raw rows
// are 16-byte aligned, and the next item's token inputs are copied into
// shared memory while the current one is computed. flags: NULL, or one word
// per chunk image, set once the image is complete (publish_image).
template <bool VEC, class Next>
__device__ void prepare_items(const kda_params& p, const int gtid, const uint32_t bar, unsigned char* sm,
                              unsigned char* __restrict__ ws, uint32_t* flags, Next next) {
  const int tid = gtid, warp = tid >> 5, lane = tid & 31;
  const PpLayout SL = pp_layout(VEC);
  unsigned char* stage = sm + SL.stage;
  unsigned char* stok = sm + SL.tok;
  float* red = reinterpret_cast<float*>(sm + SL.red);
  float* fcp = reinterpret_cast<float*>(sm + SL.fcp);
  float* rn = reinterpret_cast<float*>(sm + SL.rn);
  float* sbeta = reinterpret_cast<float*>(sm + SL.beta);
  float* xtile = reinterpret_cast<float*>(sm + SL.xpose + warp * XPOSE_WARP_BYTES);
  auto gsync = [&]() { bar_sync(bar, CH_THREADS); };

  PrepItem cur = next(0);
  uint16_t blogit_next = 0;
  if (VEC && cur.ok) {
    issue_token_copies(p, cur.c0, cur.h, cur.Tc, stok, tid);
    cp_async_commit();
    if (tid < cur.Tc) blogit_next = load_bits(p.beta_logit, cur.c0, tid, cur.h, 0);
  }
  long long last_img = -1;  // the image whose flag is still to be set

  for (int k = 0, buf = 0; cur.ok; ++k, buf ^= 1) {
    const PrepItem nxt = next(k + 1);
    const int c0 = cur.c0, Tc = cur.Tc, h = cur.h;
    unsigned char* gimg = ws + cur.img * kPrefillChunkImageBytes;
    TokenRegs<CH> L;
    if constexpr (VEC) {
      L.blogit = blogit_next;
      L.alog = 0.0f;
      L.dtb = 0.0f;
      if (p.gate_mode == KDA_GATE_RAW) {
        L.alog = p.A_log[h];
        L.dtb = p.dt_bias[(int64_t)h * KD + tid];
      }
      if (nxt.ok) {  // the next item's inputs fly while this one is computed
        issue_token_copies(p, nxt.c0, nxt.h, nxt.Tc, stok + (buf ^ 1) * PP_TOK_BYTES, tid);
        blogit_next = tid < nxt.Tc ? load_bits(p.beta_logit, nxt.c0, tid, nxt.h, 0) : (uint16_t)0;
      }
      cp_async_commit();
      cp_async_wait_prev();  // this item's copies have landed (each thread's own)
      gsync();               // and everyone's
      const uint16_t* tk = reinterpret_cast<const uint16_t*>(stok + buf * PP_TOK_BYTES) + tid;
#pragma unroll
      for (int t = 0; t < CH; ++t) {
        L.qv[t] = tk[(0 * CH + t) * KD];
        L.kv[t] = tk[(1 * CH + t) * KD];
        L.vv[t] = tk[(2 * CH + t) * KD];
        L.gv[t] = tk[(3 * CH + t) * KD];
      }
    } else {
      zero_tokens(L);
      load_tokens(p, c0, h, Tc, L);  // thread index = threadIdx.x: the group is the whole CTA here
    }

    // L2 norms: block sums of q_t^2 (value t) and k_t^2 (value CH + t).
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      const float q = bf16_bits_to_float(L.qv[t]), kq = bf16_bits_to_float(L.kv[t]);
      tile_put(xtile, lane, t, __fmul_rn(q, q));
      tile_put(xtile, lane, CH + t, __fmul_rn(kq, kq));
    }
    __syncwarp();
    {
      const float s = tile_row_sum(xtile, lane);
      __syncwarp();
      red[warp * 32 + lane] = s;
    }
    gsync();
    if (tid < 2 * CH) rn[tid] = inv_norm(block_sum(red, 0, tid));
    gsync();

    // Channel tid: the normalised vectors, the gate, P_t.
    const FastGate gate(p, L.alog);
    if (tid < CH) sbeta[tid] = tid < Tc ? gate.beta(bf16_bits_to_float(L.blogit)) : 0.0f;
    float qh[CH], kh[CH], dd[CH], P[CH];
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      qh[t] = __fmul_rn(bf16_bits_to_float(L.qv[t]), rn[t]);
      kh[t] = __fmul_rn(bf16_bits_to_float(L.kv[t]), rn[CH + t]);
      dd[t] = t < Tc ? __expf(gate.g(bf16_bits_to_float(L.gv[t]), L.dtb)) : 1.0f;
    }
    {
      float run = 1.0f;
#pragma unroll
      for (int t = 0; t < CH; ++t) {
        run = __fmul_rn(run, dd[t]);
        P[t] = run;
      }
    }

    // Coefficients M[a][b] (flat a CH + b): a > b holds cc[a][b], a <= b holds
    // ec[b][a]; block sums of per-channel products with w a running product.
#pragma unroll
    for (int a0 = 0; a0 < CH; a0 += 32 / CH) {
      float vals[32];
#pragma unroll
      for (int r = 0; r < 32 / CH; ++r) {
        const int a = a0 + r;
#pragma unroll
        for (int b2 = 0; b2 < CH; ++b2) vals[r * CH + b2] = 0.0f;
        float w = 1.0f;  // w_{a,b} for b = a-1, a-2, ...
#pragma unroll
        for (int b2 = CH - 1; b2 >= 0; --b2) {
          if (b2 < a) {
            w = __fmul_rn(w, dd[b2 + 1]);
            vals[r * CH + b2] = __fmul_rn(__fmul_rn(w, kh[b2]), kh[a]);
          }
        }
        float w2 = 1.0f;  // w_{b,a} for b = a, a+1, ...
#pragma unroll
        for (int b2 = 0; b2 < CH; ++b2) {
          if (b2 >= a) {
            if (b2 > a) w2 = __fmul_rn(w2, dd[b2]);
            vals[r * CH + b2] = __fmul_rn(__fmul_rn(w2, kh[a]), qh[b2]);
          }
        }
      }
      red[((1 + a0 * CH / 32) * 4 + warp) * 32 + lane] = warp_sum32(vals, xtile, lane);
    }
    // The decayed keys of channel tid: K~_s = (d_{s+1} ... d_{15}) k_s.
    float Kt[CH];
    {
      float wl = 1.0f;
#pragma unroll
      for (int s = CH - 1; s >= 0; --s) {
        Kt[s] = __fmul_rn(wl, kh[s]);
        wl = __fmul_rn(wl, dd[s]);
      }
    }
    gsync();  // partial sums, beta
    for (int i = tid; i < CH * CH; i += CH_THREADS) {
      const float v = block_sum(red, 1 + (i >> 5), i & 31);
      fcp[2 * i] = v;
      fcp[2 * ((i % CH) * CH + i / CH) + 1] = v;
    }
    gsync();

    // Forward substitution, channel tid (W, Q) and value row tid (U, O) as
    // packed pairs: (W_t, U_t) = beta_t ((P_t k_t, v_t) - sum_{s<t} cc[t][s] (W_s, U_s)),
    // (Q_t, O_t) = (P_t q_t, 0) - (1, -1) sum_{s<=t} ec[t][s] (W_s, U_s).
    f32x2 wu[CH];
    float Qc[CH], Ov[CH];
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      f32x2 ce[CH];
#pragma unroll
      for (int s2 = 0; s2 <= t / 2; ++s2) {
        const float4 c = reinterpret_cast<const float4*>(fcp + 2 * t * CH)[s2];
        ce[2 * s2] = pk2(c.x, c.y);
        ce[2 * s2 + 1] = pk2(c.z, c.w);
      }
      f32x2 acc0 = pk2(0.0f, 0.0f), acc1 = pk2(0.0f, 0.0f);
#pragma unroll
      for (int s = 0; s < t; ++s) {
        float c, e;
        upk2(ce[s], c, e);
        (void)e;
        if (s & 1)
          acc1 = fma2(pk2(c, c), wu[s], acc1);
        else
          acc0 = fma2(pk2(c, c), wu[s], acc0);
      }
      const float bt = sbeta[t];
      const f32x2 rhs = pk2(__fmul_rn(P[t], kh[t]), bf16_bits_to_float(L.vv[t]));
      wu[t] = mul2(pk2(bt, bt), sub2(rhs, add2(acc0, acc1)));
      f32x2 e0 = pk2(0.0f, 0.0f), e1 = pk2(0.0f, 0.0f);
#pragma unroll
      for (int s = 0; s <= t; ++s) {
        float c, e;
        upk2(ce[s], c, e);
        (void)c;
        if (s & 1)
          e1 = fma2(pk2(e, e), wu[s], e1);
        else
          e0 = fma2(pk2(e, e), wu[s], e0);
      }
      float ew, eu;
      upk2(add2(e0, e1), ew, eu);
      Qc[t] = __fsub_rn(__fmul_rn(P[t], qh[t]), ew);
      Ov[t] = eu;
    }

    // The image: XB and KW staged, then one bulk store; U, O and P_{C-1}
    // straight to global memory. Before the stage is rewritten the previous
    // item's bulk store has read it (with flags: has completed, and that
    // item's image is published).
    if (tid == 0) {
      if (flags != nullptr && last_img >= 0)
        publish_image(flags, last_img);
      else
        bulk_wait_read_all();
    }
    gsync();
    {
      const Sw128Col col = sw128_col(64, tid);
#pragma unroll
      for (int t = 0; t < CH; ++t) {
        float w, u;
        upk2(wu[t], w, u);
        store_split_at(stage + IMG_XB, stage + IMG_XB + IMG_XB_LO, sw128_at(col, t), -w);
        store_split_at(stage + IMG_XB, stage + IMG_XB + IMG_XB_LO, sw128_at(col, CH + t), Qc[t]);
      }
      store_row_split3(stage + IMG_KW, IMG_KW_PART, tid, Kt);
    }
    float* gU = reinterpret_cast<float*>(gimg + IMG_U);
    float* gO = reinterpret_cast<float*>(gimg + IMG_O);
#pragma unroll
    for (int t = 0; t < CH; ++t) {
      float w, u;
      upk2(wu[t], w, u);
      gU[t * KD + tid] = u;
      gO[t * KD + tid] = Ov[t];
    }
    reinterpret_cast<float*>(gimg + IMG_PL)[tid] = P[CH - 1];
    fence_proxy_async_smem();
    gsync();
    if (tid == 0) {
      bulk_s2g(gimg + IMG_XB, stage, IMG_STAGED);
      bulk_commit();
    }
    last_img = cur.img;
    cur = nxt;
  }
  gsync();  // every thread's plain stores of the last image before its flag
  if (tid == 0) {
    if (flags != nullptr && last_img >= 0)
      publish_image(flags, last_img);
    else
      bulk_wait_all();
  }
  if (VEC) asm volatile("cp.async.wait_all;" ::: "memory");
}

// CTA (sequence, head, z) prepares chunks z, z + Z, z + 2Z, ... of its
// sequence (the two-launch schedule, configuration 5). p: t_stride = b_stride
// in every activation view (token t of a chunk starting at row c0 is (b = c0, t)).
template <bool VEC>
__global__ void __launch_bounds__(CH_THREADS) kda_prefill_prepare_kernel(const kda_params p,
                                                                         const int32_t* __restrict__ cu,
                                                                         const int num_seqs, const int Z,
                                                                         unsigned char* __restrict__ ws,
                                                                         const long long ws_images) {
  // The chain kernel's CTAs may launch once every CTA of this grid has
  // started; they wait for the whole grid before they read a chunk image.
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  int* scratch = reinterpret_cast<int*>(sm + pp_layout(VEC).scratch);

  const int item = blockIdx.x;
  const int z = item % Z, sh = item / Z;
  const int seq = sh / p.H, h = sh - seq * p.H;
  if (seq >= num_seqs) return;
  const int t0 = cu[seq], t1 = cu[seq + 1];
  if (t0 < 0 || t1 < t0 || t1 > p.B) return;  // the chain kernel reports it
  const int n = p.state_indices[seq];
  if (n < 0 || n >= p.N) return;  // inactive: the chain kernel writes zero outputs
  const int nch = (t1 - t0 + CH - 1) / CH;
  if (z >= nch) return;
  const int base = chunk_base(cu, seq, p.B, scratch);
  auto next = [&](int k) {
    const int j = z + k * Z;
    PrepItem it;
    it.c0 = t0 + j * CH;
    it.Tc = min(CH, t1 - it.c0);
    it.h = h;
    it.img = (long long)(base + j) * p.H + h;
    it.ok = j < nch && it.img < ws_images;  // beyond ws_images only with overlapping token ranges (undefined)
    return it;
  };
  prepare_items<VEC>(p, threadIdx.x, 0u, sm, ws, nullptr, next);
}

// ---------------------------------------------------------------- chain

// 288 threads. Threads 0..255 (warps 0-7) work on the state: thread i is
// value row i % 128 of half i / 128; in the state's conversion a half takes
// 64 of the 128 key columns, in the epilogue 8 of the 16 tokens. Warp 8
// issues the tensor-core products and the chunk-image copies, so that the
// conversion never waits for an issue: the state warps signal it through
// named barriers (bar.arrive) and go on.
constexpr int CN_WORKERS = 256;
constexpr int CN_THREADS = CN_WORKERS + 32;
constexpr int CN_MMA_WARP = CN_WORKERS / 32;
constexpr uint32_t CN_TMEM_COLS = 512;
constexpr uint32_t CN_D = 128;   // D of the first product: columns 128..191 (hi.hi + lo.hi, then hi.lo)
constexpr uint32_t CN_AS = 256;  // S as two bf16 parts, the first product's A operand: part p at 256 + 64 p
constexpr uint32_t CN_AU = 384;  // u as three bf16 parts, the update's A operand: part p at 384 + 8 p
constexpr int CN_NBUF = 3;       // chunk images in flight
constexpr uint32_t CN_IMG_STRIDE = (kPrefillChunkImageBytes + 1023u) & ~1023u;
// Named barriers between the state warps and the issuing warp.
constexpr uint32_t CN_BAR_ROUND0 = 1, CN_BAR_ROUND1 = 2, CN_BAR_U = 3;

struct CnLayout {
  uint32_t a, img, bar, tslot, scratch, total;
};

__host__ __device__ inline CnLayout cn_layout() {
  CnLayout L{};
  uint32_t o = 0;
  L.a = o;  // the slot's bf16 state (first chunk), 128-byte swizzle
  o += 128u * 256u;
  L.img = o;
  o += CN_NBUF * CN_IMG_STRIDE;
  L.bar = o;  // barA, barD, barU, barI[CN_NBUF]
  o += 64u;
  L.tslot = o;
  o += 16u;
  L.scratch = o;  // one int per warp (chunk_base)
  o += 64u;
  L.total = o;
  return L;
}

__host__ __device__ inline size_t cn_smem_bytes() { return (size_t)cn_layout().total + 1024; }

// Chunk image `img` has been published (publish_image); false if the bounded wait gave up.
__device__ __forceinline__ bool wait_image_bounded(const uint32_t* flags, long long img) {
  const uint32_t* f = flags + img;
  auto ready = [&]() {
    uint32_t v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(f) : "memory");
    return v != 0u;
  };
  bool ok = ready();
  if (!ok) {
    const unsigned long long t0 = global_timer_ns();
    for (unsigned it = 1; it < WAIT_LIMIT_ITERS; ++it) {
      __nanosleep(64);
      if ((ok = ready())) break;
      if ((it & 255u) == 0 && global_timer_ns() - t0 > WAIT_LIMIT_NS) break;
    }
  }
  if (ok) asm volatile("fence.proxy.async.global;" ::: "memory");  // the image is read by bulk copies
  return ok;
}

// The chain over items it0, it0 + stride, ... (item = (sequence, head)) by
// one CTA of 288 threads (or 320: a tenth warp that only copies images) with
// shared memory `sm` (cn_layout). flags: NULL when the images are complete
// before the chain starts (two launches), else each image's copy waits for
// its flag (one launch, preparation running beside). Thread `loader` issues
// the image copies: lane 0 of the issuing warp, or of the tenth warp, which
// takes part in no per-round barrier, so that a flag wait never holds up a
// product.
template <bool TMA>
__device__ __forceinline__ void chain_items(const CUtensorMap* smap_p, const kda_params& p, const int32_t* __restrict__ cu,
                            const int num_seqs, const unsigned char* __restrict__ ws, const long long ws_images,
                            const uint32_t* flags, const int it0, const int stride, const int loader,
                            unsigned char* sm) {
  const CUtensorMap& smap = *smap_p;
  const int tid = threadIdx.x, warp = tid >> 5;
  const bool worker = tid < CN_WORKERS, issuer = warp == CN_MMA_WARP;
  const int row = tid & (KD - 1), hf = tid >> 7;  // meaningful in the state warps
  const int total = num_seqs * p.H;

  const CnLayout SL = cn_layout();
  unsigned char* sA = sm + SL.a;
  unsigned char* sImg = sm + SL.img;
  uint64_t* barA = reinterpret_cast<uint64_t*>(sm + SL.bar);  // the slot's state copy
  uint64_t* barD = barA + 1;                                   // first product
  uint64_t* barU = barA + 2;                                   // update product
  uint64_t* barI = barA + 3;                                   // chunk images, one per buffer
  uint32_t* tslot = reinterpret_cast<uint32_t*>(sm + SL.tslot);
  int* scratch = reinterpret_cast<int*>(sm + SL.scratch);
  uint16_t* outp = static_cast<uint16_t*>(p.out);

  if (tid == 0) {
    mbar_init(barA, 1);
    mbar_init(barD, 1);
    mbar_init(barU, 1);
    for (int b = 0; b < CN_NBUF; ++b) mbar_init(barI + b, 1);
  }
  if (warp == 0) tmem_alloc(tslot, CN_TMEM_COLS);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tslot;
  const uint32_t row_tmem = tmem + ((uint32_t)((warp & 3) * 32) << 16);  // lane `row`, column 0

  uint32_t phA = 0, phD = 0, phU = 0;
  uint32_t phI = 0u, pendI = 0u;  // per image buffer b, bit b: its barrier's phase, a copy in flight
  bool pendA = false, pendD = false, pendU = false;
  bool broken = false;

  for (int it = it0; it < total; it += stride) {
    const int seq = it / p.H, h = it - seq * p.H;
    const int t0 = cu[seq], t1 = cu[seq + 1];
    const int n = p.state_indices[seq];
    if (t0 < 0 || t1 < t0 || t1 > p.B) {
      if (tid == 0 && h == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_SEQLENS);
      continue;
    }
    const int64_t ob = (int64_t)h * p.out_h_stride + row;  // output element of row `row`, + token row * out_b_stride
    if (n < 0 || n >= p.N || broken) {
      if (worker)
        for (int t = t0 + hf; t < t1; t += 2) outp[(int64_t)t * p.out_b_stride + ob] = 0;
      continue;
    }
    if (t0 == t1) continue;
    const int base = chunk_base(cu, seq, p.B, scratch);
    const int nch = (t1 - t0 + CH - 1) / CH;
    if ((long long)(base + nch) * p.H > ws_images) {  // only overlapping token ranges get here (undefined)
      if (worker)
        for (int t = t0 + hf; t < t1; t += 2) outp[(int64_t)t * p.out_b_stride + ob] = 0;
      continue;
    }
    uint16_t* gstate = static_cast<uint16_t*>(p.state) + (int64_t)n * p.state_slot_stride + (int64_t)h * KD * KD;
    // Chunk j's image into buffer bb, once it is published (one launch);
    // a wait that gives up issues nothing, and the chain's own bounded wait
    // on the buffer then reports it.
    auto issue_image = [&](int j, int bb) {
      const long long img = (long long)(base + j) * p.H + h;
      if (flags != nullptr && !wait_image_bounded(flags, img)) return;
      mbar_expect_tx(barI + bb, kPrefillChunkImageBytes);
      bulk_g2s(sImg + bb * CN_IMG_STRIDE, ws + img * (long long)kPrefillChunkImageBytes, kPrefillChunkImageBytes,
               barI + bb);
    };

    if constexpr (TMA) {
      if (tid == 0) {
        mbar_expect_tx(barA, KD * KD * 2);
        tma_load_3d(sA, &smap, 0, h * KD, n, barA);
        tma_load_3d(sA + KD * 128, &smap, 64, h * KD, n, barA);
      }
      pendA = true;
    } else if (worker) {
      for (int r = hf; r < KD; r += 2)
        *reinterpret_cast<uint16_t*>(sA + sw128_offset(KD, r, row)) = gstate[(int64_t)r * KD + row];
    }
    for (int j = 0; j < min(CN_NBUF, nch); ++j) {
      if (tid == loader) issue_image(j, j);
      pendI |= 1u << j;
    }

    bool first = true, ok = true;
    for (int j = 0; j < nch; ++j) {
      const int c0 = t0 + j * CH, Tc = min(CH, t1 - c0);
      const int b = j % CN_NBUF;
      unsigned char* im = sImg + b * CN_IMG_STRIDE;

      // 1. The previous update has finished with S, u and its chunk image; on
      // the first chunk the slot's state has arrived; this chunk's image has.
      {
        bool w_ok = true;
        if (pendU) w_ok = mbar_wait_bounded(barU, phU);
        if (TMA && first && w_ok) w_ok = mbar_wait_bounded(barA, phA);
        if (w_ok) w_ok = mbar_wait_bounded(barI + b, (phI >> b) & 1u);
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
      phI ^= 1u << b;
      pendI &= ~(1u << b);
      if (j >= 1 && j + 2 < nch) {  // chunk j + 2 into the buffer chunk j - 1 has released
        const int bn = (j + 2) % CN_NBUF;
        if (tid == loader) issue_image(j + 2, bn);
        pendI |= 1u << bn;
      }
      tc_fence_after();

      // 2. Each half of the state warps loads its two 32-column blocks of row
      // `row` at once; in two rounds it converts one block into its bf16
      // parts (tensor memory, the A operand) and signals the issuing warp,
      // which issues the first product's K steps that the round completed
      // (block cb holds K steps 2 cb and 2 cb + 1); then S <- P_{C-1} S for
      // both blocks, off the products' path (the update, which adds to S,
      // comes after the u phase's store wait). D[row][t'] = sum_k S[row][k] XB[t'][k]:
      // the high parts of both, the low part of S with the high rows of XB,
      // the high part of S with the low rows (the first chunk's S is exact in
      // one part; its low part is written as zero).
      if (worker) {
        const float* splast = reinterpret_cast<const float*>(im + IMG_PL);
        float s[2][32];  // the thread's two 32-column blocks, cb = 2 hf and 2 hf + 1
        if (!first) tmem_ld32x2(row_tmem + 64 * hf, s[0], s[1]);
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
          const int cb = 2 * hf + rd;
          if (first) {  // the slot's bf16 row, exact: one part
            uint32_t hw[16];
#pragma unroll
            for (int c = 0; c < 4; ++c) {
              const uint4 raw = *reinterpret_cast<const uint4*>(sA + sw128_offset(KD, row, cb * 32 + 8 * c));
              hw[4 * c] = raw.x;
              hw[4 * c + 1] = raw.y;
              hw[4 * c + 2] = raw.z;
              hw[4 * c + 3] = raw.w;
            }
#pragma unroll
            for (int q = 0; q < 16; ++q) unpack_bf16x2(hw[q], s[rd][2 * q], s[rd][2 * q + 1]);
            tmem_st16(row_tmem + CN_AS + cb * 16, hw);
            uint32_t zw[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) zw[q] = 0u;
            tmem_st16(row_tmem + CN_AS + 64 + cb * 16, zw);  // the low part of an exact state is zero
          } else {
            uint32_t hw[16], lw[16];
#pragma unroll
            for (int q = 0; q < 16; ++q) {
              const float s0 = s[rd][2 * q], s1 = s[rd][2 * q + 1];
              hw[q] = pack_bf16x2(s0, s1);
              lw[q] = f32x2_to_bf16x2(sub2(pk2(s0, s1), bf16x2_to_f32x2(hw[q])));
            }
            tmem_st16(row_tmem + CN_AS + cb * 16, hw);
            tmem_st16(row_tmem + CN_AS + 64 + cb * 16, lw);
          }
          tmem_st_wait();
          tc_fence_before();
          bar_arrive(rd == 0 ? CN_BAR_ROUND0 : CN_BAR_ROUND1, CN_THREADS);
        }
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {  // S <- P_{C-1} S, both blocks after both rounds
          const int cb = 2 * hf + rd;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            const float4 pl = *reinterpret_cast<const float4*>(splast + cb * 32 + 4 * c);
            f32x2 a = mul2(pk2(pl.x, pl.y), pk2(s[rd][4 * c], s[rd][4 * c + 1]));
            f32x2 bb = mul2(pk2(pl.z, pl.w), pk2(s[rd][4 * c + 2], s[rd][4 * c + 3]));
            upk2(a, s[rd][4 * c], s[rd][4 * c + 1]);
            upk2(bb, s[rd][4 * c + 2], s[rd][4 * c + 3]);
          }
          tmem_st32(row_tmem + cb * 32, s[rd]);  // waited for by the u phase's tmem_st_wait, before the update
        }
      } else if (issuer) {
        // Every operand is formed before the first barrier, so that the issue
        // itself (while the state warps convert, on the same schedulers) is
        // the products alone.
        const uint32_t x0 = smem_addr(im + IMG_XB);
        const uint32_t tb = __shfl_sync(0xffffffffu, tmem, 0), xb = __shfl_sync(0xffffffffu, x0, 0);
        // N = 64 (the 32 high rows of XB, then its 32 low rows) and N = 32
        // (the high rows alone) from the same K-step address.
        constexpr uint32_t idesc64 = idesc_bf16_f32(128, 4 * CH), idesc32 = idesc_bf16_f32(128, 2 * CH);
        static_assert(IMG_XB_LO == 32u * 128u, "the low rows follow the high rows");
        uint64_t bh[8];
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) bh[kk] = sw128_desc(xb + (kk >> 2) * (64 * 128) + (kk & 3) * 32);
        const uint32_t dcol = tb + CN_D, acol = tb + CN_AS;
#pragma unroll
        for (int rd = 0; rd < 2; ++rd) {
          bar_sync(rd == 0 ? CN_BAR_ROUND0 : CN_BAR_ROUND1, CN_THREADS);
          tc_fence_after();
#pragma unroll
          for (int i = 0; i < 4; ++i) {  // K steps of blocks rd and 2 + rd
            const int kk = (i < 2 ? 2 * rd : 4 + 2 * rd) + (i & 1);
            tc_mma_bf16_ta_w(dcol, acol + kk * 8, bh[kk], idesc64, (rd > 0 || i > 0) ? 1u : 0u);
            tc_mma_bf16_ta_w(dcol, acol + 64 + kk * 8, bh[kk], idesc32, 1u);
          }
        }
        tc_commit_w(barD);
      }
      pendD = true;
      ok = __syncthreads_and(mbar_wait_bounded(barD, phD)) != 0;
      if (!ok) break;
      phD ^= 1u;
      pendD = false;
      tc_fence_after();

      // 3. Tokens 8 hf .. 8 hf + 7 of row `row`: u_t = U_t + D_t as three bf16
      // parts into tensor memory (the update's A operand); 4. the issuing warp
      // issues S += sum_t u_t K~_t (the products of order <= 2 of the three
      // parts of each) while the state warps form the chunk's outputs.
      if (worker) {
        float dx[8], dy[8];
        {
          // x and y of tokens 8 hf .., then their hi.lo sums, by one wait
          const uint32_t at[4] = {row_tmem + CN_D + 8 * hf, row_tmem + CN_D + CH + 8 * hf,
                                  row_tmem + CN_D + 2 * CH + 8 * hf, row_tmem + CN_D + 3 * CH + 8 * hf};
          float d4[4][8];
          tmem_ld8x4(at, d4);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            dx[i] = __fadd_rn(d4[0][i], d4[2][i]);
            dy[i] = __fadd_rn(d4[1][i], d4[3][i]);
          }
        }
        const float* gu = reinterpret_cast<const float*>(im + IMG_U) + (8 * hf) * KD + row;
        {
          uint32_t w0[4], w1[4], w2[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const f32x2 u = add2(pk2(gu[(2 * q) * KD], gu[(2 * q + 1) * KD]), pk2(dx[2 * q], dx[2 * q + 1]));
            w0[q] = f32x2_to_bf16x2(u);
            const f32x2 r1 = sub2(u, bf16x2_to_f32x2(w0[q]));
            w1[q] = f32x2_to_bf16x2(r1);
            w2[q] = f32x2_to_bf16x2(sub2(r1, bf16x2_to_f32x2(w1[q])));
          }
          tmem_st4(row_tmem + CN_AU + 4 * hf, w0);
          tmem_st4(row_tmem + CN_AU + 8 + 4 * hf, w1);
          tmem_st4(row_tmem + CN_AU + 16 + 4 * hf, w2);
        }
        tmem_st_wait();
        tc_fence_before();
        bar_arrive(CN_BAR_U, CN_THREADS);
        const float* go = reinterpret_cast<const float*>(im + IMG_O) + (8 * hf) * KD + row;
        uint16_t* orow = outp + (int64_t)(c0 + 8 * hf) * p.out_b_stride + ob;
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float o = __fmul_rn(p.scale, __fadd_rn(dy[i], go[i * KD]));
          if (8 * hf + i < Tc) *orow = float_to_bf16_bits(o);
          orow += p.out_b_stride;
        }
      } else if (issuer) {
        bar_sync(CN_BAR_U, CN_THREADS);
        tc_fence_after();
        const uint32_t tb = __shfl_sync(0xffffffffu, tmem, 0);
        const uint32_t w0 = __shfl_sync(0xffffffffu, smem_addr(im + IMG_KW), 0);
        constexpr uint32_t idesc = idesc_bf16_f32(128, 128);
#pragma unroll
        for (int q = 0; q < 6; ++q) {
          const uint32_t pa = q < 3 ? (uint32_t)q : (q == 4 ? 1u : 0u);
          const uint32_t pb = q < 3 ? 0u : (q == 5 ? 2u : 1u);
          tc_mma_bf16_ta_w(tb, tb + CN_AU + 8 * pa, sw32_desc(w0 + pb * IMG_KW_PART), idesc, 1u);
        }
        tc_commit_w(barU);
      }
      pendU = true;
      first = false;
    }
    if (worker) tmem_st_wait();  // a rescale still in flight after a wait that gave up

    if (ok) {  // the final state, rounded to bf16 once; row `row`, columns 64 hf .. 64 hf + 63, into the slot
      ok = __syncthreads_and(mbar_wait_bounded(barU, phU)) != 0;
      if (ok) {
        phU ^= 1u;
        pendU = false;
        tc_fence_after();
        if (worker) {
          uint16_t* grow = gstate + (int64_t)row * KD;
#pragma unroll 1
          for (int cb = 2 * hf; cb < 2 * hf + 2; ++cb) {
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
    }
    if (!ok) {  // a bounded wait gave up: the sequence is skipped, and every later one
      broken = true;
      if (tid == 0 && p.error_word != nullptr) atomicOr(p.error_word, KDA_ERR_TIMEOUT);
      if (worker)
        for (int t = t0 + hf; t < t1; t += 2) outp[(int64_t)t * p.out_b_stride + ob] = 0;
    }
    tc_fence_before();
    __syncthreads();  // this item's tensor-memory and shared-memory use is done
    tc_fence_after();
  }

  // Anything still in flight after a wait that gave up gets one more bounded
  // wait before the tensor memory is released and the CTA leaves.
  if (tid == 0) {
    if (pendA) mbar_drain_bounded(barA, phA);
    if (pendD) mbar_drain_bounded(barD, phD);
    if (pendU) mbar_drain_bounded(barU, phU);
    for (int b = 0; b < CN_NBUF; ++b)
      if ((pendI >> b) & 1u) mbar_drain_bounded(barI + b, (phI >> b) & 1u);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, CN_TMEM_COLS);
  }
}

// The chain of the two-launch schedule (configuration 5): after the
// preparation grid, persistent over (sequence, head) items.
template <bool TMA>
__global__ void __launch_bounds__(CN_THREADS, 1)
    kda_prefill_chain_kernel(const __grid_constant__ CUtensorMap smap, const kda_params p,
                             const int32_t* __restrict__ cu, const int num_seqs,
                             const unsigned char* __restrict__ ws, const long long ws_images) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  // The preparation grid has finished and its chunk images are visible.
  asm volatile("griddepcontrol.wait;" ::: "memory");
  chain_items<TMA>(&smap, p, cu, num_seqs, ws, ws_images, nullptr, blockIdx.x, gridDim.x, CN_WORKERS, sm);
}

// ---------------------------------------------------------------- one launch

// The single-launch schedule (configuration 6), a cooperative grid of one CTA
// per SM, 320 threads: CTA c < num_seqs * H carries chain c (its tenth warp
// copies the images); every other CTA runs two preparation groups (warps 0-3
// and 4-7) over the chunk images in chunk-major
// order (chunk 0 of every chain, then chunk 1, ...), publishing each image with
// a flag that the chains wait for. The preparation never waits for a chain,
// and every CTA is resident (cooperative launch), so every wait ends.
constexpr int FU_MAX_SEQS = 32;
constexpr uint32_t FU_TABLE = 2 * PP_GROUP_STRIDE;  // the sequence table, after the two groups' regions
static_assert(28672u + 2u * PP_TOK_BYTES + 9u * 512u + 2048u + 128u + 64u + 4u * XPOSE_WARP_BYTES + 16u <=
                  PP_GROUP_STRIDE,
              "a preparation group's shared memory");

constexpr int FU_THREADS = CN_THREADS + 32;

__device__ __noinline__ void fused_prepare_role(const kda_params* pp, const int32_t* __restrict__ cu,
                                                const int num_seqs, const int nchains, unsigned char* __restrict__ ws,
                                                const long long ws_images, uint32_t* flags, unsigned char* sm);

template <bool TMA>
__global__ void __launch_bounds__(FU_THREADS, 1)
    kda_prefill_fused_kernel(const __grid_constant__ CUtensorMap smap, const __grid_constant__ kda_params p,
                             const int32_t* __restrict__ cu, const int num_seqs, unsigned char* __restrict__ ws,
                             const long long ws_images, uint32_t* flags) {
  extern __shared__ unsigned char smem_raw[];
  unsigned char* sm = smem_raw + ((1024u - (smem_addr(smem_raw) & 1023u)) & 1023u);
  const int nchains = num_seqs * p.H;  // at most half the grid (host)
  if ((int)blockIdx.x < nchains) {
    chain_items<TMA>(&smap, p, cu, num_seqs, ws, ws_images, flags, blockIdx.x, nchains, CN_THREADS, sm);
    return;
  }
  fused_prepare_role(&p, cu, num_seqs, nchains, ws, ws_images, flags, sm);
}

// The preparation role of the one-launch kernel, compiled as a function of its
// own (not inlined), so that its register demand does not shape the chain
// role's code in the same kernel.
__device__ __noinline__ void fused_prepare_role(const kda_params* pp, const int32_t* __restrict__ cu,
                                                const int num_seqs, const int nchains, unsigned char* __restrict__ ws,
                                                const long long ws_images, uint32_t* flags, unsigned char* sm) {
  const kda_params& p = *pp;
  // Sequence table: first row, chunk count, first image, active.
  int* st0 = reinterpret_cast<int*>(sm + FU_TABLE);
  int* snch = st0 + FU_MAX_SEQS;
  int* sbase = snch + FU_MAX_SEQS;
  int* smax = sbase + FU_MAX_SEQS;
  if (threadIdx.x == 0) {
    int base = 0, mx = 0;
    for (int s2 = 0; s2 < num_seqs; ++s2) {
      const int a = cu[s2], b = cu[s2 + 1];
      const bool wf = a >= 0 && b >= a && b <= p.B;  // well formed
      const int nc = wf ? (b - a + CH - 1) / CH : 0;
      const int n = p.state_indices[s2];
      st0[s2] = a;
      sbase[s2] = base;
      snch[s2] = (wf && n >= 0 && n < p.N) ? nc : 0;  // chunks to prepare
      base += nc;
      mx = max(mx, snch[s2]);
    }
    smax[0] = mx;
  }
  __syncthreads();
  if (threadIdx.x >= 2 * CH_THREADS) return;  // warps 8 and 9 have no preparation role
  const int g = threadIdx.x / CH_THREADS, gtid = threadIdx.x % CH_THREADS;
  const long long Q = 2LL * (gridDim.x - nchains);
  const long long slots = (long long)smax[0] * nchains;
  long long pos = 2LL * (blockIdx.x - nchains) + g - Q;  // advanced by Q before each use
  const int t1_cap = p.B;
  auto next = [=](int) mutable {
    PrepItem it;
    it.ok = false;
    for (pos += Q; pos < slots; pos += Q) {
      const int j = (int)(pos / nchains), c = (int)(pos % nchains);
      const int s2 = c / p.H, h = c - s2 * p.H;
      if (j >= snch[s2]) continue;
      const long long img = (long long)(sbase[s2] + j) * p.H + h;
      if (img >= ws_images) continue;  // only overlapping token ranges (undefined)
      it.c0 = st0[s2] + j * CH;
      it.Tc = min(CH, min(cu[s2 + 1], t1_cap) - it.c0);
      it.h = h;
      it.img = img;
      it.ok = true;
      break;
    }
    return it;
  };
  prepare_items<true>(p, gtid, 1u + (uint32_t)g, sm + g * PP_GROUP_STRIDE, ws, flags, next);
}

// ---------------------------------------------------------------- host side

// The workspace of kda_prefill_static: one fixed array per device that loads
// the library, for callers that cannot allocate. Host code must not pass the
// array's name to a kernel (on the host it names a stand-in, not device
// memory); prefill_static_workspace gives its device address.
static __device__ __align__(256) unsigned char g_prefill_static_ws[KDA_PREFILL_STATIC_BYTES];

cudaError_t prefill_static_workspace(void** ptr) {
  constexpr int kMaxDevices = 256;
  static std::mutex mu;
  static void* addr[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(mu);
  if (addr[dev] == nullptr) {  // once per device, with that device current
    void* a = nullptr;
    if ((e = cudaGetSymbolAddress(&a, g_prefill_static_ws)) != cudaSuccess) return e;
    addr[dev] = a;
  }
  *ptr = addr[dev];
  return cudaSuccess;
}

long long prefill_chunk_images(int B, int num_seqs, int H) {
  return ((long long)(B + CH - 1) / CH + num_seqs) * (long long)H;
}

size_t prefill_workspace_size(int B, int num_seqs, int H) {
  const long long images = prefill_chunk_images(B, num_seqs, H);
  return (size_t)images * kPrefillChunkImageBytes + (((size_t)images * 4u + 15u) & ~(size_t)15u);
}

template <bool TMA>
static cudaError_t launch_fused(const CUtensorMap& map, const kda_params& q, const int32_t* cu, int num_seqs,
                                unsigned char* ws, long long images, uint32_t* flags, int sms, cudaStream_t s) {
  auto kern = kda_prefill_fused_kernel<TMA>;
  const size_t smem = std::max(cn_smem_bytes(), (size_t)FU_TABLE + 4u * FU_MAX_SEQS * 4u + 1024u);
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  int per_sm = 0;
  if ((e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, FU_THREADS, smem)) != cudaSuccess) return e;
  if (per_sm < 1) return cudaErrorCooperativeLaunchTooLarge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)sms);  // one CTA per SM, all resident
  cfg.blockDim = dim3(FU_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, map, q, cu, num_seqs, ws, images, flags);
}

cudaError_t launch_prefill_fused(const kda_params& p, const int32_t* cu, int num_seqs, void* ws, bool bulk,
                                 cudaStream_t s) {
  const long long images = prefill_chunk_images(p.B, num_seqs, p.H);
  unsigned char* w = static_cast<unsigned char*>(ws);
  uint32_t* flags = reinterpret_cast<uint32_t*>(w + images * kPrefillChunkImageBytes);
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  if (num_seqs > FU_MAX_SEQS || 2LL * num_seqs * p.H > sms) return cudaErrorInvalidConfiguration;
  if ((e = cudaMemsetAsync(flags, 0, (size_t)images * 4u, s)) != cudaSuccess) return e;
  kda_params q = p;  // token t of a chunk is activation row c0 + t
  q.q.t_stride = q.q.b_stride;
  q.k.t_stride = q.k.b_stride;
  q.v.t_stride = q.v.b_stride;
  q.g_raw.t_stride = q.g_raw.b_stride;
  q.beta_logit.t_stride = q.beta_logit.b_stride;
  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  if (bulk) {
    if ((e = state_tensor_map(p, &map)) != cudaSuccess) return e;
    return launch_fused<true>(map, q, cu, num_seqs, w, images, flags, sms, s);
  }
  return launch_fused<false>(map, q, cu, num_seqs, w, images, flags, sms, s);
}

bool prefill_rows_aligned16(const kda_params& p) {
  auto ok = [](const kda_view& v) {
    return (reinterpret_cast<uintptr_t>(v.ptr) & 15u) == 0 && v.b_stride % 8 == 0 && v.h_stride % 8 == 0;
  };
  return ok(p.q) && ok(p.k) && ok(p.v) && ok(p.g_raw);
}

template <bool TMA>
static cudaError_t launch_chain(const CUtensorMap& map, const kda_params& q, const int32_t* cu, int num_seqs,
                                const unsigned char* ws, long long images, int sms, cudaStream_t s) {
  auto kern = kda_prefill_chain_kernel<TMA>;
  const size_t smem = cn_smem_bytes();
  static std::atomic<bool> smem_set{false};  // one flag per instantiation
  cudaError_t e = set_smem_limit_once(kern, smem, smem_set);
  if (e != cudaSuccess) return e;
  const long long items = (long long)num_seqs * q.H;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(items, (long long)sms));
  cfg.blockDim = dim3(CN_THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  // The chain's set-up (barriers, tensor memory) overlaps the preparation
  // grid's last CTAs; its CTAs wait for that grid at griddepcontrol.wait.
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, map, q, cu, num_seqs, ws, images);
}

cudaError_t launch_prefill_chain(const kda_params& p, const int32_t* cu, int num_seqs, void* ws, bool bulk,
                                 cudaStream_t s) {
  const long long images = prefill_chunk_images(p.B, num_seqs, p.H);
  int dev = 0, sms = 0;
  cudaError_t e;
  if ((e = cudaGetDevice(&dev)) != cudaSuccess) return e;
  if ((e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev)) != cudaSuccess) return e;
  kda_params q = p;  // token t of a chunk is activation row c0 + t
  q.q.t_stride = q.q.b_stride;
  q.k.t_stride = q.k.b_stride;
  q.v.t_stride = q.v.b_stride;
  q.g_raw.t_stride = q.g_raw.b_stride;
  q.beta_logit.t_stride = q.beta_logit.b_stride;

  // Preparation: Z CTAs per (sequence, head), enough for about 8 CTAs per SM
  // when there are few sequences, never more than a sequence can have chunks.
  {
    const bool vec = prefill_rows_aligned16(q);
    auto kern = vec ? kda_prefill_prepare_kernel<true> : kda_prefill_prepare_kernel<false>;
    const size_t smem = pp_smem_bytes(vec);
    static std::atomic<bool> smem_set_vec{false}, smem_set_plain{false};
    if ((e = set_smem_limit_once(kern, smem, vec ? smem_set_vec : smem_set_plain)) != cudaSuccess) return e;
    const long long per = (long long)num_seqs * p.H;
    const long long want = 8LL * sms;
    long long Z = std::max(1LL, (want + per - 1) / per);
    Z = std::min(Z, (long long)(p.B + CH - 1) / CH);
    Z = std::max(Z, 1LL);
    const long long grid = per * Z;
    if (grid > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
    kern<<<(unsigned)grid, CH_THREADS, smem, s>>>(q, cu, num_seqs, (int)Z, static_cast<unsigned char*>(ws), images);
    if ((e = cudaGetLastError()) != cudaSuccess) return e;
  }

  CUtensorMap map;
  memset(&map, 0, sizeof(map));
  const unsigned char* cws = static_cast<const unsigned char*>(ws);
  if (bulk) {
    if ((e = state_tensor_map(p, &map)) != cudaSuccess) return e;
    return launch_chain<true>(map, q, cu, num_seqs, cws, images, sms, s);
  }
  return launch_chain<false>(map, q, cu, num_seqs, cws, images, sms, s);
}

}  // namespace kda
