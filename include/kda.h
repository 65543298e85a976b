/*
 * kda.h - C ABI of the GB300 (sm_103a) KDA gated delta-rule serving step.
 *
 * KDA (Kimi Delta Attention) keeps, per sequence slot and head, a 128x128
 * state S (keys x values). One decode step on a slot and head:
 *
 *   q_hat = q / sqrt(|q|^2 + 1e-6),  k_hat likewise            (L2 norm)
 *   g_c   = lower_bound * sigmoid(exp(A_log[h]) * (g_raw_c + dt_bias[h][c]))
 *   S     <- diag(exp(g)) S                          (per key channel c)
 *   u     =  sigmoid(beta_logit) * (v - S^T k_hat)
 *   S     <- S + k_hat u^T
 *   o     =  scale * S^T q_hat
 *
 * Sources (FlashInfer pull-request pages):
 *   "feat(kda): add packed-input CuTe decode kernel" (PR #4417): the T=1
 *     step on a bf16 pool [N,12,128,128] updated in place through
 *     state_indices, rows outside the pool give zero output and leave the
 *     pool untouched (opening paragraph); raw gate with lower_bound=-5,
 *     beta logits, in-kernel q/k L2 norm, fp32 internal math, strided
 *     q/k/v/g views and padded pools (section "T=1 fast path inside
 *     recurrent_kda"); the fused output (section "Kernel design").
 *   "feat(kda): ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)"
 *     (PR #4864): T-token speculative verify against a (k_hat, u, G) ring
 *     cache with fold into the checkpoint at flush_min (sections "What it
 *     does", "API", "Caching").
 *
 * Conventions shared by every call
 *   - Every tensor pointer is a DEVICE pointer owned by the caller. The
 *     library allocates nothing, never synchronizes, never reads device
 *     memory on the host, and enqueues its kernels on `stream` (a
 *     cudaStream_t; NULL is the legacy default stream).
 *   - The return value is the result of host-side validation of the
 *     arguments and of the launch itself. Nothing is launched unless it is
 *     KDA_OK. kda_last_error() then describes the failure.
 *   - bf16 values are IEEE bfloat16 (2 bytes); fp32 is IEEE binary32.
 *   - state_indices[b] outside [0, N) marks row b inactive: its outputs are
 *     zero and no state, ring or hist_len word is touched. This is not an
 *     error. Two active rows with the same index in one call are undefined.
 *   - The state pool is laid out [N][H][V][K] with K contiguous: the stored
 *     row for value index v holds S[0..K-1][v]. Slot n starts
 *     state_slot_stride elements after slot n-1 (padded pools allowed).
 *   - A state pool whose base is 16-byte aligned and whose slot stride is a
 *     multiple of 8 elements is moved with bulk asynchronous copies;
 *     otherwise a plain-load variant of the same kernel runs (same results,
 *     bit for bit). Neither case is an error.
 *   - `out` must not overlap the state pool or any input.
 *   - The calls are deterministic: the same inputs give the same bits across
 *     CUDA-graph replays, and whatever the CUDA-core launch configuration
 *     (0-3); the tensor-core verify configuration (4) sums the dot products
 *     in another order and agrees with them to rounding.
 *   - Arithmetic is fp32 with fp32 CUDA math functions; the state and the
 *     outputs are rounded to bf16 (round to nearest even) when stored.
 */
#ifndef KDA_GB300_KDA_H
#define KDA_GB300_KDA_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
  KDA_OK = 0,
  KDA_EINVAL = 1,        /* an argument is malformed (null, misaligned, negative, overlapping) */
  KDA_EUNSUPPORTED = 2,  /* well-formed but outside what the library supports (K or V != 128, H > 64, T > 16) */
  KDA_ELAUNCH = 3        /* the CUDA launch was rejected (no sm_103a device, bad stream, ...) */
} kda_status;

/* Bits a kernel ORs into the optional device error word (kda_params.error_word). */
#define KDA_ERR_HIST_LEN 1u /* a ring slot's hist_len was outside [0, W]; that slot was skipped */
#define KDA_ERR_TIMEOUT 2u  /* a bounded wait (1 s) for an async copy gave up; that tile was skipped: zero
                               output, its state (and ring entries) untouched; a ring call still resets
                               hist_len of rows that reached flush_min (stream-ordered, unaware of the skip) */
#define KDA_ERR_CACHE_BASE 4u /* a ring slot's cache_base was outside [0, W); that slot was skipped */

/* kda_params.gate_mode: how g_raw and beta_logit are read (source: PR #4417, "T=1 fast path
   inside recurrent_kda", which covers both recurrent_kda calling conventions). */
#define KDA_GATE_RAW 0         /* g = lower_bound * sigmoid(exp(A_log) * (g_raw + dt_bias)), beta = sigmoid(beta_logit) */
#define KDA_GATE_PRECOMPUTED 1 /* g_raw holds the log-space decay g, beta_logit holds beta; A_log, dt_bias,
                                  lower_bound unused (A_log and dt_bias may be NULL) */

/* Largest number of tokens kda_verify and kda_verify_ring accept. */
#define KDA_MAX_T 16

/*
 * A strided bf16 activation tensor [B][T][H][D] with D contiguous: element
 * (b, t, h, c) is at ((const uint16_t*)ptr)[b*b_stride + t*t_stride +
 * h*h_stride + c]. Strides are in elements and must be >= 0. t_stride is
 * ignored when T == 1. Any 2-byte alignment is accepted, so q, k and v can
 * be zero-copy views into one fused projection row, e.g. a packed QKV row
 * [3][H][128] has b_stride = row length and offsets 0, H*128, 2*H*128.
 */
typedef struct {
  const void* ptr;
  int64_t b_stride;
  int64_t t_stride;
  int64_t h_stride;
} kda_view;

/* Arguments of one step over B rows. T is passed to the call. */
typedef struct {
  int32_t B; /* batch rows, >= 0; B == 0 launches nothing */
  int32_t H; /* heads, 1..64 (Kimi K3 at TP=8 uses 12) */
  int32_t K; /* key dimension; must be 128 */
  int32_t V; /* value dimension; must be 128 */
  int32_t N; /* slots in the state pool, >= 0; N == 0 makes every row inactive */

  kda_view q, k, v, g_raw; /* bf16 [B][T][H][128]; g_raw is g itself under KDA_GATE_PRECOMPUTED */
  kda_view beta_logit;     /* bf16 [B][T][H]; h_stride steps heads (D = 1); beta itself under
                              KDA_GATE_PRECOMPUTED */
  const float* A_log;      /* fp32 [H] */
  const float* dt_bias;    /* fp32 [H][K] */
  float lower_bound;       /* gate lower bound, the pages use -5 */
  float scale;             /* output scale, 1 for o = S^T q_hat */

  void* state;               /* bf16 [N][H][V][K], updated in place */
  int64_t state_slot_stride; /* elements between slots, >= H*V*K when N > 1 */
  const int32_t* state_indices; /* int32 [B] */

  void* out; /* bf16 [B][T][H][V] */
  int64_t out_b_stride, out_t_stride, out_h_stride; /* elements, V contiguous */

  uint32_t* error_word;    /* optional device word (NULL = none); KDA_ERR_* bits are ORed in */
  int32_t config_override; /* -1: kda_select_config decides; else an index < kda_num_configs() */
  int32_t gate_mode;       /* KDA_GATE_RAW (0) or KDA_GATE_PRECOMPUTED (1) */
} kda_params;

/*
 * T=1 decode: one step for every row of p (source: PR #4417, opening
 * paragraph and "T=1 fast path inside recurrent_kda"). Reads q, k, v,
 * g_raw, beta_logit with T = 1, updates each active row's slot in place and
 * writes out[b][0][h][:].
 */
kda_status kda_decode(const kda_params* p, void* stream);

/*
 * T-token speculative verify (source: PR #4864, "API": T is the draft length
 * inferred from q's shape, 8 and 4 in the pages). Equal to T consecutive
 * kda_decode calls on the same slots: the state is rounded to bf16 after
 * every token, kept on chip between tokens, and written back once. The
 * CUDA-core configurations (0-3) are equal bit for bit; configuration 4
 * computes each token's two dot products of every state row on the tensor
 * cores (the query vectors in three bf16 parts, fp32 accumulation) and is
 * equal to rounding. Writes out[b][t][h][:] for t < T. 1 <= T <= KDA_MAX_T.
 */
kda_status kda_verify(const kda_params* p, int32_t T, void* stream);

/* The ring cache of PR #4864 ("Caching"), indexed by the same pool slots. */
typedef struct {
  void* k_cache; /* bf16 [N][H][W][K]: L2-normalised keys k_hat of past tokens */
  void* u_cache; /* bf16 [N][H][W][V]: corrections u = beta (v - (D S)^T k_hat) */
  void* g_cache; /* fp32 [N][H][W][K]: cumulative log-decay G, restarting at 0 after a fold */
  int64_t k_slot_stride, u_slot_stride, g_slot_stride; /* elements between slots, >= H*W*128 */
  int32_t* hist_len; /* int32 [N], live entries per slot; set to 0 on a fold when restart_hist_on_flush */
  int32_t W;         /* ring width (entries per slot and head), 1..64; the pages use 16 and 32 */
  int32_t flush_min; /* fold when hist_len >= flush_min; needs flush_min >= 1 and flush_min-1+T <= W */
  int32_t restart_hist_on_flush; /* nonzero: a fold writes hist_len = 0 */
  const int32_t* cache_base; /* optional int32 [N]: ring position P of slot n is entry (cache_base[n] + P) mod W;
                                NULL means 0 for every slot. Read, never written. */
} kda_ring_params;

/*
 * Ring-cache verify with replay and fold (source: PR #4864, "What it does",
 * "API", "Caching"). For each active row b, slot n = state_indices[b],
 * h = hist_len[n]:
 *   - h outside [0, W]: KDA_ERR_HIST_LEN is ORed into p->error_word and the
 *     row is skipped (zero output, nothing touched); likewise a cache_base
 *     outside [0, W) with KDA_ERR_CACHE_BASE;
 *   - ring positions are circular from cache_base[n] (the page names this
 *     argument without defining it; a per-slot ring start is its plainest
 *     reading): position P is stored at entry (cache_base[n] + P) mod W;
 *   - the current state is the checkpoint p->state[n] replayed through ring
 *     entries j < h: S <- diag(exp(G_j - G_{j-1})) S + k_j u_j^T, G_{-1} = 0;
 *   - if h >= flush_min the state is folded first: the checkpoint becomes
 *     its bf16 rounding, new tokens start at ring position 0 and G at 0,
 *     and hist_len[n] = 0 if restart_hist_on_flush; otherwise new tokens go
 *     to positions h..h+T-1 and G continues from G_{h-1};
 *   - token t at position P: G_P = fp32(G_{P-1} + g_t); D = exp(G_P - G_{P-1});
 *     k~ = bf16(k_hat_t); u = beta_t (v_t - (D S)^T k~); u~ = bf16(u);
 *     S <- D S + k~ u~^T; out[b][t] = scale S^T q_hat_t; (k~, u~, G_P) are
 *     written at position P.
 * The checkpoint is written only by a fold. hist_len is otherwise left to
 * the caller, who adds the number of accepted draft tokens afterwards.
 * The ring kernel works on whole heads: p->config_override must be -1 or the
 * 128-row configuration (3), anything else returns KDA_EUNSUPPORTED. Its
 * 2T dot products per state row, and a fold's replay, run on the tensor
 * cores with fp32 accumulation (operands split into bf16 parts, exact to
 * 2^-17 relative for the query vectors and 2^-25 for the fold's history
 * keys).
 */
kda_status kda_verify_ring(const kda_params* p, int32_t T, const kda_ring_params* r, void* stream);

/*
 * Launch configurations and the per-batch selector (source: PR #4417,
 * "Kernel design", the per-batch policy bullet: the decode picks its kernel
 * shape and value-row tile from the batch size, smaller tiles for small
 * batches and whole-head tiles once the batch fills the GPU, and a tile_v
 * override forces one for sweeps; the thresholds here are this library's own,
 * measured on GB300). kda_params.config_override takes an index. 0-3:
 * CUDA-core tiles of 16, 32, 64 and 128 value rows per CTA; 4: whole heads with
 * the dot products on the tensor cores, kda_verify with T > 1 only
 * (KDA_EUNSUPPORTED otherwise).
 *   kda_num_configs:   the number of configurations (5).
 *   kda_config_tile_v: rows of V per CTA of a configuration; -1 outside 0..4.
 * Pure host functions: no device, no CUDA call.
 */
int32_t kda_num_configs(void);
int32_t kda_config_tile_v(int32_t config);
/* The configuration kda_decode (T = 1) and kda_verify (T > 1) pick for B rows
   (same source; -1 if B < 0 or T is outside 1..KDA_MAX_T). */
int32_t kda_select_config(int32_t B, int32_t T);
/* The configuration kda_verify_ring picks for B rows and T tokens (same source):
   always 3, whole heads, because the ring kernel's product takes all 128 state
   rows of a head at once (-1 as above). */
int32_t kda_select_ring_config(int32_t B, int32_t T);

/* Message for the last non-OK status returned on this host thread ("" if none),
   the error convention every call above follows: a kda_status return value for
   host-side validation and launch, and this thread-local text beside it (source:
   PR #4417, review comments asking that tile overrides and arguments be checked
   before launch and rejected with a clear configuration error rather than reach
   the kernel). The pointer stays valid until the next call on the same thread. */
const char* kda_last_error(void);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_H */
