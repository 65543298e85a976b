/*
 * kda_prefill.h - varlen prefill on the bf16 state pool of kda.h.
 *
 * Source: "feat(kda): add CuTe DSL recurrent prefill backend" (FlashInfer
 * PR #4605): recurrent_kda prefill over packed sequences described by
 * cu_seqlens (offsets that start at zero and never decrease), with a
 * caller-owned initial state read from and written back to an indexed state
 * pool in place, and explicit output buffers (Description and review
 * sections). The pages give no arithmetic beyond the KDA step itself; this
 * library's reading:
 *
 *   For sequence i, tokens t = cu_seqlens[i] .. cu_seqlens[i+1]-1 in order,
 *   starting from S = the bf16 slot state_indices[i], every token applies the
 *   kda_decode step (kda.h) to S in fp32, writes o_t = scale * S_t^T q_hat_t
 *   (rounded to bf16) to out row t, and keeps S in fp32 for the next token.
 *   After the last token, S is rounded to bf16 (round to nearest even) once
 *   and stored in the slot. A one-token sequence is exactly one kda_decode
 *   step: bit for bit in configurations 0-3, to rounding in configuration 4.
 *
 * The activations are kda_decode's T = 1 views with one row per token:
 * q, k, v, g_raw bf16 [B][H][128] and beta_logit bf16 [B][H], B = the total
 * number of token rows; out bf16 [B][H][V]. t_stride and out_t_stride are
 * ignored. Everything else in kda_params (pool, gate convention, scale,
 * error word, alignment rules) means what it means for kda_decode, except:
 *   - state_indices has num_seqs entries, one slot per sequence; a slot
 *     outside [0, N) makes the sequence inactive: its out rows are zero and
 *     the pool is not touched;
 *   - B == 0 or num_seqs == 0 launches nothing;
 *   - config_override is -1 (the library chooses: 4), 0..3 (the recurrence
 *     token by token on the CUDA cores, value-row tiles of kda_config_tile_v())
 *     or 4 (chunks of 16 tokens with the chunk math on the tensor cores, the
 *     page's BT16 chunked form: per chunk, every value row's dot products with
 *     the chunk's decayed keys and queries as one product, a 16-step scalar
 *     recurrence per row, and the state update as a second product onto the
 *     fp32 state held in tensor memory; its products take the fp32 operands
 *     as bf16 parts: the state and the vectors to about 2^-17 relative in the
 *     dot products, u and the decayed keys to about 2^-24 in the update).
 *     Both compute the reading above; they round differently within fp32.
 *
 * cu_seqlens is a DEVICE int32 array [num_seqs + 1], read only by the kernel
 * (the host never reads device memory). Sequence i is skipped, and
 * KDA_ERR_SEQLENS is ORed into the error word, when cu_seqlens[i] < 0,
 * cu_seqlens[i+1] < cu_seqlens[i] or cu_seqlens[i+1] > B. Out rows that no
 * valid sequence covers are not written. An empty sequence touches nothing.
 * Two active sequences with the same slot, or overlapping token ranges, are
 * undefined.
 */
#ifndef KDA_GB300_KDA_PREFILL_H
#define KDA_GB300_KDA_PREFILL_H

#include <stddef.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* Bit a prefill kernel ORs into kda_params.error_word for a sequence whose
   cu_seqlens bounds are out of order or outside [0, B]. */
#define KDA_ERR_SEQLENS 8u

/* The packed sequences of one prefill call. */
typedef struct {
  const int32_t* cu_seqlens; /* device int32 [num_seqs + 1]; may be NULL when num_seqs == 0 */
  int32_t num_seqs;          /* >= 0 */
} kda_seqs;

/*
 * Varlen prefill: every sequence of s, in place on its slot (the reading
 * above). Host-side validation: p and s non-NULL, num_seqs >= 0; with
 * num_seqs > 0, kda_decode's checks with T = 1 (config_override -1..4) and
 * cu_seqlens non-NULL and 4-byte aligned (KDA_EINVAL or KDA_EUNSUPPORTED
 * otherwise).
 */
kda_status kda_prefill(const kda_params* p, const kda_seqs* s, void* stream);

/* The configuration kda_prefill picks for num_seqs sequences of H heads: 4, the
   chunked tensor-core kernel (source: PR #4605, Description: the BT16 chunked
   backend); -1 for negative num_seqs or H < 1. */
int32_t kda_select_prefill_config(int32_t num_seqs, int32_t H);

/*
 * Two-stage prefill with a caller-owned workspace.
 *
 * Source: PR #4605, the embedded #4675 commit text (Description): the
 * long-sequence prefill as a two-stage BT16 portfolio, a preparation stage
 * and then a recurrence-chain stage; the review threads pass the stages'
 * shared data through a caller-owned workspace (RecurrentKDAPrefillWorkspace).
 *
 * Configurations 5 and 6 of kda_prefill_ws compute the reading above in two
 * stages on the caller's stream. The first prepares every 16-token chunk of
 * every (sequence, head) at once: norms, gates, the chunk's 16 x 16
 * coefficients, and then by forward substitution the chunk's contribution to
 * u and o in a form that no longer depends on the state. It writes these
 * into the workspace. The second carries each (sequence, head) through its
 * chunks in order, the fp32 state in tensor memory, with two tensor-core
 * products per chunk: the state against the prepared vectors as two bf16
 * parts (exact to about 2^-17), and the update from u and the decayed keys
 * as three bf16 parts (exact to about 2^-24). Its results agree with
 * configurations 0-4 to rounding, not bit for bit.
 *   5: the stages as two launches, the chain after the whole preparation.
 *   6: both stages in one cooperative launch of one CTA per SM: num_seqs * H
 *      CTAs carry the chains while the others prepare the chunks in chunk
 *      order (chunk 0 of every chain first), and each chain waits (bounded)
 *      for a chunk's ready flag before reading it; bit for bit equal to 5.
 *      Needs num_seqs <= 32, 2 * num_seqs * H <= the device's SM count and
 *      the q, k, v and g_raw rows 16-byte aligned (pointer, b_stride and
 *      h_stride); the call clears the flags (cudaMemsetAsync on the stream).
 *
 * workspace: device memory of at least kda_prefill_workspace_bytes(B,
 * num_seqs, H) bytes, 16-byte aligned, owned by the caller, overlapping none
 * of the call's inputs, outputs or the state pool. Its contents on entry do
 * not matter and on return are unspecified; two calls in flight at once need
 * two workspaces.
 *
 * config_override: -1 lets kda_select_prefill_ws_config choose (its choice of
 * 6 becomes 5 when 6's conditions do not hold); 0..4 run kda_prefill's
 * configurations (the workspace is then not used and may be NULL); 5 and 6
 * the two stages. Validation as kda_prefill's, plus KDA_EINVAL for
 * configuration 5 or 6 with a NULL, unaligned, too small or overlapping
 * workspace, and KDA_EUNSUPPORTED for configuration 6 outside its conditions. Errors found on the device (KDA_ERR_SEQLENS,
 * KDA_ERR_TIMEOUT) are reported as kda_prefill reports them.
 */
kda_status kda_prefill_ws(const kda_params* p, const kda_seqs* s, void* workspace, size_t workspace_bytes,
                          void* stream);

/* Workspace bytes kda_prefill_ws needs in configurations 5 and 6 for B token
   rows, num_seqs sequences and H heads: n = (ceil(B / 16) + num_seqs) * H
   chunk images of 45568 bytes, then n 4-byte ready flags padded to a multiple
   of 16 bytes; 0 when B <= 0, num_seqs <= 0 or H < 1. */
size_t kda_prefill_workspace_bytes(int32_t B, int32_t num_seqs, int32_t H);

/* The configuration kda_prefill_ws picks: two stages when the sequences
   average at least 512 tokens (B >= 512 num_seqs) — 6 (one launch) for at
   most 32 sequences and 64 (sequence, head) chains, else 5 —, otherwise 4;
   -1 for negative B or num_seqs or H < 1. Source: PR #4605, #4675 commit text
   (Description): the preparation-and-chain schedules are selected from the
   physical device and the input shape. */
int32_t kda_select_prefill_ws_config(int32_t B, int32_t num_seqs, int32_t H);

/*
 * Two-stage prefill that allocates nothing, with the workspace inside the
 * library. No source page describes it: this entry point exists for callers
 * of this library that cannot call cudaMalloc when they run a prefill (a
 * step captured into a CUDA graph in global capture mode, where allocation
 * calls are not permitted; a plugin whose host framework owns all device
 * memory and forbids allocation while it enqueues work; a server that
 * reserved all device memory for its state pools at start-up).
 *
 * It runs configuration 5 of kda_prefill_ws with the workspace in a fixed
 * array of KDA_PREFILL_STATIC_BYTES (64 MiB) compiled into the library:
 * every GPU that loads the library holds those 64 MiB until the process
 * exits. The caller passes inputs and outputs as for kda_prefill_ws.
 *   - Limit: a call whose kda_prefill_workspace_bytes(B, num_seqs, H) exceeds
 *     64 MiB (more than 1472 chunk images with their flags; e.g. one sequence
 *     of more than 1936 tokens at H = 12) is rejected with KDA_EUNSUPPORTED and a message
 *     giving both sizes, before anything is launched; use kda_prefill_ws.
 *   - Set-up: the first call on a device looks up the array's device address
 *     with that device current; make that first call before any stream
 *     capture. Later calls only launch.
 *   - Sharing: every call uses the same array, which keeps the last call's
 *     contents; nothing in it has to start at zero (a call reads only what it
 *     wrote itself). Calls that overlap on the GPU (other streams, other host
 *     threads) race on the array and give undefined results.
 *   - config_override: -1 or 5 (both run configuration 5), else KDA_EINVAL;
 *     everything else as kda_prefill_ws.
 */
#define KDA_PREFILL_STATIC_BYTES (64u * 1024u * 1024u)
kda_status kda_prefill_static(const kda_params* p, const kda_seqs* s, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_PREFILL_H */
