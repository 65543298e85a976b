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

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_PREFILL_H */
