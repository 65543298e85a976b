/*
 * kda_fp8.h - T=1 decode, T-token verify and the ring verify on an fp8 (E4M3) state pool: the C ABI.
 *
 * Source: "feat(kda): add packed-input CuTe decode kernel" (PR #4417),
 * section "Nsight Compute": the bf16 decode at B=512 already runs at the
 * machine's ceiling for its access pattern, so the remaining headroom is
 * fewer bytes per state element, for example an fp8 state. The pages fix no
 * format for it; this call implements the library's reading:
 *
 *   - codes: one byte per state element, the OCP 8-bit floating-point format
 *     E4M3 (1 sign bit, 4 exponent bits with bias 7, 3 mantissa bits;
 *     exponent field 0 holds the subnormals M * 2^-9; S.1111.111 is NaN; no
 *     infinities; largest finite magnitude 448), laid out [N][H][V][K] with
 *     K contiguous like the bf16 pool;
 *   - one fp32 scale per state row (slot, head, value index v), a power of
 *     two 2^e, laid out [N][H][V]: the row's key k holds code_k * 2^e;
 *   - the step is kda_decode's arithmetic on those exact values, and the
 *     output comes from the unrounded new state (rounded to bf16);
 *   - each updated row is requantized, decided in fp32: m = max_k |s'_k|,
 *     e = the smallest integer with m * 2^-e <= 448 (0 for an all-zero row,
 *     -134 when m < 2^-126), codes = E4M3 round-to-nearest-even of
 *     s' * 2^-e.
 * The codes of NaN (0x7F, 0xFF) must not occur in the pool; a scale that is
 * not a power of two in [2^-149, 2^127] gives undefined results.
 *
 * Everything in kda.h's conventions holds, with these differences:
 *   - kda_params.state points to the uint8 codes; state_slot_stride is in
 *     elements (bytes) and is at least H*V*K when N > 1.
 *   - The scales travel in a kda_fp8_pool. Both are read and rewritten in
 *     place for active rows only.
 *   - Bulk asynchronous copies are used when the codes' base is 16-byte
 *     aligned with a slot stride that is a multiple of 16, and the scales'
 *     base is 16-byte aligned with a slot stride that is a multiple of 4;
 *     otherwise a plain-load variant runs (same results, bit for bit).
 *   - config_override selects the rows of V per CTA like kda_decode's
 *     (0-3: 16, 32, 64, 128; -1: kda_select_config(B, 1)); 4 is
 *     KDA_EUNSUPPORTED.
 * The pages have no counterpart of this call's output to compare with: it is
 * checked against this library's fp64 oracle of the reading above.
 */
#ifndef KDA_GB300_KDA_FP8_H
#define KDA_GB300_KDA_FP8_H

#include <stdint.h>

#include "kda.h"

#ifdef __cplusplus
extern "C" {
#endif

/* The row scales of an fp8 state pool. */
typedef struct {
  float* scale;              /* fp32 [N][H][V], powers of two; DEVICE, caller-owned, in/out */
  int64_t scale_slot_stride; /* elements between slots; >= H*V when N > 1 */
} kda_fp8_pool;

/* One T=1 decode step on an fp8 pool. p as for kda_decode except p->state
   (uint8 E4M3 codes); f holds the scales. Returns KDA_EINVAL for a NULL or
   misaligned scale array (4 bytes), a slot stride below H*V, or `out`
   overlapping the codes or the scales; KDA_EUNSUPPORTED for
   config_override 4; otherwise as kda_decode. */
kda_status kda_decode_fp8(const kda_params* p, const kda_fp8_pool* f, void* stream);

/* T-token speculative verify on an fp8 pool (source: as kda_decode_fp8, with
   the verify of "feat(kda): ReplaySSM verify+flush decode kernel for Kimi K3
   (KDA)" (PR #4864), section "API": T draft tokens of each row on one slot).
   The reading: T kda_decode_fp8 steps in order on the same slot, the row
   requantized after every token (as kda_verify rounds the bf16 state after
   every token), so the call equals T kda_decode_fp8 calls bit for bit. p and
   f as for kda_decode_fp8 with kda_verify's token views ([B][T][H][...] by
   b_stride / t_stride / h_stride) and out [B][T][H][V]; 1 <= T <= KDA_MAX_T.
   config_override 0..3 as kda_decode_fp8's; -1: kda_select_config(B, T),
   with whole-head tiles where that picks configuration 4 (which, like 4
   given explicitly, has no fp8 form: KDA_EUNSUPPORTED). Errors as
   kda_decode_fp8 and kda_verify. */
kda_status kda_verify_fp8(const kda_params* p, int32_t T, const kda_fp8_pool* f, void* stream);

/* Ring-cache verify with replay and fold (kda_verify_ring) on an fp8
   checkpoint pool (source: as kda_verify_fp8; the ring from "feat(kda):
   ReplaySSM verify+flush decode kernel for Kimi K3 (KDA)" (PR #4864),
   sections "What it does", "API" and "Caching", whose ring entries k~, u~ stay
   bf16 and G fp32). The reading: the checkpoint S_0 is the pool's exact
   values codes * 2^e; the call is kda_verify_ring's on that checkpoint,
   except that a fold requantizes the folded state row by row by this
   header's rule (decided in fp32) instead of rounding it to bf16, writes
   codes and scales in place, and the call continues from their exact values.
   The kernel reads the checkpoint through the ring's bf16 product operand,
   exact for every row whose largest magnitude is at least 2^-108. p as for
   kda_verify_ring with p->state the E4M3 codes (16-byte aligned, slot stride
   a multiple of 16 when N > 1), r as for kda_verify_ring, f the scales.
   Errors as kda_verify_ring and kda_decode_fp8, plus KDA_EINVAL for codes not
   16-byte aligned. */
kda_status kda_verify_ring_fp8(const kda_params* p, int32_t T, const kda_ring_params* r, const kda_fp8_pool* f,
                               void* stream);

#ifdef __cplusplus
}
#endif

#endif /* KDA_GB300_KDA_FP8_H */
