// kda_launch.h - internal launchers behind the C ABI (not part of the public header).
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>

#include <atomic>

#include "kda.h"
#include "kda_fp8.h"

namespace kda {

// Raise a kernel's dynamic shared-memory limit on its first launch only, so
// that later calls (including calls made during CUDA-graph capture) make no
// attribute call. `done` must be a flag owned by that one kernel (a static
// local of the per-kernel launcher). A failed attempt is retried next launch.
template <typename Kernel>
cudaError_t set_smem_limit_once(Kernel kern, size_t bytes, std::atomic<bool>& done) {
  if (done.load(std::memory_order_acquire)) return cudaSuccess;
  const cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess) done.store(true, std::memory_order_release);
  return e;
}

// T-token step (T = 1 is decode). tile_v in {16, 32, 64, 128}; bulk selects
// the bulk-copy staging of the state (16-byte aligned pool) over plain loads.
cudaError_t launch_step(const kda_params& p, int T, int tile_v, bool bulk, cudaStream_t s);

// The state pool as a 3-D bf16 tensor map {128 keys, H * 128 value rows, N
// slots}, {64, 128, 1} boxes, 128-byte swizzle (the tensor core's K-major
// operand layout); needs a 16-byte aligned pool and slot stride.
cudaError_t state_tensor_map(const kda_params& p, CUtensorMap* out);
// A token view as {128 values, H heads, rows} in {128, 1, 16} boxes (kda_tmap.cu).
cudaError_t token_tensor_map(const kda_view& v, int rows, int H, CUtensorMap* out);
// A T-token view as {128 values, H heads, T tokens, B rows} in {128, 1, TT, 1} boxes (kda_tmap.cu).
cudaError_t token_tensor_map_bt(const kda_view& v, int B, int T, int H, int TT, CUtensorMap* out);

// T-token verify with the two dot products of every state row per token on
// the tensor cores; one CTA per (row, head). bulk as above.
cudaError_t launch_verify_tc(const kda_params& p, int T, bool bulk, cudaStream_t s);

// Ring-cache verify with replay and fold, one CTA per (row, head). bulk
// selects tensor-map copies of the checkpoint (16-byte aligned pool) over
// plain loads and stores.
cudaError_t launch_ring(const kda_params& p, int T, const kda_ring_params& r, bool bulk, cudaStream_t s);

// The same with the checkpoint in an fp8 pool (p.state: E4M3 codes; f8: row
// scales; plain loads and stores).
cudaError_t launch_ring_fp8(const kda_params& p, int T, const kda_ring_params& r, const kda_fp8_pool& f8,
                            cudaStream_t s);

// Bytes of one chunk image of the two-stage prefill (kda_prefill_chain.cu):
// the operands of one 16-token chunk of one head.
constexpr uint32_t kPrefillChunkImageBytes = 45568u;

// Chunk images a two-stage prefill of B token rows, num_seqs sequences and H
// heads may write: (ceil(B / 16) + num_seqs) * H.
long long prefill_chunk_images(int B, int num_seqs, int H);

// Workspace bytes of the two-stage prefill: the chunk images, then one ready
// flag (4 bytes) per image for the single-launch schedule, padded to 16.
size_t prefill_workspace_size(int B, int num_seqs, int H);

// q, k, v and g_raw rows 16-byte aligned (the preparation's vector copies).
bool prefill_rows_aligned16(const kda_params& p);

// The single-launch two-stage prefill (configuration 6): a cooperative grid of
// one CTA per SM, num_seqs * H chain CTAs (at most half the SMs, num_seqs <= 32)
// and preparation CTAs beside them; needs prefill_rows_aligned16.
cudaError_t launch_prefill_fused(const kda_params& p, const int32_t* cu, int num_seqs, void* ws, bool bulk,
                                 cudaStream_t s);

// Two-stage varlen prefill: the preparation kernel writes every chunk's image
// into `ws` (prefill_chunk_images(...) images, 16-byte aligned), then the
// chain kernel runs each (sequence, head) through its chunks. bulk as above.
cudaError_t launch_prefill_chain(const kda_params& p, const int32_t* cu, int num_seqs, void* ws, bool bulk,
                                 cudaStream_t s);

// The device address of the fixed workspace of kda_prefill_static on the
// current device (looked up on the first call per device).
cudaError_t prefill_static_workspace(void** ptr);

}  // namespace kda
