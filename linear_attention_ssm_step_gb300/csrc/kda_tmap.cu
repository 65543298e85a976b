// kda_tmap.cu - tensor maps of the state pool, for tensor-map (TMA) copies.
// Host code: the encoder comes from the driver through the runtime's entry
// point query, so the library links no driver library of its own.
#include <cuda.h>
#include <cuda_runtime.h>

#include "kda_device.cuh"
#include "kda_launch.h"

namespace kda {

typedef CUresult (*EncodeTiledFn)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                  const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_tiled() {
  static const EncodeTiledFn fn = [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess)
      return static_cast<EncodeTiledFn>(nullptr);
    return reinterpret_cast<EncodeTiledFn>(f);
  }();
  return fn;
}

// The state pool as a 3-D bf16 tensor {128 keys, H * 128 value rows, N slots}
// read and written in {64, 128, 1} boxes with the 128-byte swizzle. The last
// map is kept per host thread, keyed by pool address and shape.
cudaError_t state_tensor_map(const kda_params& p, CUtensorMap* out) {
  struct Cached {
    const void* ptr = nullptr;
    int N = 0, H = 0;
    int64_t stride = 0;
    CUtensorMap map;
  };
  thread_local Cached cache;
  const int64_t slot = p.N > 1 ? p.state_slot_stride : (int64_t)p.H * KD * KD;
  if (cache.ptr == p.state && cache.N == p.N && cache.H == p.H && cache.stride == slot) {
    *out = cache.map;
    return cudaSuccess;
  }
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)KD, (cuuint64_t)p.H * KD, (cuuint64_t)p.N};
  const cuuint64_t strides[2] = {(cuuint64_t)KD * 2, (cuuint64_t)slot * 2};
  const cuuint32_t box[3] = {64, 128, 1};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap map;
  const CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, p.state, dims, strides, box, estr,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cache.ptr = p.state;
  cache.N = p.N;
  cache.H = p.H;
  cache.stride = slot;
  cache.map = map;
  *out = map;
  return cudaSuccess;
}

// A token view (q, k, v or g_raw: bf16 rows of H heads x 128 values) as a 3-D
// tensor {128 values, H heads, rows} read in {128, 1, 16} boxes without
// swizzle: one box is 16 consecutive rows of one head, rows past the last
// reading as zeros. Needs every row 16-byte aligned. Four maps are kept per
// host thread, keyed by address, strides and shape.
cudaError_t token_tensor_map(const kda_view& v, int rows, int H, CUtensorMap* out) {
  struct Cached {
    const void* ptr = nullptr;
    int rows = 0, H = 0;
    int64_t b_stride = 0, h_stride = 0;
    CUtensorMap map;
  };
  thread_local Cached cache[4];
  thread_local int next = 0;
  for (const Cached& c : cache)
    if (c.ptr == v.ptr && c.rows == rows && c.H == H && c.b_stride == v.b_stride && c.h_stride == v.h_stride) {
      *out = c.map;
      return cudaSuccess;
    }
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[3] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)rows};
  const cuuint64_t strides[2] = {(cuuint64_t)v.h_stride * 2, (cuuint64_t)v.b_stride * 2};
  const cuuint32_t box[3] = {(cuuint32_t)KD, 1, 16};
  const cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap map;
  const CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(v.ptr), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Cached& c = cache[next];
  next = (next + 1) % 4;
  c.ptr = v.ptr;
  c.rows = rows;
  c.H = H;
  c.b_stride = v.b_stride;
  c.h_stride = v.h_stride;
  c.map = map;
  *out = map;
  return cudaSuccess;
}

// A T-token view (q, k, v or g_raw of a verify: bf16 [B][T][H][128]) as a
// 4-D tensor {128 values, H heads, T tokens, B rows} read in {128, 1, TT, 1}
// boxes without swizzle: one box is a row's TT token slots of one head, slots
// past T reading as zeros. Needs every row 16-byte aligned. Four maps are kept
// per host thread.
cudaError_t token_tensor_map_bt(const kda_view& v, int B, int T, int H, int TT, CUtensorMap* out) {
  struct Cached {
    const void* ptr = nullptr;
    int B = 0, T = 0, H = 0, TT = 0;
    int64_t b_stride = 0, t_stride = 0, h_stride = 0;
    CUtensorMap map;
  };
  thread_local Cached cache[4];
  thread_local int next = 0;
  for (const Cached& c : cache)
    if (c.ptr == v.ptr && c.B == B && c.T == T && c.H == H && c.TT == TT && c.b_stride == v.b_stride &&
        c.t_stride == v.t_stride && c.h_stride == v.h_stride) {
      *out = c.map;
      return cudaSuccess;
    }
  const EncodeTiledFn fn = encode_tiled();
  if (fn == nullptr) return cudaErrorNotSupported;
  const cuuint64_t dims[4] = {(cuuint64_t)KD, (cuuint64_t)H, (cuuint64_t)T, (cuuint64_t)B};
  const cuuint64_t strides[3] = {(cuuint64_t)v.h_stride * 2, (cuuint64_t)v.t_stride * 2, (cuuint64_t)v.b_stride * 2};
  const cuuint32_t box[4] = {(cuuint32_t)KD, 1, (cuuint32_t)TT, 1};
  const cuuint32_t estr[4] = {1, 1, 1, 1};
  CUtensorMap map;
  const CUresult r = fn(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(v.ptr), dims, strides, box,
                        estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  Cached& c = cache[next];
  next = (next + 1) % 4;
  c.ptr = v.ptr;
  c.B = B;
  c.T = T;
  c.H = H;
  c.TT = TT;
  c.b_stride = v.b_stride;
  c.t_stride = v.t_stride;
  c.h_stride = v.h_stride;
  c.map = map;
  *out = map;
  return cudaSuccess;
}

}  // namespace kda
