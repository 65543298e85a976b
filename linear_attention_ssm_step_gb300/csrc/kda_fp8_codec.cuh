// kda_fp8_codec.cuh - the fp8 (E4M3) state pool's conversions, shared by the
// kernels that read or write it (kda_fp8.cu, kda_ring.cu). The format is the
// library's reading of the decode page's fp8 headroom (include/kda_fp8.h):
// E4M3 codes, one power-of-two fp32 scale per state row, requantization
// decided in fp32 (m = the row's largest magnitude, e = the smallest integer
// with m 2^-e <= 448, codes = round-to-nearest-even of s 2^-e).
#pragma once

#include <cuda_fp16.h>

#include "kda_device.cuh"

namespace kda {

// Two E4M3 codes (low byte first) -> their exact values as an fp32 pair.
__device__ __forceinline__ f32x2 e4m3x2_to_f32x2(uint32_t two) {
  uint32_t h2;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"(static_cast<unsigned short>(two & 0xffffu)));
  const float2 f = __half22float2(*reinterpret_cast<const __half2*>(&h2));
  return pk2(f.x, f.y);
}

// An fp32 pair -> two E4M3 codes (low byte = low value), round to nearest
// even, saturating at 448.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(f32x2 v) {
  float lo, hi;
  upk2(v, lo, hi);
  unsigned short r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^e as an fp32 value, exactly, for -149 <= e <= 127.
__device__ __forceinline__ float pow2f(int e) {
  return e >= -126 ? __uint_as_float((uint32_t)(e + 127) << 23) : __uint_as_float(1u << (e + 149));
}

// The smallest integer e with m 2^-e <= 448 for m >= 0 (fp32 bits): with
// m = M 2^E, 1 <= M < 2 and 448 = 1.75 2^8, e = E - 8 when M <= 1.75 (the
// fraction field at most 0x600000), else E - 7; 0 for m = 0 and -134 below
// the normal range.
__device__ __forceinline__ int row_exponent(float m) {
  const uint32_t bits = __float_as_uint(m);
  if (bits == 0u) return 0;
  const int biased = (int)(bits >> 23);
  if (biased == 0) return -134;
  return biased - 127 - 8 + ((bits & 0x7fffffu) > 0x600000u ? 1 : 0);
}

}  // namespace kda
