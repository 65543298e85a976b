// kda_chunk.cuh - building blocks shared by the kernels that process a chunk
// of tokens of one (row, head) at once with the tensor cores (the ring verify
// and the chunked prefill): block sums of per-channel products through
// per-warp transpose tiles, bf16 multi-part splits of fp32 operands, and the
// token inputs of a chunk held in registers (thread i = key channel i and
// value row i of a 128-thread CTA).
#pragma once

#include "kda_device.cuh"
#include "kda_tc.cuh"

namespace kda {

// Per-warp tile for summing 32 values over the warp's 32 lanes: row i holds
// value i of every lane, rows 36 floats apart (16-byte aligned, and each
// group of 8 lanes reading 16 bytes of 8 different rows hits 32 different
// banks).
constexpr int XPOSE_LD = 36;
constexpr uint32_t XPOSE_WARP_BYTES = 32u * XPOSE_LD * 4u;

__device__ __forceinline__ float round_bf16(float x) { return bf16_bits_to_float(float_to_bf16_bits(x)); }

__device__ __forceinline__ f32x2 add2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("add.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

__device__ __forceinline__ f32x2 sub2(f32x2 a, f32x2 b) {
  f32x2 d;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(d) : "l"(a), "l"(b));
  return d;
}

// Warp sums of per-lane values through a per-warp shared-memory tile: lane r
// puts its value i at row i, column r (the 32 lanes' stores of one value are
// one contiguous row), then lane l sums row l over the 32 lanes as a fixed
// pairwise tree on packed pairs. tile_put_* write the values; tile_row_sum
// (after a __syncwarp) returns the sum of value `row`.
__device__ __forceinline__ void tile_put(float* tile, int lane, int i, float x) { tile[i * XPOSE_LD + lane] = x; }

__device__ __forceinline__ void tile_put2(float* tile, int lane, int i, f32x2 x) {
  float lo, hi;
  upk2(x, lo, hi);
  tile[2 * i * XPOSE_LD + lane] = lo;
  tile[(2 * i + 1) * XPOSE_LD + lane] = hi;
}

__device__ __forceinline__ float tile_row_sum(const float* tile, int row) {
  const float4* r = reinterpret_cast<const float4*>(tile + row * XPOSE_LD);
  f32x2 s[16];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float4 f = r[q];
    s[2 * q] = pk2(f.x, f.y);
    s[2 * q + 1] = pk2(f.z, f.w);
  }
#pragma unroll
  for (int w = 1; w < 16; w <<= 1)
#pragma unroll
    for (int m = 0; m < 16; m += 2 * w) s[m] = add2(s[m], s[m + w]);
  float lo, hi;
  upk2(s[0], lo, hi);
  return __fadd_rn(lo, hi);
}

// The warp sum of value `lane` of 32 per-lane values.
__device__ __forceinline__ float warp_sum32(const float (&v)[32], float* tile, int lane) {
#pragma unroll
  for (int i = 0; i < 32; ++i) tile_put(tile, lane, i, v[i]);
  __syncwarp();
  const float s = tile_row_sum(tile, lane);
  __syncwarp();  // the tile is free again
  return s;
}

// The same for 32 values held as 16 packed pairs (value 2i low, 2i + 1 high).
__device__ __forceinline__ float warp_sum32(const f32x2 (&v)[16], float* tile, int lane) {
#pragma unroll
  for (int i = 0; i < 16; ++i) tile_put2(tile, lane, i, v[i]);
  __syncwarp();
  const float s = tile_row_sum(tile, lane);
  __syncwarp();
  return s;
}

// The block sum of value l of a 32-value chunk: its four warp partials in warp order.
__device__ __forceinline__ float block_sum(const float* part, int chunk, int l) {
  const float* q = part + chunk * 128 + l;
  return __fadd_rn(__fadd_rn(__fadd_rn(q[0], q[32]), q[64]), q[96]);
}

// x as bf16 hi + lo (hi = bf16(x), lo = bf16(x - hi); |x - hi - lo| <= 2^-17 |x|)
// at element (row, k) of the two B-operand halves.
// Column k of a K-major, 128-byte-swizzled operand of R rows (sw128_offset):
// the part of the offset that does not depend on the row, and the column's
// 16-byte chunk within its 128-byte row, formed once per column.
struct Sw128Col {
  uint32_t base, chunk;
};

__device__ __forceinline__ Sw128Col sw128_col(int R, int k) {
  return Sw128Col{(uint32_t)(k >> 6) * (uint32_t)R * 128u + ((uint32_t)(k & 7) << 1), (uint32_t)((k >> 3) & 7)};
}

// sw128_offset(R, r, k) for the column of `c`.
__device__ __forceinline__ uint32_t sw128_at(const Sw128Col& c, int r) {
  return c.base + (uint32_t)r * 128u + ((c.chunk ^ (uint32_t)(r & 7)) << 4);
}

// store_split at a precomputed offset.
__device__ __forceinline__ void store_split_at(unsigned char* hi, unsigned char* lo, uint32_t off, float x) {
  const uint16_t xh = float_to_bf16_bits(x);
  const uint16_t xl = float_to_bf16_bits(__fsub_rn(x, bf16_bits_to_float(xh)));
  *reinterpret_cast<uint16_t*>(hi + off) = xh;
  *reinterpret_cast<uint16_t*>(lo + off) = xl;
}

template <int NB>
__device__ __forceinline__ void store_split(unsigned char* hi, unsigned char* lo, int row, int k, float x) {
  const uint16_t xh = float_to_bf16_bits(x);
  const uint16_t xl = float_to_bf16_bits(__fsub_rn(x, bf16_bits_to_float(xh)));
  const uint32_t off = sw128_offset(NB, row, k);
  *reinterpret_cast<uint16_t*>(hi + off) = xh;
  *reinterpret_cast<uint16_t*>(lo + off) = xl;
}

// x as three bf16 parts (exact to 2^-25 |x|) at element (row, j) of three
// 32-byte-swizzled operands `part` bytes apart.
__device__ __forceinline__ void store_split3(unsigned char* base, uint32_t part, int row, int j, float x) {
  const uint16_t x0 = float_to_bf16_bits(x);
  const float r1 = __fsub_rn(x, bf16_bits_to_float(x0));
  const uint16_t x1 = float_to_bf16_bits(r1);
  const uint16_t x2 = float_to_bf16_bits(__fsub_rn(r1, bf16_bits_to_float(x1)));
  const uint32_t off = sw32_offset(128, row, j);
  *reinterpret_cast<uint16_t*>(base + off) = x0;
  *reinterpret_cast<uint16_t*>(base + part + off) = x1;
  *reinterpret_cast<uint16_t*>(base + 2 * part + off) = x2;
}

// Token inputs of one item in registers, as loaded (bf16 bits, converted
// where they are used, so that the loads all fly together): q, k, g of key
// channel tid and v of value row tid, for every token slot (zero past T).
template <int TT>
struct TokenRegs {
  uint16_t qv[TT], kv[TT], gv[TT], vv[TT];
  uint16_t blogit;
  float alog, dtb;  // A_log[h] and dt_bias[h][tid] (raw gate)
};

__device__ __forceinline__ uint16_t load_bits(const kda_view& vw, int b, int t, int h, int c) {
  const uint16_t* ptr = static_cast<const uint16_t*>(vw.ptr);
  return ptr[(int64_t)b * vw.b_stride + (int64_t)t * vw.t_stride + (int64_t)h * vw.h_stride + c];
}

// Slots t >= T are never loaded and keep the zeros set once by zero_tokens.
template <int TT>
__device__ __forceinline__ void zero_tokens(TokenRegs<TT>& L) {
#pragma unroll
  for (int t = 0; t < TT; ++t) L.qv[t] = L.kv[t] = L.gv[t] = L.vv[t] = 0;
  L.blogit = 0;
  L.alog = L.dtb = 0.0f;
}

// The addresses are formed once per tensor and stepped by t_stride, so that
// each load costs one add.
template <int TT>
__device__ __forceinline__ void load_tokens(const kda_params& p, int b, int h, int T, TokenRegs<TT>& L) {
  const int tid = threadIdx.x;
  const uint16_t* qb = static_cast<const uint16_t*>(p.q.ptr) + ((int64_t)b * p.q.b_stride + (int64_t)h * p.q.h_stride + tid);
  const uint16_t* kb = static_cast<const uint16_t*>(p.k.ptr) + ((int64_t)b * p.k.b_stride + (int64_t)h * p.k.h_stride + tid);
  const uint16_t* gb =
      static_cast<const uint16_t*>(p.g_raw.ptr) + ((int64_t)b * p.g_raw.b_stride + (int64_t)h * p.g_raw.h_stride + tid);
  const uint16_t* vb = static_cast<const uint16_t*>(p.v.ptr) + ((int64_t)b * p.v.b_stride + (int64_t)h * p.v.h_stride + tid);
#pragma unroll
  for (int t = 0; t < TT; ++t) {
    if (t < T) {
      L.qv[t] = *qb;
      L.kv[t] = *kb;
      L.gv[t] = *gb;
      L.vv[t] = *vb;
    }
    qb += p.q.t_stride;
    kb += p.k.t_stride;
    gb += p.g_raw.t_stride;
    vb += p.v.t_stride;
  }
  if (tid < T) L.blogit = load_bits(p.beta_logit, b, tid, h, 0);
  if (p.gate_mode == KDA_GATE_RAW) {
    L.alog = p.A_log[h];
    L.dtb = p.dt_bias[(int64_t)h * KD + tid];
  }
}

// The gate of the chunk kernels (ring verify, chunked prefill): the formulas
// of Gate with the fast exponential (__expf) and the approximate reciprocal.
// Their relative errors, a few 1e-7 (g to about 5 x 2^-22 absolute, so the
// decay exp(g) to about 2^-20 relative), stay inside the tolerances of G, the
// decays, u~ and the prefill state; the ring's history weights and fold keep
// the IEEE exponential.
__device__ __forceinline__ float rcp_approx(float x) {
  float r;
  asm("rcp.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
  return r;
}

struct FastGate {
  bool raw;
  float a_h, lower_bound;
  __device__ __forceinline__ FastGate(const kda_params& p, float alog) {
    raw = p.gate_mode == KDA_GATE_RAW;
    a_h = raw ? __expf(alog) : 0.0f;
    lower_bound = p.lower_bound;
  }
  __device__ __forceinline__ float g(float g_in, float dtb) const {
    if (!raw) return g_in;
    const float z = __fmul_rn(a_h, __fadd_rn(g_in, dtb));
    return __fmul_rn(lower_bound, rcp_approx(__fadd_rn(1.0f, __expf(-z))));
  }
  __device__ __forceinline__ float beta(float b_in) const {
    return raw ? rcp_approx(__fadd_rn(1.0f, __expf(-b_in))) : b_in;
  }
};

// 16 fp32 values x[0..15] (K = 0..15) of row `row` of a K-major operand with
// the 32-byte swizzle (sw32_offset, R = 128) as three bf16 parts `part` bytes
// apart: x0 = bf16(x), x1 = bf16(x - x0), x2 = bf16(x - x0 - x1) as
// store_split3 forms them, each part's row in two 16-byte stores.
__device__ __forceinline__ void store_row_split3(unsigned char* base, uint32_t part, int row, const float (&x)[16]) {
  uint32_t w0[8], w1[8], w2[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) {
    const float a = x[2 * q], b = x[2 * q + 1];
    w0[q] = pack_bf16x2(a, b);
    float a0, b0;
    unpack_bf16x2(w0[q], a0, b0);
    const float ra = __fsub_rn(a, a0), rb = __fsub_rn(b, b0);
    w1[q] = pack_bf16x2(ra, rb);
    float a1, b1;
    unpack_bf16x2(w1[q], a1, b1);
    w2[q] = pack_bf16x2(__fsub_rn(ra, a1), __fsub_rn(rb, b1));
  }
  const uint32_t sw = ((uint32_t)row >> 2) & 1u;
  const uint32_t o0 = (uint32_t)row * 32u + (sw << 4), o1 = (uint32_t)row * 32u + ((1u ^ sw) << 4);
  *reinterpret_cast<uint4*>(base + o0) = make_uint4(w0[0], w0[1], w0[2], w0[3]);
  *reinterpret_cast<uint4*>(base + o1) = make_uint4(w0[4], w0[5], w0[6], w0[7]);
  *reinterpret_cast<uint4*>(base + part + o0) = make_uint4(w1[0], w1[1], w1[2], w1[3]);
  *reinterpret_cast<uint4*>(base + part + o1) = make_uint4(w1[4], w1[5], w1[6], w1[7]);
  *reinterpret_cast<uint4*>(base + 2 * part + o0) = make_uint4(w2[0], w2[1], w2[2], w2[3]);
  *reinterpret_cast<uint4*>(base + 2 * part + o1) = make_uint4(w2[4], w2[5], w2[6], w2[7]);
}

}  // namespace kda
