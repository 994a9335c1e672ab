// mxfp8.cuh -- MXFP8 block quantisation shared by the quantisers (mxfp8.cu)
// and the fused epilogue of the block-scaled dA GEMM (gemm_mx.cu): E4M3
// values, one UE8M0 power-of-two scale per 32 consecutive elements along a
// GEMM's K.
//
// Scale rule: the smallest power of two 2^X with amax / 2^X <= 448, so no
// element of a block saturates; X is clamped to [-127, 127] and stored as the
// E8M0 code X + 127; an all-zero block gets code 0.  Values are scaled by 2^-X
// (exact) and converted with CUDA's round-to-nearest-even, saturating E4M3
// conversion.  Scales are stored in 512-byte atoms of 128 rows x 128 K (the
// layout tcgen05.cp.32x128b.warpx4 copies into tensor memory), rows grouped
// by an SfLayout.
#pragma once

#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {

// E8M0 exponent of a block's scale from its non-negative amax (branch-free).
__device__ __forceinline__ int mx_scale_exp(float amax) {
  const uint32_t b = __float_as_uint(amax);
  const int eb = static_cast<int>((b >> 23) & 0xFF);
  // amax = m 2^(eb-127), m in [1,2); 448 = 1.75 2^8, so X = eb - 135, plus one when m > 1.75
  const int X = (eb - 135) + ((b & 0x7FFFFFu) > 0x600000u ? 1 : 0);
  // zero (and below 2^-126: far under the smallest E4M3 step of any scale) -> -127
  return eb == 0 ? -127 : max(-127, min(127, X));
}

__device__ __forceinline__ float pow2_neg(int X) {  // 2^-X for X in [-127, 126]
  return __uint_as_float(static_cast<uint32_t>(127 - X) << 23);
}

// (a s, b s) with one paired multiply (each lane rounded as a plain fp32 product;
// s is a power of two here, so the products are exact).
__device__ __forceinline__ float2 mul2(float a, float b, float s) {
  uint64_t x, y, r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(x) : "f"(a), "f"(b));
  asm("mov.b64 %0, {%1, %1};" : "=l"(y) : "f"(s));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(x), "l"(y));
  float2 o;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(r));
  return o;
}

// Paired fp32 arithmetic on (x, y) pairs, each lane rounded as the plain fp32
// operation (PTX .f32x2).
struct F2 {
  uint64_t r;
};
__device__ __forceinline__ F2 f2(float a, float b) {
  F2 o;
  asm("mov.b64 %0, {%1, %2};" : "=l"(o.r) : "f"(a), "f"(b));
  return o;
}
__device__ __forceinline__ float2 f2_get(F2 x) {
  float2 o;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(o.x), "=f"(o.y) : "l"(x.r));
  return o;
}
__device__ __forceinline__ F2 f2_mul(F2 a, F2 b) {
  F2 o;
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
  return o;
}
__device__ __forceinline__ F2 f2_sub(F2 a, F2 b) {
  F2 o;
  asm("sub.rn.f32x2 %0, %1, %2;" : "=l"(o.r) : "l"(a.r), "l"(b.r));
  return o;
}
__device__ __forceinline__ F2 f2_fma(F2 a, F2 b, F2 c) {
  F2 o;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(o.r) : "l"(a.r), "l"(b.r), "l"(c.r));
  return o;
}

// Four E4M3 codes of a s, b s, c s, d s, a's in the lowest byte.
__device__ __forceinline__ uint32_t pack_e4m3x4_scaled(float a, float b, float c, float d, float s) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(mul2(a, b, s), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(mul2(c, d, s), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// Quantise 32 values held in registers; writes 32 code bytes; returns the E8M0 code.
__device__ __forceinline__ uint8_t quant32(const float (&v)[32], uint4 *dst) {
  float m[8];  // eight independent max chains, then a tree
#pragma unroll
  for (int j = 0; j < 8; ++j) m[j] = fabsf(v[j]);
#pragma unroll
  for (int i = 8; i < 32; i += 8)
#pragma unroll
    for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(v[i + j]));
  const float amax = fmaxf(fmaxf(fmaxf(m[0], m[1]), fmaxf(m[2], m[3])),
                           fmaxf(fmaxf(m[4], m[5]), fmaxf(m[6], m[7])));
  const int X = mx_scale_exp(amax);
  const float s = pow2_neg(X);  // exact; an all-zero block stays zero
  uint32_t w[8];
#pragma unroll
  for (int q = 0; q < 8; ++q)
    w[q] = pack_e4m3x4_scaled(v[4 * q], v[4 * q + 1], v[4 * q + 2], v[4 * q + 3], s);
  dst[0] = make_uint4(w[0], w[1], w[2], w[3]);
  dst[1] = make_uint4(w[4], w[5], w[6], w[7]);
  return static_cast<uint8_t>(X + 127);
}

// Byte of (row r of segment sg, K block 0) in a scale-atom buffer of K columns
// whose rows are cut into segments of `seg` rows and groups of kGroup rows (a
// caller that knows the segment: no division by the segment length, and the
// group size's divisions become multiplications); K block kb of the same row
// adds atom_kblock(kb).
template <int kGroup>
__device__ __forceinline__ size_t atom_row_sg(int sg, int r, int K, int seg) {
  const int g = r / kGroup, rr = r - g * kGroup;
  constexpr int apg = (kGroup + 127) >> 7;
  const int gps = (seg + kGroup - 1) / kGroup;
  const size_t rb = (static_cast<size_t>(sg) * gps + g) * apg + (rr >> 7);
  const int w = rr & 127;
  return rb * (K >> 7) * 512 + (w & 31) * 16 + (w >> 5) * 4;
}
__device__ __forceinline__ size_t atom_kblock(int kblock) {
  return static_cast<size_t>(kblock >> 2) * 512 + (kblock & 3);
}

// Byte of (row, K block) in a scale-atom buffer of K columns grouped by L.
__device__ __forceinline__ size_t atom_byte(int row, int kblock, int K, SfLayout L) {
  const int sg = row / L.seg, r = row - sg * L.seg;
  const int g = r / L.group, rr = r - g * L.group;
  const int gps = (L.seg + L.group - 1) / L.group, apg = (L.group + 127) >> 7;
  const size_t rb = (static_cast<size_t>(sg) * gps + g) * apg + (rr >> 7);
  const int w = rr & 127;
  return (rb * (K >> 7) + (kblock >> 2)) * 512 + (w & 31) * 16 + (w >> 5) * 4 + (kblock & 3);
}

}  // namespace moe
