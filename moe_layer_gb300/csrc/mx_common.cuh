// Device helpers of the MX block format (E4M3 elements, E8M0 scales): the
// block scale rule X = 2^(floor(log2(amax)) - 8) and the tcgen05.cp scale
// block layout.  Shared by the quantization kernels and the GEMM epilogues.
#pragma once
#include <stdint.h>

#include "ptx.cuh"

namespace moe {

// floor(log2(a)) for a > 0 (fp32, normal or subnormal).
__device__ __forceinline__ int floor_log2(float a) {
  const uint32_t b = __float_as_uint(a);
  const int e = static_cast<int>((b >> 23) & 0xFF);
  if (e != 0) return e - 127;
  const uint32_t m = b & 0x7FFFFFu;  // subnormal: a = m * 2^-149
  return (31 - __clz(static_cast<int>(m))) - 149;
}

// Unbiased exponent of the block scale for a block maximum (-127 for an
// all-zero block); the E8M0 code is this plus 127.
__device__ __forceinline__ int mx_scale_exp(float amax) {
  if (!(amax > 0.f)) return -127;
  const int e = floor_log2(amax) - 8;
  return e < -127 ? -127 : (e > 127 ? 127 : e);
}

// Two values to two E4M3 codes (round to nearest even, saturating to +-448):
// `lo` in bits 0..7, `hi` in bits 8..15.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// 2^-e for a block exponent e in [-127, 119] (exact, built from its bits;
// a finite block maximum gives e <= 127 - 8).
__device__ __forceinline__ float mx_inv_scale(int e) {
  return __uint_as_float(static_cast<uint32_t>(127 - e) << 23);
}

// Quantizes 32 values with scale 2^e into 32 E4M3 bytes (two 16-byte words).
// v * 2^-e is exact in fp32 whenever its magnitude is at least 2^-126; below
// that the E4M3 code is zero either way.
__device__ __forceinline__ void quant32(const float* v, int e, uint4& lo, uint4& hi) {
  const float inv = mx_inv_scale(e);
  uint32_t w[8];
#pragma unroll
  for (int i = 0; i < 8; ++i)
    w[i] = e4m3x2(v[4 * i] * inv, v[4 * i + 1] * inv) | (e4m3x2(v[4 * i + 2] * inv, v[4 * i + 3] * inv) << 16);
  lo = make_uint4(w[0], w[1], w[2], w[3]);
  hi = make_uint4(w[4], w[5], w[6], w[7]);
}

// Quantizes 32 values in place of a row: writes the 32 codes to dst (32-byte
// aligned, one 256-bit store) and returns the E8M0 code of their block.
__device__ __forceinline__ uint32_t quant32_store(const float* v, uint8_t* dst) {
  float amax = 0.f;
#pragma unroll
  for (int i = 0; i < 32; ++i) amax = fmaxf(amax, fabsf(v[i]));
  const int e = mx_scale_exp(amax);
  uint4 lo, hi;
  quant32(v, e, lo, hi);
  st_global_v8(dst, lo, hi);
  return static_cast<uint32_t>(e + 127);
}

// Byte offset of the scale word (four 32-column blocks) of row `row` and
// 128-column group `kgroup` for an operand with rblocks = rows / 128.
__device__ __forceinline__ size_t sf_word_offset(int64_t row, int64_t kgroup, int64_t rblocks) {
  return static_cast<size_t>((kgroup * rblocks + row / 128) * 512 + 16 * (row % 32) +
                             4 * ((row % 128) / 32));
}
// Byte offset of the scale of (MN index mn, reduction index k) for an operand
// whose MN extent is rblocks * 128.
__device__ __forceinline__ size_t sf_byte_offset(int64_t mn, int64_t k, int64_t rblocks) {
  return sf_word_offset(mn, k / 128, rblocks) + static_cast<size_t>((k % 128) / 32);
}

}  // namespace moe
