// mx.cuh -- MXFP8 encoding on the device: E4M3 elements with one E8M0 scale
// per 32 elements along a GEMM's K (OCP Microscaling Formats v1.0; the pages
// name the format only: kucoin page "Cursor's MoK réalise une amélioration des
// performances de 2,37x sur NVIDIA GB300 NVL72", section 02).
//
// Scale exponent X = floor(log2(amax)) - 8 (8 = largest E4M3 exponent),
// clamped to [-127, 127]; an all-zero block (or one whose amax is below the
// smallest normal float) gets -127.  Scale byte = X + 127.  Elements are
// v * 2^-X rounded to nearest-even E4M3 with saturation at +-448 (the PTX
// cvt.rn.satfinite conversion); scaling by a power of two is exact.
//
// Scale-factor layout ("atoms"): for a K-major operand of R rows (R % 128 == 0)
// and K columns (K % 128 == 0), the scales of rows [128 i, 128 i + 128) and
// K blocks [4 j, 4 j + 4) form one 512-byte atom at index i * (K / 128) + j;
// inside it, row r and block b sit at byte (r % 32) * 16 + ((r / 32) % 4) * 4
// + b % 4.  This is the order tcgen05.cp 32x128b.warpx4 expects when it copies
// one atom into four TMEM columns for a block-scaled UMMA.
#pragma once
#include <cuda_bf16.h>
#include <cuda_fp8.h>
#include <stdint.h>

namespace moe {

__host__ __device__ __forceinline__ size_t sf_atom_offset(int64_t row, int kb, int kblocks) {
  const int64_t kgroups = kblocks >> 2;
  const int64_t atom = (row >> 7) * kgroups + (kb >> 2);
  return (size_t)atom * 512 + (size_t)(row & 31) * 16 + (size_t)((row >> 5) & 3) * 4 + (size_t)(kb & 3);
}

// E8M0 exponent X of a block whose absolute maximum is `amax` (finite, >= 0).
__device__ __forceinline__ int mx_block_exponent(float amax) {
  const int eb = (__float_as_int(amax) >> 23) & 0xFF;   // biased exponent; 0 for zero / subnormal
  if (eb == 0) return -127;
  const int x = eb - 127 - 8;
  return x < -127 ? -127 : x;                          // x <= 254-135 = 119: no upper clamp needed
}

// Quantise 32 floats with exponent X into 32 E4M3 bytes (little-endian order).
__device__ __forceinline__ void mx_encode32(const float* v, int X, uint32_t (&out)[8]) {
  const float inv = __int_as_float((127 - X) << 23);   // 2^-X, a normal float for X in [-127, 126]
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp8x2_storage_t lo = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i] * inv, v[4 * i + 1] * inv),
                                                             __NV_SATFINITE, __NV_E4M3);
    const __nv_fp8x2_storage_t hi = __nv_cvt_float2_to_fp8x2(make_float2(v[4 * i + 2] * inv, v[4 * i + 3] * inv),
                                                             __NV_SATFINITE, __NV_E4M3);
    out[i] = (uint32_t)lo | ((uint32_t)hi << 16);
  }
}

__device__ __forceinline__ float amax32(const float* v) {
  float m = 0.0f;
#pragma unroll
  for (int i = 0; i < 32; ++i) m = fmaxf(m, fabsf(v[i]));
  return m;
}

}  // namespace moe
