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

// 32 bf16 values (64 contiguous bytes) widened to fp32.
__device__ __forceinline__ void load_bf16x32_f(const __nv_bfloat16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 q = __ldg(s + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
      v[8 * c + 2 * i] = f.x;
      v[8 * c + 2 * i + 1] = f.y;
    }
  }
}

// One 32-element block: E4M3 bytes to q, its E8M0 scale byte to *sfp.
__device__ __forceinline__ void quant_block_store(const float* v, uint8_t* q, uint8_t* sfp) {
  const int X = mx_block_exponent(amax32(v));
  uint32_t o[8];
  mx_encode32(v, X, o);
  uint4* dq = reinterpret_cast<uint4*>(q);
  dq[0] = make_uint4(o[0], o[1], o[2], o[3]);
  dq[1] = make_uint4(o[4], o[5], o[6], o[7]);
  *sfp = (uint8_t)(X + 127);
}

}  // namespace moe
