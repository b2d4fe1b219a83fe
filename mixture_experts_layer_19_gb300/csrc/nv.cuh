// nv.cuh -- NVFP4 encoding on the device: E2M1 elements (OCP Microscaling
// Formats v1.0), one E4M3 scale per 16 elements along a GEMM's K, and an fp32
// scale for the whole tensor (NVIDIA's NVFP4).  The pages name NVFP4 kernels
// only (fluidifia page "Cursor ouvre MoK, un mégakernel qui accélère
// l'entraînement MoE", section "Quand la communication devient le vrai
// problème").
//
// Every step that decides a code is IEEE fp32 with round-to-nearest-even:
//   rc = 1 / (6 g)                      once per tensor (g = tensor scale)
//   s  = E4M3_satfinite(amax * rc)      per 16-element block
//   r  = 1 / (s g)                      per block; s == 0 gives zero codes
//   code = E2M1_satfinite(v * r)        per element, sign kept (-0 is code 8)
// Weights: g = amax(tensor) / 2688 (2688 = 6 * 448); activations: g = 1.
//
// Packing: element 2i in the low nibble of byte i.  Scale atoms: the MXFP8
// atom layout (mx.cuh) with 16-element blocks, so one 512-byte atom covers
// 128 rows x 64 elements of K, which is one kind::mxf4nvf4 MMA's K.
#pragma once
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>
#include <stdint.h>

#include "mx.cuh"

namespace moe {

constexpr float kNvScaleDenom = 2688.0f;  // largest E2M1 (6) times largest E4M3 (448)

__device__ __forceinline__ float nv_rc(float g) { return __frcp_rn(__fmul_rn(6.0f, g)); }

__device__ __forceinline__ float e4m3_value(uint8_t s) {
  const __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)s, __NV_E4M3);
  return __half2float(__half(h));
}

// Quantise 16 floats (one block): returns the E4M3 scale byte and writes the
// 8 packed E2M1 bytes (little-endian) into out.
// amax: the block's largest magnitude, max over i of fabsf(v[i]) (fmaxf
// order, NaN ignored), computed by the caller.
__device__ __forceinline__ uint8_t nv_encode16_amax(const float* v, float amax, float rc, float g, uint2& out) {
  const uint8_t s = (uint8_t)__nv_cvt_float_to_fp8(__fmul_rn(amax, rc), __NV_SATFINITE, __NV_E4M3);
  const float sv = e4m3_value(s);
  if (sv == 0.0f) {
    out = make_uint2(0u, 0u);
    return s;
  }
  const float r = __frcp_rn(__fmul_rn(sv, g));
  uint32_t w[2] = {0u, 0u};
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const __nv_fp4x2_storage_t p = __nv_cvt_float2_to_fp4x2(
        make_float2(__fmul_rn(v[2 * i], r), __fmul_rn(v[2 * i + 1], r)), __NV_E2M1, cudaRoundNearest);
    w[i >> 2] |= (uint32_t)p << (8 * (i & 3));
  }
  out = make_uint2(w[0], w[1]);
  return s;
}

// The same with the block's amax taken here.
__device__ __forceinline__ uint8_t nv_encode16(const float* v, float rc, float g, uint2& out) {
  float amax = 0.0f;
#pragma unroll
  for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
  return nv_encode16_amax(v, amax, rc, g, out);
}

// 32 floats -> 16 packed bytes (two blocks); returns the two scale bytes
// (first block in the low byte).
__device__ __forceinline__ uint32_t nv_encode32(const float* v, float rc, float g, uint4& out) {
  uint2 lo, hi;
  const uint32_t s0 = nv_encode16(v, rc, g, lo);
  const uint32_t s1 = nv_encode16(v + 16, rc, g, hi);
  out = make_uint4(lo.x, lo.y, hi.x, hi.y);
  return s0 | (s1 << 8);
}

}  // namespace moe
