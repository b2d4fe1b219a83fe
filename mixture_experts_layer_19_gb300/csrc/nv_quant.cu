// nv_quant.cu -- NVFP4 quantisers (encoding rules in nv.cuh).
//
//  * amax_kernel / tensor_scale_kernel: the tensor scale g = amax / 2688 of
//    one or two bf16 tensors (the weights, once per optimiser step; Wg and Wu
//    share one scale), 1 for an all-zero tensor;
//  * nv_quant_rows_kernel: a bf16 row-major [rows, K] matrix -> packed E2M1
//    [rows, K / 2] + scale atoms, blocks of 16 along K;
//    (the tokens, X or dY, use tensor scale 1 and are quantised straight
//    into their sorted rows by quant_scatter_rows_kernel in mx_quant.cu);
//  * nv_quant_transpose_kernel: a weight's backward orientation, quantised
//    along its other axis.
// One thread per 32 elements: 64 input bytes, 16 output bytes, 2 scale bytes.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "nv.cuh"

namespace moe {

namespace {

__device__ __forceinline__ void load32_bf16(const __nv_bfloat16* src, float* v) {
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

// Encode 32 values at element column c0 (a multiple of 32) of row r.
__device__ __forceinline__ void nv_store32(const float* v, float rc, float g, uint8_t* q_row, uint8_t* sf,
                                           int64_t r, int c0, int kblocks) {
  uint4 o;
  const uint32_t s2 = nv_encode32(v, rc, g, o);
  *reinterpret_cast<uint4*>(q_row + c0 / 2) = o;
  *reinterpret_cast<uint16_t*>(sf + sf_atom_offset(r, c0 / 16, kblocks)) = (uint16_t)s2;
}

}  // namespace

// Largest |x| over bf16 tensors, as the bit pattern of a non-negative float
// (whose integer order is its value order), via atomicMax.
__global__ void __launch_bounds__(256) amax_kernel(const __nv_bfloat16* __restrict__ a, int64_t na,
                                                   const __nv_bfloat16* __restrict__ b, int64_t nb,
                                                   unsigned int* __restrict__ out) {
  float m = 0.0f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  for (int pass = 0; pass < 2; ++pass) {
    const __nv_bfloat16* x = pass == 0 ? a : b;
    const int64_t n = pass == 0 ? na : nb;
    if (!x) continue;
    const int64_t nv = n / 8;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nv; i += stride) {
      const uint4 q = __ldg(reinterpret_cast<const uint4*>(x) + i);
      const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[j]));
        m = fmaxf(m, fmaxf(fabsf(f.x), fabsf(f.y)));
      }
    }
    for (int64_t i = nv * 8 + blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += stride)
      m = fmaxf(m, fabsf(__bfloat162float(x[i])));
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  __shared__ float red[8];
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    float t = 0.0f;
    for (int w = 0; w < (int)(blockDim.x >> 5); ++w) t = fmaxf(t, red[w]);
    atomicMax(out, __float_as_uint(t));
  }
}

__global__ void tensor_scale_kernel(float* g) {
  const float amax = __uint_as_float(*reinterpret_cast<unsigned int*>(g));
  *g = amax > 0.0f ? __fdiv_rn(amax, kNvScaleDenom) : 1.0f;
}

__global__ void __launch_bounds__(256) nv_quant_rows_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows,
                                                            int K, const float* __restrict__ gp,
                                                            uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const float g = gp ? __ldg(gp) : 1.0f;
  const float rc = nv_rc(g);
  const int chunks = K >> 5;
  const int64_t total = rows * chunks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / chunks;
    const int c0 = (int)(i - r * chunks) * 32;
    float v[32];
    load32_bf16(src + r * K + c0, v);
    nv_store32(v, rc, g, q + r * (K / 2), sf, r, c0, K / 16);
  }
}

// src [E][A][B] bf16 -> q [E][B][A / 2] packed E2M1 quantised along A, scale
// atoms over rows E * B with K = A.  One CTA transposes a 128 (A) x 64 (B)
// tile through shared memory (the skewed layout of the MXFP8 transposer:
// row stride 88, columns shifted by 8 per 32-row block); thread i then owns
// output row b0 + i / 4 and the 32 A-elements 32 (i % 4) onwards.
__global__ void __launch_bounds__(256) nv_quant_transpose_kernel(const __nv_bfloat16* __restrict__ src, int E,
                                                                 int A, int B, const float* __restrict__ gp,
                                                                 uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  constexpr int kStride = 88;
  __shared__ __align__(16) __nv_bfloat16 tile[128 * kStride];
  const float g = gp ? __ldg(gp) : 1.0f;
  const float rc = nv_rc(g);
  const int na = A / 128, nb = B / 64;
  const int64_t ntiles = (int64_t)E * na * nb;
  const int tid = threadIdx.x;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int e = (int)(t / (na * nb));
    const int rem = (int)(t - (int64_t)e * na * nb);
    const int a0 = (rem / nb) * 128, b0 = (rem % nb) * 64;
    const int piece = tid & 7;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int r = pass * 32 + (tid >> 3);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + ((int64_t)e * A + a0 + r) * B + b0) + piece);
      *reinterpret_cast<uint4*>(tile + r * kStride + 8 * (r >> 5) + piece * 8) = v;
    }
    __syncthreads();
    const int b = tid >> 2, j = tid & 3;
    float v[32];
#pragma unroll
    for (int m = 0; m < 32; ++m) v[m] = __bfloat162float(tile[(32 * j + m) * kStride + 8 * j + b]);
    const int64_t orow = (int64_t)e * B + b0 + b;
    nv_store32(v, rc, g, q + orow * (A / 2), sf, orow, a0 + 32 * j, A / 16);
    __syncthreads();
  }
}

cudaError_t launch_nv_tensor_scale(const void* a, int64_t na, const void* b, int64_t nb, float* g, int grid,
                                   cudaStream_t st) {
  cudaError_t e = cudaMemsetAsync(g, 0, sizeof(float), st);
  if (e != cudaSuccess) return e;
  amax_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(a), na,
                                    reinterpret_cast<const __nv_bfloat16*>(b), nb,
                                    reinterpret_cast<unsigned int*>(g));
  e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  tensor_scale_kernel<<<1, 1, 0, st>>>(g);
  return cudaGetLastError();
}

cudaError_t launch_nv_quant_rows(const void* src, int64_t rows, int K, const float* g, void* q, void* sf, int grid,
                                 cudaStream_t st) {
  nv_quant_rows_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), rows, K, g,
                                             reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(sf));
  return cudaGetLastError();
}

cudaError_t launch_nv_quant_transpose(const void* src, int E, int A, int B, const float* g, void* q, void* sf,
                                      int grid, cudaStream_t st) {
  nv_quant_transpose_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), E, A, B, g,
                                                  reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(sf));
  return cudaGetLastError();
}

}  // namespace moe
