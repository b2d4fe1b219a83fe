// gemm_router.cu -- the router GEMM in front of the layer and its backward.
//
// The pages have the router re-decide each token's experts at every step
// (kucoin page "Cursor's MoK réalise une amélioration des performances de
// 2,37x sur NVIDIA GB300 NVL72", section 01) and print no router; the plain
// reading is a linear map logits = X Wr^T (Wr [E, d], no bias).  Its
// backward adds dlogits Wr into dX and writes dWr = dlogits^T X.  All three
// run on the tcgen05 GEMM of gemm.cuh (one CTA per tile), with dlogits
// rounded to bf16 for the tensor cores.  The logits and dWr GEMMs have few
// output tiles (T/128 and E/128 x d/256), so their K range is split over
// enough tiles to fill the GPU; the fp32 partials are summed in split order
// by split_sum_kernel.
#include "gemm.cuh"
#include "kernels.h"

namespace moe {

__global__ void __launch_bounds__(256) to_bf16_kernel(const float* __restrict__ src, __nv_bfloat16* __restrict__ dst,
                                                      int64_t n) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __float2bfloat16_rn(src[i]);
}

cudaError_t launch_to_bf16(const float* src, void* dst, int64_t n, int grid, cudaStream_t st) {
  to_bf16_kernel<<<grid, 256, 0, st>>>(src, reinterpret_cast<__nv_bfloat16*>(dst), n);
  return cudaGetLastError();
}

// Split-K partial sums: out[i] = part[0][i] + part[1][i] + ... + part[S-1][i]
// in split order (fp32), as fp32 (logits) or rounded once to bf16 (dWr).
__global__ void __launch_bounds__(256) split_sum_kernel(const float4* __restrict__ part, int S, int64_t n4,
                                                        float4* __restrict__ out_f32, uint2* __restrict__ out_bf16) {
  for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < n4; i += (int64_t)gridDim.x * blockDim.x) {
    float4 a = part[i];
    for (int s = 1; s < S; ++s) {
      const float4 b = part[(size_t)s * n4 + i];
      a.x += b.x;
      a.y += b.y;
      a.z += b.z;
      a.w += b.w;
    }
    if (out_f32) out_f32[i] = a;
    else out_bf16[i] = make_uint2(pack_bf16(a.x, a.y), pack_bf16(a.z, a.w));
  }
}

cudaError_t launch_split_sum(const float* part, int S, int64_t n, float* out_f32, void* out_bf16, int grid,
                             cudaStream_t st) {
  split_sum_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const float4*>(part), S, n / 4,
                                         reinterpret_cast<float4*>(out_f32), reinterpret_cast<uint2*>(out_bf16));
  return cudaGetLastError();
}

cudaError_t launch_gemm_router(int kind, const GemmArgs& a, int grid, cudaStream_t st) {
  switch (kind) {
    case kRouter: return gemm_launch<kRouter>(a, grid, st);
    case kRouterDX: return gemm_launch<kRouterDX>(a, grid, st);
    default: return gemm_launch<kRouterDW>(a, grid, st);
  }
}

cudaError_t prepare_gemm_router() {
  cudaError_t e = gemm_prepare<kRouter>();
  if (e == cudaSuccess) e = gemm_prepare<kRouterDX>();
  if (e == cudaSuccess) e = gemm_prepare<kRouterDW>();
  return e;
}

}  // namespace moe
