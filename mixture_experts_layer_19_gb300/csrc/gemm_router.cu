// gemm_router.cu -- the router GEMM in front of the layer and its backward.
//
// The pages have the router re-decide each token's experts at every step
// (kucoin page "Cursor's MoK réalise une amélioration des performances de
// 2,37x sur NVIDIA GB300 NVL72", section 01) and print no router; the plain
// reading is a linear map logits = X Wr^T (Wr [E, d], no bias).  Its
// backward adds dlogits Wr into dX and writes dWr = dlogits^T X.  All three
// run on the tcgen05 GEMM of gemm.cuh (one CTA per tile), with dlogits
// rounded to bf16 for the tensor cores.
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
