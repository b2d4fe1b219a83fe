// gemm_mx.cu -- launchers of the MXFP8 forward expert GEMMs (gemm_mx.cuh).
#include "gemm_mx.cuh"
#include "kernels.h"

namespace moe {

template <int KIND>
static cudaError_t launch_mx_one(const MxArgs& a, int grid, cudaStream_t st) {
  gemm_mx_kernel<KIND><<<grid, MxTraits<KIND>::threads, MxTraits<KIND>::smem_bytes, st>>>(a);
  return cudaGetLastError();
}
template <int KIND>
static cudaError_t prepare_mx_one() {
  return cudaFuncSetAttribute(gemm_mx_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MxTraits<KIND>::smem_bytes);
}

cudaError_t launch_gemm_mx(int kind, const MxArgs& a, int grid, cudaStream_t st) {
  return kind == kUp ? launch_mx_one<kUp>(a, grid, st) : launch_mx_one<kDown>(a, grid, st);
}
cudaError_t prepare_gemm_mx(int kind) { return kind == kUp ? prepare_mx_one<kUp>() : prepare_mx_one<kDown>(); }

}  // namespace moe
