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
  switch (kind) {
    case kUp: return launch_mx_one<kUp>(a, grid, st);
    case kDown: return launch_mx_one<kDown>(a, grid, st);
    case kBwdU: return launch_mx_one<kBwdU>(a, grid, st);
    default: return launch_mx_one<kBwdX>(a, grid, st);
  }
}
cudaError_t prepare_gemm_mx(int kind) {
  switch (kind) {
    case kUp: return prepare_mx_one<kUp>();
    case kDown: return prepare_mx_one<kDown>();
    case kBwdU: return prepare_mx_one<kBwdU>();
    default: return prepare_mx_one<kBwdX>();
  }
}

}  // namespace moe
