// gemm_mx.cu -- launchers of the block-scaled expert GEMMs (gemm_mx.cuh):
// MXFP8 and NVFP4 variants of the up, down, bwd-u, bwd-x and weight-gradient
// kinds.
#include "gemm_mx.cuh"
#include "kernels.h"

namespace moe {

template <int KIND, bool NV>
static cudaError_t launch_mx_one(const MxArgs& a, int grid, cudaStream_t st) {
  gemm_mx_kernel<KIND, NV><<<grid, MxTraits<KIND, NV>::threads, MxTraits<KIND, NV>::smem_bytes, st>>>(a);
  return cudaGetLastError();
}
template <int KIND, bool NV>
static cudaError_t prepare_mx_one() {
  return cudaFuncSetAttribute(gemm_mx_kernel<KIND, NV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              MxTraits<KIND, NV>::smem_bytes);
}

template <bool NV>
static cudaError_t launch_kind(int kind, const MxArgs& a, int grid, cudaStream_t st) {
  switch (kind) {
    case kUp: return launch_mx_one<kUp, NV>(a, grid, st);
    case kDown: return launch_mx_one<kDown, NV>(a, grid, st);
    case kBwdU: return launch_mx_one<kBwdU, NV>(a, grid, st);
    case kWgradD: return launch_mx_one<kWgradD, NV>(a, grid, st);
    case kWgradGU: return launch_mx_one<kWgradGU, NV>(a, grid, st);
    default: return launch_mx_one<kBwdX, NV>(a, grid, st);
  }
}
template <bool NV>
static cudaError_t prepare_kind(int kind) {
  switch (kind) {
    case kUp: return prepare_mx_one<kUp, NV>();
    case kDown: return prepare_mx_one<kDown, NV>();
    case kBwdU: return prepare_mx_one<kBwdU, NV>();
    case kWgradD: return prepare_mx_one<kWgradD, NV>();
    case kWgradGU: return prepare_mx_one<kWgradGU, NV>();
    default: return prepare_mx_one<kBwdX, NV>();
  }
}

cudaError_t launch_gemm_mx(int kind, const MxArgs& a, int grid, cudaStream_t st, bool nv) {
  return nv ? launch_kind<true>(kind, a, grid, st) : launch_kind<false>(kind, a, grid, st);
}
cudaError_t prepare_gemm_mx(int kind, bool nv) { return nv ? prepare_kind<true>(kind) : prepare_kind<false>(kind); }

}  // namespace moe
