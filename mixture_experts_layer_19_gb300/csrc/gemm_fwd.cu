// gemm_fwd.cu -- forward expert GEMMs: [a|b] = Xg [Wg;Wu]^T with the SwiGLU
// epilogue h = silu(a) * b (kucoin page "Cursor's MoK réalise une
// amélioration des performances de 2,37x sur NVIDIA GB300 NVL72", section 02:
// SwiGLU runs inside the grouped-GEMM datapath), and y = h Wd^T whose
// epilogue writes each sorted row back (the push-combine residue, same page).
#include "gemm.cuh"
#include "kernels.h"

namespace moe {

template <int KIND>
static cudaError_t launch_one(const GemmArgs& a, int grid, cudaStream_t st) {
  gemm_kernel<KIND><<<grid, KindTraits<KIND>::threads, KindTraits<KIND>::smem_bytes, st>>>(a);
  return cudaGetLastError();
}
template <int KIND>
static cudaError_t prepare_one() {
  return cudaFuncSetAttribute(gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              KindTraits<KIND>::smem_bytes);
}

cudaError_t launch_gemm_fwd(int kind, const GemmArgs& a, int grid, cudaStream_t st) {
  return kind == kUp ? launch_one<kUp>(a, grid, st) : launch_one<kDown>(a, grid, st);
}
cudaError_t prepare_gemm_fwd(int kind) { return kind == kUp ? prepare_one<kUp>() : prepare_one<kDown>(); }

}  // namespace moe
