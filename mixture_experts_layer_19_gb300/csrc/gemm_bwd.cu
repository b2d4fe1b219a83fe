// gemm_bwd.cu -- backward expert GEMMs.  The pages state only that backward
// reverses the two communication steps (pull reverse-combine, push
// reverse-dispatch: kucoin page "Cursor's MoK réalise une amélioration des
// performances de 2,37x sur NVIDIA GB300 NVL72", section 02); the arithmetic
// is the calculus of the forward:
//   u  = dY Wd                      (epilogue: dh = w u, da, db, w h, <u, h>)
//   dx = da Wg + db Wu              (written per sorted row, reduced per token later)
//   dWd[e] = dY^T (w h), dWg[e] = da^T x, dWu[e] = db^T x   (K = the expert's rows)
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

cudaError_t launch_gemm_bwd(int kind, const GemmArgs& a, int grid, cudaStream_t st) {
  switch (kind) {
    case kBwdU: return launch_one<kBwdU>(a, grid, st);
    case kBwdX: return launch_one<kBwdX>(a, grid, st);
    case kWgradD: return launch_one<kWgradD>(a, grid, st);
    default: return launch_one<kWgradGU>(a, grid, st);
  }
}
cudaError_t prepare_gemm_bwd(int kind) {
  switch (kind) {
    case kBwdU: return prepare_one<kBwdU>();
    case kBwdX: return prepare_one<kBwdX>();
    case kWgradD: return prepare_one<kWgradD>();
    default: return prepare_one<kWgradGU>();
  }
}

}  // namespace moe
