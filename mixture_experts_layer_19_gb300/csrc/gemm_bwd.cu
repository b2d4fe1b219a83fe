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

cudaError_t launch_gemm_bwd(int kind, const GemmArgs& a, int grid, cudaStream_t st) {
  switch (kind) {
    case kBwdU: return gemm_launch<kBwdU>(a, grid, st);
    case kBwdX: return gemm_launch<kBwdX>(a, grid, st);
    case kWgradD: return gemm_launch<kWgradD>(a, grid, st);
    default: return gemm_launch<kWgradGU>(a, grid, st);
  }
}
cudaError_t prepare_gemm_bwd(int kind) {
  switch (kind) {
    case kBwdU: return gemm_prepare<kBwdU>();
    case kBwdX: return gemm_prepare<kBwdX>();
    case kWgradD: return gemm_prepare<kWgradD>();
    default: return gemm_prepare<kWgradGU>();
  }
}
}  // namespace moe
