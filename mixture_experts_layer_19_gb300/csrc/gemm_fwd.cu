// gemm_fwd.cu -- forward expert GEMMs: [a|b] = Xg [Wg;Wu]^T with the SwiGLU
// epilogue h = silu(a) * b (kucoin page "Cursor's MoK réalise une
// amélioration des performances de 2,37x sur NVIDIA GB300 NVL72", section 02:
// SwiGLU runs inside the grouped-GEMM datapath), and y = h Wd^T whose
// epilogue writes each sorted row back (the push-combine residue, same page).
#include "gemm.cuh"
#include "kernels.h"

namespace moe {

cudaError_t launch_gemm_fwd(int kind, const GemmArgs& a, int grid, cudaStream_t st) {
  return kind == kUp ? gemm_launch<kUp>(a, grid, st) : gemm_launch<kDown>(a, grid, st);
}
cudaError_t prepare_gemm_fwd(int kind) { return kind == kUp ? gemm_prepare<kUp>() : gemm_prepare<kDown>(); }

}  // namespace moe
