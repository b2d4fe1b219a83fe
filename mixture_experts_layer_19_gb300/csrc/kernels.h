// kernels.h -- internal launch interface between the C ABI (api.cu) and the
// kernels (routing.cu, gemm_*.cu).  Not part of the public ABI.
#pragma once
#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

constexpr int kTileRows = 128;  // expert segments are padded to this many sorted rows

// Device pointers of the routing state a forward writes into the caller's
// saved context (all int32 unless noted).
struct RoutingPtrs {
  int32_t* idx;        // [T*k] expert of each pair
  float* w;            // [T*k] gate weight of each pair (fp32)
  int32_t* dest;       // [T*k] padded sorted row of each pair
  int32_t* counts;     // [E]
  int32_t* offsets;    // [E+1] unpadded exclusive prefix of counts
  int32_t* poff;       // [E+1] padded segment starts
  int32_t* mtile_off;  // [E+1] prefix of 128-row tiles
  int32_t* totals;     // [4]: padded rows in use, routed pairs
  int32_t* perm_src;   // [R_pad] flat pair index of each padded sorted row, -1 = padding
};

int route_chunks(int T);
cudaError_t launch_router(const float* logits, int T, int E, int k, int32_t* chunk_hist, const RoutingPtrs& rp,
                          cudaStream_t st);
cudaError_t launch_scan(int T, int E, const int32_t* chunk_hist, int32_t* chunk_base, const RoutingPtrs& rp,
                        cudaStream_t st);
cudaError_t launch_permute(int T, int E, int k, const int32_t* chunk_base, const RoutingPtrs& rp, cudaStream_t st);
// Sorted rows G[r] = X[perm_src[r] / k] (X1 / G1 optional), written token by
// token through dest; padding rows (perm_src < 0) zeroed.
cudaError_t launch_gather(const void* X0, const void* X1, const int32_t* perm_src, const int32_t* dest,
                          const int32_t* totals, int T, int k, int d, void* G0, void* G1, int grid, cudaStream_t st);
cudaError_t launch_combine(const void* S, const int32_t* dest, const float* w, int T, int k, int d, void* Y,
                           int grid, cudaStream_t st);
cudaError_t launch_router_grad(const float* dgp, const int32_t* dest, const int32_t* idx, const float* w, int T,
                               int k, int E, int ntu, float* dg, float* dlogits, int grid, cudaStream_t st);
cudaError_t launch_unpad_routing(const RoutingPtrs& rp, int R, int32_t* perm_out, int32_t* dest_out,
                                 cudaStream_t st);

struct GemmArgs;
// kind: 0 up (+SwiGLU), 1 down (gemm_fwd.cu); 2 bwd-u (+SwiGLU backward), 3 bwd-x, 4 wgrad down,
// 5 wgrad gate/up (gemm_bwd.cu).  prepare_* raises the dynamic shared-memory limit.
cudaError_t launch_gemm_fwd(int kind, const GemmArgs& a, int grid, cudaStream_t st);
cudaError_t prepare_gemm_fwd(int kind);
cudaError_t launch_gemm_bwd(int kind, const GemmArgs& a, int grid, cudaStream_t st);
cudaError_t prepare_gemm_bwd(int kind);
// Expert parallelism over R virtual ranks on one GPU (ep.cu).  Cooperative
// launches of R * G CTAs; ctr holds 3R + 1 flags, zero between launches.
struct EpArgs {
  int R, G;                 // virtual ranks, CTAs per rank
  int T, d, F, E, k, ntu;   // shapes; ntu = <u, h> partials per pair
  int nch;                  // 64-token chunks
  RoutingPtrs rp;           // routing state (saved context)
  const float* logits;      // dispatch: router logits [T, E]
  int32_t* chunk_hist;      // dispatch: per-chunk expert counts
  int32_t* chunk_base;
  const uint4* X;           // token rows (dispatch / backward pull)
  const uint4* dY;          // backward pull: upstream gradient rows
  uint4* Xg;                // sorted rows pulled by the expert ranks
  uint4* dYg;
  const uint4* Ys;          // push: sorted result rows (y, or dx per pair)
  uint4* slot;              // push: home slots [T * k, d] bf16
  const float* dgp;         // push (backward): [sorted rows, ntu] partials, or null
  float* dgslot;            // push (backward): home copies [T * k, ntu]
  uint4* out;               // home output [T, d] bf16 (Y or dX)
  const float* w_out;       // combine weights (forward) or null (dX: plain sum)
  float* dg;                // backward: [T, k]
  float* dlogits;           // backward: [T, E] or null
  int* ctr;
  int32_t* status;
  uint64_t timeout_ns;
};
cudaError_t launch_ep_dispatch(const EpArgs& a, cudaStream_t st);
cudaError_t launch_ep_pull(const EpArgs& a, cudaStream_t st);
cudaError_t launch_ep_push(const EpArgs& a, cudaStream_t st);
cudaError_t prepare_ep();

// Router GEMM (gemm_router.cu): kind 6 logits, 7 dX += dlogits Wr, 8 dWr.
// out = sum over s < S of part[s] (n values each, n % 4 == 0), in split order,
// into out_f32 or (out_f32 null) rounded once into bf16 out_bf16.
cudaError_t launch_split_sum(const float* part, int S, int64_t n, float* out_f32, void* out_bf16, int grid,
                             cudaStream_t st);
cudaError_t launch_gemm_router(int kind, const GemmArgs& a, int grid, cudaStream_t st);
cudaError_t prepare_gemm_router();
cudaError_t launch_to_bf16(const float* src, void* dst, int64_t n, int grid, cudaStream_t st);

// MXFP8 (mx_quant.cu, gemm_mx.cu)
cudaError_t launch_quant_rows(const void* src, int64_t rows, int K, void* q, void* sf, int grid, cudaStream_t st);
cudaError_t launch_quant_transpose(const void* src, int E, int A, int B, void* q, void* sf, int grid,
                                   cudaStream_t st);
// Block-scaled weight gradients (wgrad_quant.cu): the sorted rows of two
// token tensors, transposed and quantised along the sorted rows (A = row
// capacity, B = columns): out[c, r] = Q(src[perm_src[r] / k, c]).  Waits
// are bounded by timeout_ns (kStatusTimeout into status); stall != 0 (test
// hook) keeps the producer warps from copying anything; grid: two CTAs per SM.
cudaError_t launch_gather_transpose_q(bool nv, const void* X0, const void* X1, const int32_t* perm_src,
                                      const int32_t* totals, int k, int A, int B, void* q0, void* sf0, void* q1,
                                      void* sf1, int32_t* status, uint64_t timeout_ns, int stall, int grid,
                                      cudaStream_t st);
cudaError_t prepare_gather_transpose_q(bool nv);   // its dynamic shared memory size, once
// dst[i] = src[i] widened from bf16, i < n (debug dumps).
cudaError_t launch_widen_bf16(const void* src, float* dst, int64_t n, int grid, cudaStream_t st);
// Sorted rows <- token-quantised rows (E4M3 or packed E2M1 bytes, row_bytes
// per row, and nblk scale bytes per row in the atom layout).
// Block-scaled sorted rows straight from the bf16 token rows: each token
// quantised along d once (MXFP8, or NVFP4 with tensor scale 1) and written to
// its k sorted rows through dest; padding rows (perm_src < 0) zeroed.
cudaError_t launch_quant_scatter_rows(bool nv, const void* src, const int32_t* perm_src, const int32_t* dest,
                                      const int32_t* totals, int T, int k, int d, void* q, void* sf, int grid,
                                      cudaStream_t st);
struct MxArgs;
// kind 0 up, 1 down, 2 bwd-u, 3 bwd-x, 4 wgrad down, 5 wgrad gate/up (K = each
// expert's tokens, transposed operands quantised along the tokens); nv: the
// NVFP4 variant (E2M1 operands,
// E4M3 scales per 16, tensor scales in MxArgs::tsB)
cudaError_t launch_gemm_mx(int kind, const MxArgs& a, int grid, cudaStream_t st, bool nv = false);
cudaError_t prepare_gemm_mx(int kind, bool nv = false);

// NVFP4 (nv_quant.cu): g = amax(a, b) / 2688 written to the device float *g
cudaError_t launch_nv_tensor_scale(const void* a, int64_t na, const void* b, int64_t nb, float* g, int grid,
                                   cudaStream_t st);
cudaError_t launch_nv_quant_rows(const void* src, int64_t rows, int K, const float* g, void* q, void* sf, int grid,
                                 cudaStream_t st);
cudaError_t launch_nv_quant_transpose(const void* src, int E, int A, int B, const float* g, void* q, void* sf,
                                      int grid, cudaStream_t st);

// Ring-buffer forward megakernel (megakernel.cu)
struct MegaArgs;
cudaError_t launch_plan_minibatches(const int32_t* mtile_off, int E, int mbt, int cap, int nt1, int nt2,
                                    int counters_len, int* counters, int32_t* mb_start, int32_t* phase_start,
                                    int32_t* n_mb, cudaStream_t st);
cudaError_t launch_fwd_megakernel(const MegaArgs& a, int grid, bool fused, cudaStream_t st);  // fused: one-launch forward
cudaError_t prepare_fwd_megakernel();
// Backward megakernel (megakernel_bwd.cu): B1-B4 and B6 of the BF16 layer in
// one cooperative launch over the saved layout (grid = one CTA per SM).
struct BwdMegaArgs;
cudaError_t launch_bwd_megakernel(const BwdMegaArgs& a, int grid, cudaStream_t st);
cudaError_t prepare_bwd_megakernel();
struct MegaMxArgs;
cudaError_t launch_fwd_megakernel_mx(const MegaMxArgs& a, int grid, bool fused, cudaStream_t st);  // fused: one launch
cudaError_t prepare_fwd_megakernel_mx();

// Record the detail string moe_last_error() returns on this thread.
void set_error_detail(const char* msg);

}  // namespace moe
