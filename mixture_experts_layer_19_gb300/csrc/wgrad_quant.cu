// wgrad_quant.cu -- the block-scaled weight gradients' token operands: the
// sorted rows of X and dY (row r <- token perm_src[r] / k, padding rows zero),
// gathered, transposed and quantised along the sorted rows in one pass:
//   out[c, r] = Q(src[perm_src[r] / k, c]),  out [cols, A], scale atoms over
//   the cols rows with K = A (blocks of 32 rows for MXFP8, 16 for NVFP4 with
//   tensor scale 1).
// It replaces a bf16 gather of both tensors followed by two transposing
// quantisers.  One CTA takes a 128 (rows) x 64 (cols) tile of each source
// through shared memory (the skewed layout of the weight transposers: row
// stride 88, columns shifted by 8 per 32-row block); thread i then owns
// output row b0 + i / 4 and the 32 sorted rows 32 (i % 4) onwards.  Tiles at
// or past the rows in use (totals[0], a multiple of 128) are skipped.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "mx.cuh"
#include "nv.cuh"

namespace moe {

template <bool NV>
__global__ void __launch_bounds__(256) gather_transpose_q_kernel(
    const __nv_bfloat16* __restrict__ X0, const __nv_bfloat16* __restrict__ X1, const int32_t* __restrict__ perm_src,
    const int32_t* __restrict__ totals, int k, int A, int B, uint8_t* __restrict__ q0, uint8_t* __restrict__ sf0,
    uint8_t* __restrict__ q1, uint8_t* __restrict__ sf1) {
  constexpr int kStride = 88;
  __shared__ __align__(16) __nv_bfloat16 tile[128 * kStride];
  __shared__ int src_row[128];
  const int rows_used = __ldg(totals);
  const int na = A / 128, nb = B / 64;
  const int64_t ntiles = (int64_t)na * nb;
  const int tid = threadIdx.x;
  const float rc1 = nv_rc(1.0f);
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int a0 = (int)(t / nb) * 128, b0 = (int)(t % nb) * 64;
    if (a0 >= rows_used) continue;   // uniform per CTA
    if (tid < 128) {
      const int r = a0 + tid;
      const int src = r < rows_used ? __ldg(perm_src + r) : -1;
      src_row[tid] = src < 0 ? -1 : src / k;
    }
    __syncthreads();
    for (int which = 0; which < 2; ++which) {
      const __nv_bfloat16* X = which == 0 ? X0 : X1;
      uint8_t* q = which == 0 ? q0 : q1;
      uint8_t* sf = which == 0 ? sf0 : sf1;
      const int piece = tid & 7;
#pragma unroll
      for (int pass = 0; pass < 4; ++pass) {
        const int r = pass * 32 + (tid >> 3);
        const int tok = src_row[r];
        uint4 v = make_uint4(0, 0, 0, 0);
        if (tok >= 0) v = __ldg(reinterpret_cast<const uint4*>(X + (int64_t)tok * B + b0) + piece);
        *reinterpret_cast<uint4*>(tile + r * kStride + 8 * (r >> 5) + piece * 8) = v;
      }
      __syncthreads();
      const int b = tid >> 2, j = tid & 3;
      float v[32];
#pragma unroll
      for (int m = 0; m < 32; ++m) v[m] = __bfloat162float(tile[(32 * j + m) * kStride + 8 * j + b]);
      const int64_t orow = b0 + b;
      if constexpr (NV) {
        uint4 o;
        const uint32_t s2 = nv_encode32(v, rc1, 1.0f, o);
        *reinterpret_cast<uint4*>(q + orow * (A / 2) + (a0 + 32 * j) / 2) = o;
        *reinterpret_cast<uint16_t*>(sf + sf_atom_offset(orow, (a0 + 32 * j) / 16, A / 16)) = (uint16_t)s2;
      } else {
        const int xe = mx_block_exponent(amax32(v));
        uint32_t o[8];
        mx_encode32(v, xe, o);
        uint4* dq = reinterpret_cast<uint4*>(q + orow * A + a0 + 32 * j);
        dq[0] = make_uint4(o[0], o[1], o[2], o[3]);
        dq[1] = make_uint4(o[4], o[5], o[6], o[7]);
        sf[sf_atom_offset(orow, (a0 + 32 * j) / 32, A / 32)] = (uint8_t)(xe + 127);
      }
      __syncthreads();
    }
  }
}

cudaError_t launch_gather_transpose_q(bool nv, const void* X0, const void* X1, const int32_t* perm_src,
                                      const int32_t* totals, int k, int A, int B, void* q0, void* sf0, void* q1,
                                      void* sf1, int grid, cudaStream_t st) {
  auto x0 = reinterpret_cast<const __nv_bfloat16*>(X0);
  auto x1 = reinterpret_cast<const __nv_bfloat16*>(X1);
  auto o0 = reinterpret_cast<uint8_t*>(q0);
  auto s0 = reinterpret_cast<uint8_t*>(sf0);
  auto o1 = reinterpret_cast<uint8_t*>(q1);
  auto s1 = reinterpret_cast<uint8_t*>(sf1);
  if (nv)
    gather_transpose_q_kernel<true><<<grid, 256, 0, st>>>(x0, x1, perm_src, totals, k, A, B, o0, s0, o1, s1);
  else
    gather_transpose_q_kernel<false><<<grid, 256, 0, st>>>(x0, x1, perm_src, totals, k, A, B, o0, s0, o1, s1);
  return cudaGetLastError();
}

}  // namespace moe
