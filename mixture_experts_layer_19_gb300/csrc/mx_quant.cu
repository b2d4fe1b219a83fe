// mx_quant.cu -- MXFP8 quantisers.
//
//  * quant_rows_kernel: a bf16 row-major [rows, K] matrix -> E4M3 [rows, K] +
//    scale atoms, blocks of 32 along K (the expert weights once per optimiser
//    step, and the public moe_mx_quantize utility).
//    The same kernel quantises the tokens (X, or dY in the backward) once per
//    token for the dispatch (MXFP8 activation quantisation inside the
//    dispatch datapath: kucoin page "Cursor's MoK réalise une amélioration des
//    performances de 2,37x sur NVIDIA GB300 NVL72", section 02).
//  * gather_rows_q_kernel: sorted row r <- the quantised row of token
//    perm_src[r] / k, element bytes and scale words; padding rows -> zero
//    bytes and zero scales (MXFP8 and NVFP4 rows alike).
// Quantisers: one thread per 32-element block: 64 contiguous input bytes, 32
// output bytes.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "mx.cuh"

namespace moe {

__global__ void __launch_bounds__(256) quant_rows_kernel(const __nv_bfloat16* __restrict__ src, int64_t rows, int K,
                                                         uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const int kblocks = K >> 5;
  const int64_t total = rows * kblocks;
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < total; i += (int64_t)gridDim.x * blockDim.x) {
    const int64_t r = i / kblocks;
    const int kb = (int)(i - r * kblocks);
    float v[32];
    load_bf16x32_f(src + r * K + kb * 32, v);
    quant_block_store(v, q + r * K + kb * 32, sf + sf_atom_offset(r, kb, kblocks));
  }
}

// src [E][A][B] bf16 -> q [E][B][A] E4M3 quantised along A (the backward
// orientation of a weight: the K of the dgrad GEMMs), scale atoms over rows
// E*B with K = A.  One CTA transposes a 128 (A) x 64 (B) tile through shared
// memory; thread i then owns output row b0 + i/4, block i%4 (four threads
// write one 128-byte output row).
__global__ void __launch_bounds__(256) quant_transpose_kernel(const __nv_bfloat16* __restrict__ src, int E, int A,
                                                              int B, uint8_t* __restrict__ q,
                                                              uint8_t* __restrict__ sf) {
  // tile of 128 A-rows x 64 B-columns.  Loads: 8 threads per row, 16 bytes
  // each, so every row is read as one 128-byte line.  Row r is stored with
  // its columns shifted by 8 * (r / 32) (row stride 88 bf16), which makes the
  // column reads of one 32-row quantisation block bank-conflict-free.
  constexpr int kStride = 88;
  __shared__ __align__(16) __nv_bfloat16 tile[128 * kStride];
  const int na = A / 128, nb = B / 64;
  const int64_t ntiles = (int64_t)E * na * nb;
  const int tid = threadIdx.x;
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int e = (int)(t / (na * nb));
    const int rem = (int)(t - (int64_t)e * na * nb);
    const int a0 = (rem / nb) * 128, b0 = (rem % nb) * 64;
    const int piece = tid & 7;
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int r = pass * 32 + (tid >> 3);
      const uint4 v = __ldg(reinterpret_cast<const uint4*>(src + ((int64_t)e * A + a0 + r) * B + b0) + piece);
      *reinterpret_cast<uint4*>(tile + r * kStride + 8 * (r >> 5) + piece * 8) = v;
    }
    __syncthreads();
    // one thread per (output row b, 32-element block j along A)
    const int b = tid >> 2, j = tid & 3;
    float v[32];
#pragma unroll
    for (int m = 0; m < 32; ++m) v[m] = __bfloat162float(tile[(32 * j + m) * kStride + 8 * j + b]);
    const int64_t orow = (int64_t)e * B + b0 + b;
    quant_block_store(v, q + orow * A + a0 + 32 * j, sf + sf_atom_offset(orow, a0 / 32 + j, A / 32));
    __syncthreads();
  }
}

// Sorted row r <- the quantised row of token perm_src[r] / k: its
// row_bytes element bytes and its scale words (4 blocks = 4 bytes per atom
// word), from the token-quantised copy (one quantisation per token, made by
// quant_rows_kernel / nv_quant_rows_kernel) into the sorted rows' atoms;
// padding rows get zero bytes and zero scales.  Same bytes as quantising each
// routed row.  nblk = scale blocks per row (a multiple of 4).
__global__ void __launch_bounds__(256) gather_rows_q_kernel(const uint8_t* __restrict__ q_tok,
                                                            const uint8_t* __restrict__ sf_tok,
                                                            const int32_t* __restrict__ perm_src,
                                                            const int32_t* __restrict__ dest,
                                                            const int32_t* __restrict__ totals, int T, int k,
                                                            int row_bytes, int nblk, uint8_t* __restrict__ q,
                                                            uint8_t* __restrict__ sf) {
  // walked by token: work item (t, part) reads a quarter of token t's codes
  // and scale words once and writes them to the token's k sorted rows
  // dest[t k + j]; then the padding rows (perm_src < 0) are zeroed
  constexpr int kParts = 4;
  const int nvec = row_bytes / 16;
  const int nwords = nblk / 4;
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int item = gw; item < T * kParts; item += warps_total) {
    const int t = item / kParts, part = item - t * kParts;
    const int v0 = part * nvec / kParts, v1 = (part + 1) * nvec / kParts;
    const int w0 = part * nwords / kParts, w1 = (part + 1) * nwords / kParts;
    const int dl = lane < k ? __ldg(dest + (size_t)t * k + lane) : 0;
    const uint4* sq = reinterpret_cast<const uint4*>(q_tok + (size_t)t * row_bytes);
    // every lane runs the same trips (the shuffles take the whole warp)
    for (int i0 = v0; i0 < v1; i0 += 128) {
      const int i = i0 + lane;
      uint4 v[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i + 32 * u < v1) v[u] = __ldg(sq + i + 32 * u);
      for (int j = 0; j < k; ++j) {
        uint4* dq = reinterpret_cast<uint4*>(q + (size_t)__shfl_sync(0xffffffffu, dl, j) * row_bytes);
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i + 32 * u < v1) dq[i + 32 * u] = v[u];
      }
    }
    for (int w00 = w0; w00 < w1; w00 += 32) {
      const int w = w00 + lane;
      const uint32_t sw =
          w < w1 ? __ldg(reinterpret_cast<const uint32_t*>(sf_tok + sf_atom_offset(t, 4 * w, nblk))) : 0u;
      for (int j = 0; j < k; ++j) {
        const int r = __shfl_sync(0xffffffffu, dl, j);
        if (w < w1) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(r, 4 * w, nblk)) = sw;
      }
    }
  }
  const int rows = totals[0];
  for (int r = gw; r < rows; r += warps_total) {
    if (__ldg(perm_src + r) >= 0) continue;
    uint4* dq = reinterpret_cast<uint4*>(q + (size_t)r * row_bytes);
    for (int i = lane; i < nvec; i += 32) dq[i] = make_uint4(0, 0, 0, 0);
    for (int w = lane; w < nwords; w += 32) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(r, 4 * w, nblk)) = 0u;
  }
}

cudaError_t launch_gather_rows_q(const void* q_tok, const void* sf_tok, const int32_t* perm_src, const int32_t* dest,
                                 const int32_t* totals, int T, int k, int row_bytes, int nblk, void* q, void* sf,
                                 int grid, cudaStream_t st) {
  gather_rows_q_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint8_t*>(q_tok),
                                             reinterpret_cast<const uint8_t*>(sf_tok), perm_src, dest, totals, T, k,
                                             row_bytes, nblk, reinterpret_cast<uint8_t*>(q),
                                             reinterpret_cast<uint8_t*>(sf));
  return cudaGetLastError();
}

cudaError_t launch_quant_transpose(const void* src, int E, int A, int B, void* q, void* sf, int grid,
                                   cudaStream_t st) {
  quant_transpose_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), E, A, B,
                                               reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(sf));
  return cudaGetLastError();
}

cudaError_t launch_quant_rows(const void* src, int64_t rows, int K, void* q, void* sf, int grid, cudaStream_t st) {
  quant_rows_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), rows, K,
                                          reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(sf));
  return cudaGetLastError();
}


}  // namespace moe
