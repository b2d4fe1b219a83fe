// mx_quant.cu -- MXFP8 quantisers.
//
//  * quant_rows_kernel: a bf16 row-major [rows, K] matrix -> E4M3 [rows, K] +
//    scale atoms, blocks of 32 along K (the expert weights once per optimiser
//    step, and the public moe_mx_quantize utility).
//    The same kernel quantises the tokens (X) once per token for the ring
//    megakernel's movers.
//  * quant_scatter_rows_kernel: each token row quantised once (MXFP8, or
//    NVFP4 with tensor scale 1) and stored into its k sorted rows; padding
//    rows -> zero bytes and zero scales.
// Quantisers: one thread per 32-element block: 64 contiguous input bytes, 32
// output bytes.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "mx.cuh"
#include "nv.cuh"

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

// S4 / B1 block-scaled: each token row (X, or dY in the backward) quantised
// along d once and written straight into its k sorted rows -- the same bytes
// and scale words as quantising every routed row (activation quantisation
// inside the dispatch: kucoin page "Cursor's MoK réalise une amélioration des
// performances de 2,37x sur NVIDIA GB300 NVL72", section 02).  Thread i of the grid-wide
// sweep takes block i of the token-major order (token t, 32-value block kb):
// it loads the 32 bf16 values, encodes them (MXFP8: E4M3 + one E8M0 scale;
// NVFP4: E2M1 + two E4M3 scales, tensor scale 1) and stores the codes to row
// dest[t k + j] for every slot j; four (MXFP8) or two (NVFP4) neighbouring
// lanes pack their scale bytes into one 4-byte atom word first.  The padding
// rows (perm_src < 0) get zero codes and scales.  d % 256 == 0, so the lanes
// that pack one word always hold the same token.
template <bool NV>
__global__ void __launch_bounds__(256) quant_scatter_rows_kernel(const __nv_bfloat16* __restrict__ src,
                                                                 const int32_t* __restrict__ perm_src,
                                                                 const int32_t* __restrict__ dest,
                                                                 const int32_t* __restrict__ totals, int T, int k,
                                                                 int d, uint8_t* __restrict__ q,
                                                                 uint8_t* __restrict__ sf) {
  const int kb32 = d / 32;                      // 32-value blocks per row
  const int row_bytes = NV ? d / 2 : d;
  const int nblk = NV ? d / 16 : d / 32;        // scale blocks per row
  const int64_t total = (int64_t)T * kb32;
  const int lane = threadIdx.x & 31;
  const int64_t warps_total = (int64_t)gridDim.x * (blockDim.x >> 5);
  const float rc1 = nv_rc(1.0f);
  for (int64_t base = ((int64_t)blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5)) * 32; base < total;
       base += warps_total * 32) {
    const int64_t i = base + lane;
    const bool valid = i < total;
    const int t = valid ? (int)(i / kb32) : 0;
    const int kb = valid ? (int)(i - (int64_t)t * kb32) : 0;
    float v[32];
    if (valid) load_bf16x32_f(src + (size_t)t * d + kb * 32, v);
    else
#pragma unroll
      for (int m = 0; m < 32; ++m) v[m] = 0.0f;
    uint4 c0, c1;
    uint32_t sword;   // this lane's scale bytes, packed with its neighbours' below
    if constexpr (NV) {
      const uint32_t s2 = nv_encode32(v, rc1, 1.0f, c0);
      c1 = make_uint4(0, 0, 0, 0);
      const uint32_t o2 = __shfl_down_sync(0xffffffffu, s2, 1);
      sword = s2 | (o2 << 16);                  // valid in even lanes: blocks 2 kb .. 2 kb + 3
    } else {
      const int xe = mx_block_exponent(amax32(v));
      uint32_t o[8];
      mx_encode32(v, xe, o);
      c0 = make_uint4(o[0], o[1], o[2], o[3]);
      c1 = make_uint4(o[4], o[5], o[6], o[7]);
      uint32_t b = (uint32_t)(xe + 127);
      b |= __shfl_down_sync(0xffffffffu, b, 1) << 8;
      b |= __shfl_down_sync(0xffffffffu, b, 2) << 16;
      sword = b;                                // valid in lanes 4n: blocks kb .. kb + 3
    }
    const bool word_lane = NV ? (lane & 1) == 0 : (lane & 3) == 0;
    if (!valid) continue;
    for (int j = 0; j < k; ++j) {
      const int r = __ldg(dest + (size_t)t * k + j);
      uint8_t* dq = q + (size_t)r * row_bytes;
      if constexpr (NV) {
        *reinterpret_cast<uint4*>(dq + kb * 16) = c0;
        if (word_lane) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(r, 2 * kb, nblk)) = sword;
      } else {
        asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(dq + kb * 32), "r"(c0.x),
                     "r"(c0.y), "r"(c0.z), "r"(c0.w), "r"(c1.x), "r"(c1.y), "r"(c1.z), "r"(c1.w)
                     : "memory");
        if (word_lane) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(r, kb, nblk)) = sword;
      }
    }
  }
  // padding rows: zero codes and scales
  const int rows = totals[0];
  const int nvec = row_bytes / 16, nwords = nblk / 4;
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  for (int r = gw; r < rows; r += (int)warps_total) {
    if (__ldg(perm_src + r) >= 0) continue;
    uint4* dq = reinterpret_cast<uint4*>(q + (size_t)r * row_bytes);
    for (int x = lane; x < nvec; x += 32) dq[x] = make_uint4(0, 0, 0, 0);
    for (int w = lane; w < nwords; w += 32) *reinterpret_cast<uint32_t*>(sf + sf_atom_offset(r, 4 * w, nblk)) = 0u;
  }
}

cudaError_t launch_quant_scatter_rows(bool nv, const void* src, const int32_t* perm_src, const int32_t* dest,
                                      const int32_t* totals, int T, int k, int d, void* q, void* sf, int grid,
                                      cudaStream_t st) {
  auto kern = nv ? quant_scatter_rows_kernel<true> : quant_scatter_rows_kernel<false>;
  kern<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), perm_src, dest, totals, T, k, d,
                             reinterpret_cast<uint8_t*>(q), reinterpret_cast<uint8_t*>(sf));
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
