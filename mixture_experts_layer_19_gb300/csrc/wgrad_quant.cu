// wgrad_quant.cu -- the block-scaled weight gradients' token operands: the
// sorted rows of X and dY (row r <- token perm_src[r] / k, padding rows zero),
// gathered, transposed and quantised along the sorted rows in one pass:
//   out[c, r] = Q(src[perm_src[r] / k, c]),  out [cols, A], scale atoms over
//   the cols rows with K = A (blocks of 32 rows for MXFP8, 16 for NVFP4 with
//   tensor scale 1).
// It replaces a bf16 gather of both tensors followed by two transposing
// quantisers.
//
// A tile is 128 sorted rows x 64 columns of both sources.  Tiles run column
// block by column block over the rows in use (totals[0]), so the grid sweeps
// one 64-column slice of X and dY at a time: a token's 128-byte segment is
// read from HBM once and its other k - 1 reads hit L2.  Four CTAs per SM;
// each thread looks up its own rows' tokens (a multiply-high by ceil(2^32/k)
// instead of a division where that is exact) and issues the loads of both
// sources before the tile's barrier.
// In shared memory a source's tile is 128 rows of 8 16-byte chunks, chunk c
// of row r stored at c ^ (r / 32 % 4): quantising thread i owns output row
// b0 + i / 4 and the 32 sorted rows 32 (i % 4) onwards, so the four threads
// of one column read four different chunks and a warp's reads are free of
// bank conflicts.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "mx.cuh"
#include "nv.cuh"

namespace moe {

namespace {

constexpr int kGtTile = 128 * 64;                                         // bf16 per source
constexpr int kGtSmem = 2 * kGtTile * (int)sizeof(__nv_bfloat16);   // 32 KB: one tile of each source

// element offset of (row r, column c) in a swizzled source tile
__device__ __forceinline__ int gt_off(int r, int c) { return r * 64 + ((((c >> 3) ^ (r >> 5)) & 7) << 3) + (c & 7); }

template <bool NV>
__device__ __forceinline__ void gt_quant_store(const __nv_bfloat16* tile, int tid, int a0, int b0, int A,
                                               float rc1, uint8_t* __restrict__ q, uint8_t* __restrict__ sf) {
  const int b = tid >> 2, j = tid & 3;
  float v[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) v[m] = __bfloat162float(tile[gt_off(32 * j + m, b)]);
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
}

}  // namespace

// kmag = ceil(2^32 / k) when every row index n satisfies n k < 2^32 (then
// n / k = umulhi(n, kmag) exactly), else 0 (plain division)
template <bool NV>
__global__ void __launch_bounds__(256) gather_transpose_q_kernel(
    const __nv_bfloat16* __restrict__ X0, const __nv_bfloat16* __restrict__ X1, const int32_t* __restrict__ perm_src,
    const int32_t* __restrict__ totals, int k, uint32_t kmag, int A, int B, uint8_t* __restrict__ q0,
    uint8_t* __restrict__ sf0, uint8_t* __restrict__ q1, uint8_t* __restrict__ sf1) {
  extern __shared__ __align__(16) unsigned char gt_smem[];
  __nv_bfloat16* tile = reinterpret_cast<__nv_bfloat16*>(gt_smem);
  const int rows_used = min(__ldg(totals), A);
  const int na = min((rows_used + 127) / 128, A / 128), nb = B / 64;
  if (na == 0) return;
  const int tid = threadIdx.x;
  const int piece = tid & 7;
  const float rc1 = nv_rc(1.0f);
  // tile (column block bb, row block ab), stepped by gridDim.x tiles at a time
  const int G = (int)gridDim.x, ga = G % na, gb = G / na;
  int ab = (int)blockIdx.x % na, bb = (int)blockIdx.x / na;
  for (; bb < nb;) {
    const int b0 = bb * 64, a0 = ab * 128;
    int tok[4];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int r = a0 + pass * 32 + (tid >> 3);
      const int src = r < rows_used ? __ldg(perm_src + r) : -1;
      tok[pass] = src < 0 ? -1 : kmag ? (int)__umulhi((uint32_t)src, kmag) : src / k;
    }
    uint4 v0[4], v1[4];
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      v0[pass] = make_uint4(0, 0, 0, 0);
      v1[pass] = make_uint4(0, 0, 0, 0);
      if (tok[pass] >= 0) {
        const int64_t off = (int64_t)tok[pass] * B + b0;
        v0[pass] = __ldg(reinterpret_cast<const uint4*>(X0 + off) + piece);
        v1[pass] = __ldg(reinterpret_cast<const uint4*>(X1 + off) + piece);
      }
    }
#pragma unroll
    for (int pass = 0; pass < 4; ++pass) {
      const int o = gt_off(pass * 32 + (tid >> 3), piece * 8);
      *reinterpret_cast<uint4*>(tile + o) = v0[pass];
      *reinterpret_cast<uint4*>(tile + kGtTile + o) = v1[pass];
    }
    __syncthreads();
    gt_quant_store<NV>(tile, tid, a0, b0, A, rc1, q0, sf0);
    gt_quant_store<NV>(tile + kGtTile, tid, a0, b0, A, rc1, q1, sf1);
    __syncthreads();
    ab += ga;
    bb += gb;
    if (ab >= na) {
      ab -= na;
      ++bb;
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
  const uint32_t kmag = (k > 1 && (uint64_t)A * (uint64_t)k <= (1ull << 32))
                            ? (uint32_t)(((1ull << 32) + (uint64_t)k - 1) / (uint64_t)k)
                            : 0u;
  auto kern = nv ? gather_transpose_q_kernel<true> : gather_transpose_q_kernel<false>;
  kern<<<grid, 256, kGtSmem, st>>>(x0, x1, perm_src, totals, k, kmag, A, B, o0, s0, o1, s1);
  return cudaGetLastError();
}

__global__ void __launch_bounds__(256) widen_bf16_kernel(const __nv_bfloat16* __restrict__ src, float* __restrict__ dst,
                                                         int64_t n) {
  for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < n; i += (int64_t)gridDim.x * blockDim.x)
    dst[i] = __bfloat162float(src[i]);
}

cudaError_t launch_widen_bf16(const void* src, float* dst, int64_t n, int grid, cudaStream_t st) {
  widen_bf16_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const __nv_bfloat16*>(src), dst, n);
  return cudaGetLastError();
}

cudaError_t prepare_gather_transpose_q(bool nv) {
  return cudaFuncSetAttribute(nv ? gather_transpose_q_kernel<true> : gather_transpose_q_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kGtSmem);
}

}  // namespace moe
