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
// read from HBM once and its other k - 1 reads hit L2.
//
// Two CTAs per SM, each four producer warps and eight quantising warps
// around a ring of kGtStages tiles in shared memory:
// - producer warp p (warps 8..11) owns the tile's rows 32 p .. 32 p + 31.
//   Lane l looks up row 32 p + l's token (a multiply-high by ceil(2^32/k)
//   instead of a division where that is exact; the next tile's lookups are
//   issued before the wait for a free stage), then copies 16-byte piece l % 8
//   of rows 32 p + l / 8 + 4 q (q < 8) of both sources with cp.async,
//   zero-filled for padding rows; each lane's copies complete one arrival on
//   the stage's full barrier;
// - quantising warp w takes source w / 4 and the 16 columns 16 (w % 4)
//   onwards; its lane l the column pair 16 (w % 4) + 2 (l % 8) (two output
//   rows) and the 32 sorted rows 32 (l / 8) onwards.  It reads its 32 bf16
//   pairs, releases the stage, then quantises and stores.
// In a stage a source's tile is four 32-row blocks of 128-byte rows, each
// block followed by 32 bytes of padding: the four row blocks a warp reads
// at once sit 8 banks apart, so its 32 four-byte reads hit 32 banks, and the
// four lanes of one column pair store one 128-byte run of each output row.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "mx.cuh"
#include "nv.cuh"
#include "ptx.cuh"

namespace moe {

namespace {

constexpr int kGtRowBytes = 64 * 2;                        // 64 bf16 columns of one sorted row
constexpr int kGtBlockBytes = 32 * kGtRowBytes + 32;       // 32 rows, then 32 bytes of padding
constexpr int kGtSrcBytes = 4 * kGtBlockBytes;             // one source's 128 x 64 tile
constexpr int kGtStageBytes = 2 * kGtSrcBytes;
constexpr int kGtStages = 3;
constexpr int kGtQuantWarps = 8;
constexpr int kGtProdWarps = 4;
constexpr int kGtThreads = 32 * (kGtQuantWarps + kGtProdWarps);
constexpr int kGtSmem = kGtStages * kGtStageBytes + 2 * kGtStages * 8 + 16;   // ring, barriers, abort flag
static_assert(kGtBlockBytes % 16 == 0 && kGtStageBytes % 128 == 0, "bulk copies need 16-byte alignment");

// 16-byte asynchronous copy global -> shared through L2 only (cp.async.cg);
// src_bytes 0 writes 16 zero bytes (nothing is read).
__device__ __forceinline__ void cp_async_16(void* dst, const void* src, uint32_t src_bytes) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(smem_u32(dst)),
               "l"(reinterpret_cast<uint64_t>(src)), "r"(src_bytes)
               : "memory");
}
// The mbarrier receives one arrival once every cp.async this thread issued
// so far has landed (the arrival is counted in the barrier's init count).
__device__ __forceinline__ void cp_async_mbar_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void cp_async_wait_all() { asm volatile("cp.async.wait_all;" ::: "memory"); }

// byte offset of sorted row r (0..127) in a source tile
__device__ __forceinline__ uint32_t gt_row(int r) { return (r >> 5) * kGtBlockBytes + (r & 31) * kGtRowBytes; }

// One 32-value block along the sorted rows of output row orow: the bf16
// words w[m] hold it in their low (h = 0) or high (h = 1) halves; amax is its
// largest magnitude (amax16[2] those of its two 16-value halves for NVFP4).
// Quantised into q / sf (the layout of moe_mx_quantize / moe_nv_quantize,
// K = A).
template <bool NV>
__device__ __forceinline__ void gt_quant_block(const uint32_t* w, int h, float amax, const float* amax16,
                                               int64_t orow, int a, int A, float rc1, uint8_t* __restrict__ q,
                                               uint8_t* __restrict__ sf) {
  float v[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) v[m] = __uint_as_float(h ? (w[m] & 0xffff0000u) : (w[m] << 16));
  if constexpr (NV) {
    uint2 lo, hi;
    const uint32_t s0 = nv_encode16_amax(v, amax16[0], rc1, 1.0f, lo);
    const uint32_t s1 = nv_encode16_amax(v + 16, amax16[1], rc1, 1.0f, hi);
    *reinterpret_cast<uint4*>(q + orow * (A / 2) + a / 2) = make_uint4(lo.x, lo.y, hi.x, hi.y);
    *reinterpret_cast<uint16_t*>(sf + sf_atom_offset(orow, a / 16, A / 16)) = (uint16_t)(s0 | (s1 << 8));
  } else {
    const int xe = mx_block_exponent(amax);
    uint32_t o[8];
    mx_encode32(v, xe, o);
    // one 256-bit store: the block's 32 codes fill one 32-byte sector
    asm volatile("st.global.v8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"l"(q + orow * A + a), "r"(o[0]), "r"(o[1]),
                 "r"(o[2]), "r"(o[3]), "r"(o[4]), "r"(o[5]), "r"(o[6]), "r"(o[7])
                 : "memory");
    sf[sf_atom_offset(orow, a / 32, A / 32)] = (uint8_t)(xe + 127);
  }
}

// Quantising warp `warp`, lane `lane`, on the stage at `stage` (see the map
// at the top): read the pairs, arrive on `empty`, quantise both columns.
// Block maxima come from the pairs with __hmax2 / __habs2, which order and
// ignore NaN as fmaxf / fabsf do on the widened values.
template <bool NV>
__device__ __forceinline__ void gt_quant_tile(const unsigned char* stage, uint64_t* empty, int warp, int lane, int a0,
                                              int b0, int A, float rc1, uint8_t* __restrict__ q0,
                                              uint8_t* __restrict__ sf0, uint8_t* __restrict__ q1,
                                              uint8_t* __restrict__ sf1) {
  const int src = warp >> 2, j = lane >> 3;
  const int col = 16 * (warp & 3) + 2 * (lane & 7);
  const unsigned char* tile = stage + src * kGtSrcBytes + col * 2;
  uint32_t w[32];
#pragma unroll
  for (int m = 0; m < 32; ++m) w[m] = *reinterpret_cast<const uint32_t*>(tile + gt_row(32 * j + m));
  __syncwarp();
  if (lane == 0) mbar_arrive(empty);
  __nv_bfloat162 mx[2];
#pragma unroll
  for (int s = 0; s < 2; ++s) {
    mx[s] = __floats2bfloat162_rn(0.0f, 0.0f);
#pragma unroll
    for (int m = 16 * s; m < 16 * s + 16; ++m)
      mx[s] = __hmax2(mx[s], __habs2(*reinterpret_cast<const __nv_bfloat162*>(&w[m])));
  }
  const __nv_bfloat162 mxa = __hmax2(mx[0], mx[1]);
  uint8_t* q = src ? q1 : q0;
  uint8_t* sf = src ? sf1 : sf0;
  const float lo16[2] = {__low2float(mx[0]), __low2float(mx[1])};
  const float hi16[2] = {__high2float(mx[0]), __high2float(mx[1])};
  gt_quant_block<NV>(w, 0, __low2float(mxa), lo16, b0 + col, a0 + 32 * j, A, rc1, q, sf);
  gt_quant_block<NV>(w, 1, __high2float(mxa), hi16, b0 + col + 1, a0 + 32 * j, A, rc1, q, sf);
}

}  // namespace

// kmag = ceil(2^32 / k) when every row index n satisfies n k < 2^32 (then
// n / k = umulhi(n, kmag) exactly), else 0 (plain division)
template <bool NV>
__global__ void __launch_bounds__(kGtThreads, 2) gather_transpose_q_kernel(
    const __nv_bfloat16* __restrict__ X0, const __nv_bfloat16* __restrict__ X1, const int32_t* __restrict__ perm_src,
    const int32_t* __restrict__ totals, int k, uint32_t kmag, int A, int B, uint8_t* __restrict__ q0,
    uint8_t* __restrict__ sf0, uint8_t* __restrict__ q1, uint8_t* __restrict__ sf1, int32_t* status,
    uint64_t timeout_ns, int stall) {
  extern __shared__ __align__(128) unsigned char gt_smem[];
  uint64_t* full = reinterpret_cast<uint64_t*>(gt_smem + kGtStages * kGtStageBytes);
  uint64_t* empty = full + kGtStages;
  int* abort_flag = reinterpret_cast<int*>(empty + kGtStages);
  const int rows_used = min(__ldg(totals), A);
  const int na = min((rows_used + 127) / 128, A / 128), ntiles = na * (B / 64);
  if ((int)blockIdx.x >= ntiles) return;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    *abort_flag = 0;
    for (int s = 0; s < kGtStages; ++s) {
      mbar_init(&full[s], 32 * kGtProdWarps);   // the producer lanes' copy completions
      mbar_init(&empty[s], kGtQuantWarps);  // one arrival per quantising warp
    }
    fence_mbar_init();
  }
  __syncthreads();
  const WaitCtl wc{status, abort_flag, timeout_ns};
  if (warp >= kGtQuantWarps) {
    if (stall) return;   // test hook: no copies, so the quantising warps' waits expire
    constexpr int R = 128 / kGtProdWarps;   // rows per producer warp
    const int r0 = (warp - kGtQuantWarps) * R;
    int i = 0;
    const int piece = lane & 7, rsub = lane >> 3;
    // tokens of the warp's rows in tile t (lane l: rows r0 + l + 32 p)
    auto lookup = [&](int t, int (&tk)[R / 32]) {
      const int a0 = (t % na) * 128;
#pragma unroll
      for (int p = 0; p < R / 32; ++p) {
        const int r = a0 + r0 + 32 * p + lane;
        const int src = t < ntiles && r < rows_used ? __ldg(perm_src + r) : -1;
        tk[p] = src < 0 ? -1 : kmag ? (int)__umulhi((uint32_t)src, kmag) : src / k;
      }
    };
    int tok[R / 32], nxt[R / 32];
    lookup(blockIdx.x, tok);
    for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
      const int s = i % kGtStages;
      lookup(t + gridDim.x, nxt);   // the next tile's lookups fly during the wait and the copies
      if (i >= kGtStages && !mbar_wait(&empty[s], (uint32_t)(i / kGtStages - 1) & 1u, wc)) break;
      const int b0 = (t / na) * 64;
      unsigned char* stage = gt_smem + s * kGtStageBytes;
#pragma unroll
      for (int q = 0; q < R / 4; ++q) {
        // row r0 + 4 q + rsub of the tile; its token sits in tok[q / 8] of lane 4 (q % 8) + rsub
        const int tk = __shfl_sync(0xffffffffu, tok[q >> 3], 4 * (q & 7) + rsub);
        const int64_t off = (int64_t)(tk < 0 ? 0 : tk) * B + b0 + piece * 8;
        const uint32_t bytes = tk < 0 ? 0u : 16u;
        unsigned char* d = stage + gt_row(r0 + 4 * q + rsub) + piece * 16;
        cp_async_16(d, X0 + off, bytes);
        cp_async_16(d + kGtSrcBytes, X1 + off, bytes);
      }
#pragma unroll
      for (int p = 0; p < R / 32; ++p) tok[p] = nxt[p];
      cp_async_mbar_arrive_noinc(&full[s]);
    }
    // every copy has landed before the warp leaves (also after an abort)
    cp_async_wait_all();
    return;
  }
  const float rc1 = nv_rc(1.0f);
  int i = 0;
  for (int t = blockIdx.x; t < ntiles; t += gridDim.x, ++i) {
    const int s = i % kGtStages;
    if (!mbar_wait(&full[s], (uint32_t)(i / kGtStages) & 1u, wc)) break;
    gt_quant_tile<NV>(gt_smem + s * kGtStageBytes, &empty[s], warp, lane, (t % na) * 128, (t / na) * 64, A, rc1, q0,
                      sf0, q1, sf1);
  }
}

cudaError_t launch_gather_transpose_q(bool nv, const void* X0, const void* X1, const int32_t* perm_src,
                                      const int32_t* totals, int k, int A, int B, void* q0, void* sf0, void* q1,
                                      void* sf1, int32_t* status, uint64_t timeout_ns, int stall, int grid,
                                      cudaStream_t st) {
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
  kern<<<grid, kGtThreads, kGtSmem, st>>>(x0, x1, perm_src, totals, k, kmag, A, B, o0, s0, o1, s1, status,
                                          timeout_ns, stall);
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
