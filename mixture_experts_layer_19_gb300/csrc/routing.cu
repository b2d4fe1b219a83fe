// routing.cu -- router top-k + softmax weights, per-chunk expert histogram,
// scan to padded expert segments, stable permutation, row gathers (pull
// dispatch and its backward residue), fixed-order weighted combine, and the
// router-weight gradient.
//
// Mixture-of-Kittens pages: the router re-decides each token's experts at
// every step, then the layout step counts tokens per expert and places each
// expert's tokens contiguously so one grouped GEMM can consume them (kucoin
// page "Cursor's MoK réalise une amélioration des performances de 2,37x sur
// NVIDIA GB300 NVL72", section 01); dispatch is a pull by source position and
// combine a push to the token's home (same page, section 02); the final
// weighted fusion belongs to the layer (section 03); results are the same run
// to run (laura-martel.com blog, section "Le déterminisme est la partie
// sous-estimée") -- here every reduction has one fixed order and the only
// atomics are integer histogram increments.
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"
#include "routing.cuh"

namespace moe {

constexpr int kRouteThreads = 512;   // 16 warps: four tokens of a 64-token chunk each

// -----------------------------------------------------------------------------
// S1: one warp per token (route_token, routing.cuh); the block also
// histograms its chunk of kRouteChunk tokens.
// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(kRouteThreads) router_kernel(const float* __restrict__ logits, int T, int E,
                                                                 int k, int32_t* __restrict__ idx,
                                                                 float* __restrict__ w,
                                                                 int32_t* __restrict__ chunk_hist) {
  __shared__ int hist[1024];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  for (int tt = warp; tt < kRouteChunk; tt += kRouteThreads / 32) {
    const int t = blockIdx.x * kRouteChunk + tt;
    if (t >= T) break;
    route_token(logits, t, E, k, lane, idx, w, hist);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) chunk_hist[(size_t)blockIdx.x * E + e] = hist[e];
}

// -----------------------------------------------------------------------------
// S2a: per-expert running sums over chunks (chunk bases), per-expert counts,
// exclusive scans of counts (unpadded offsets) and of counts rounded up to
// the 128-row tile (padded segment starts), tile prefix, padding markers.
// One block of 1024 threads; thread e owns expert e.
// -----------------------------------------------------------------------------
__device__ __forceinline__ int block_excl_scan(int v, int* warp_tot, int* total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int x = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, x, off);
    if (lane >= off) x += y;
  }
  if (lane == 31) warp_tot[warp] = x;
  __syncthreads();
  if (warp == 0) {
    int s = warp_tot[lane];
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, s, off);
      if (lane >= off) s += y;
    }
    warp_tot[lane] = s;  // inclusive
    if (lane == 31) *total = s;
  }
  __syncthreads();
  const int res = x - v + (warp > 0 ? warp_tot[warp - 1] : 0);
  __syncthreads();
  return res;
}

__global__ void __launch_bounds__(1024) scan_kernel(const int32_t* __restrict__ chunk_hist,
                                                      int32_t* __restrict__ chunk_base, int nchunks, int E,
                                                      RoutingPtrs rp) {
  __shared__ int warp_tot[32];
  __shared__ int tot0, tot1;
  const int e = threadIdx.x;
  int cnt = 0;
  if (e < E) {
    for (int c = 0; c < nchunks; ++c) {
      chunk_base[(size_t)c * E + e] = cnt;
      cnt += chunk_hist[(size_t)c * E + e];
    }
  }
  const int padded = (cnt + kTileRows - 1) / kTileRows * kTileRows;
  const int off = block_excl_scan(cnt, warp_tot, &tot0);
  const int poff = block_excl_scan(padded, warp_tot, &tot1);
  if (e < E) {
    rp.counts[e] = cnt;
    rp.offsets[e] = off;
    rp.poff[e] = poff;
    rp.mtile_off[e] = poff / kTileRows;
    for (int r = poff + cnt; r < poff + padded; ++r) rp.perm_src[r] = -1;
  }
  if (threadIdx.x == 0) {
    rp.offsets[E] = tot0;
    rp.poff[E] = tot1;
    rp.mtile_off[E] = tot1 / kTileRows;
    rp.totals[0] = tot1;  // padded rows in use
    rp.totals[1] = tot0;  // routed pairs
  }
}

// -----------------------------------------------------------------------------
// S2b: stable placement.  One warp per chunk walks its pairs in flat order,
// 32 at a time; lanes with the same expert get consecutive slots in lane
// order (match_any + popc), so within an expert the flat index increases.
// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(32) permute_kernel(const int32_t* __restrict__ chunk_base, int T, int E, int k,
                                                     RoutingPtrs rp) {
  extern __shared__ int cursor[];
  permute_chunk(chunk_base, T, E, k, blockIdx.x, rp, cursor, threadIdx.x);
}

// S4 / B1: the sorted rows of one or two token tensors (G[r] = X[perm_src[r] /
// k]), walked by token so that each token's row is read from HBM once: work
// item (t, part) reads a quarter of token t's row (four 16-byte loads in
// flight per lane and source) and writes it to the token's k sorted rows
// dest[t k + j].  A second sweep zeroes the rows with perm_src < 0 (the
// padding at the end of each expert's segment).  X1 / G1 may be null.
__global__ void __launch_bounds__(256) gather_kernel(const uint4* __restrict__ X0, const uint4* __restrict__ X1,
                                                     const int32_t* __restrict__ perm_src,
                                                     const int32_t* __restrict__ dest,
                                                     const int32_t* __restrict__ totals, int T, int k, int d,
                                                     uint4* __restrict__ G0, uint4* __restrict__ G1) {
  constexpr int kParts = 4;
  const int nvec = d / 8, pvec = nvec / kParts;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  const int gw = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  for (int item = gw; item < T * kParts; item += warps_total) {
    const int t = item / kParts, c0 = (item - t * kParts) * pvec;
    const int dl = lane < k ? __ldg(dest + (size_t)t * k + lane) : 0;
    const uint4* x0 = X0 + (size_t)t * nvec;
    const uint4* x1 = X1 ? X1 + (size_t)t * nvec : nullptr;
    // every lane runs the same trips (the shuffles below take the whole
    // warp); only the loads and stores are guarded
    for (int i0 = c0; i0 < c0 + pvec; i0 += 128) {
      const int i = i0 + lane;
      uint4 a[4], b[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (i + 32 * u < c0 + pvec) {
          a[u] = __ldg(x0 + i + 32 * u);
          if (G1) b[u] = __ldg(x1 + i + 32 * u);
        }
      for (int j = 0; j < k; ++j) {
        const size_t r = (size_t)__shfl_sync(0xffffffffu, dl, j);
        uint4* g0 = G0 + r * nvec;
        uint4* g1 = G1 ? G1 + r * nvec : nullptr;
#pragma unroll
        for (int u = 0; u < 4; ++u)
          if (i + 32 * u < c0 + pvec) {
            g0[i + 32 * u] = a[u];
            if (G1) g1[i + 32 * u] = b[u];
          }
      }
    }
  }
  const int rows = totals[0];
  const uint4 z = make_uint4(0, 0, 0, 0);
  for (int r = gw; r < rows; r += warps_total) {
    if (__ldg(perm_src + r) >= 0) continue;
    uint4* g0 = G0 + (size_t)r * nvec;
    uint4* g1 = G1 ? G1 + (size_t)r * nvec : nullptr;
    for (int i = lane; i < nvec; i += 32) {
      g0[i] = z;
      if (G1) g1[i] = z;
    }
  }
}

// -----------------------------------------------------------------------------
// S7 / B4: Y[t] = sum_j w[t,j] * S[dest[t,j]] in slot order j = 0..k-1 as an
// fp32 fmaf chain, one rounding to bf16 (w == nullptr: plain sum, for dX).
// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(128) combine_kernel(const uint4* __restrict__ S, const int32_t* __restrict__ dest,
                                                      const float* __restrict__ w, int T, int k, int d,
                                                      uint4* __restrict__ Y) {
  const int nvec = d / 8;
  for (int t = blockIdx.x; t < T; t += gridDim.x)
    for (int i = threadIdx.x; i < nvec; i += blockDim.x)
      Y[(size_t)t * nvec + i] = combine_vec<true>(S, dest, w, t, k, nvec, i);
}

// -----------------------------------------------------------------------------
// B6: dg[t,j] = sum over N tiles of the partial <u, h> (tile order), then
// dlogits[t, idx[t,j]] = w_j (dg_j - sum_i w_i dg_i), zero elsewhere.
// One warp per token.
// -----------------------------------------------------------------------------
__global__ void __launch_bounds__(256) router_grad_kernel(const float* __restrict__ dgp,
                                                          const int32_t* __restrict__ dest,
                                                          const int32_t* __restrict__ idx,
                                                          const float* __restrict__ w, int T, int k, int E,
                                                          int ntu, float* __restrict__ dg,
                                                          float* __restrict__ dlogits) {
  const int lane = threadIdx.x & 31;
  const int warps_total = gridDim.x * (blockDim.x >> 5);
  for (int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); t < T; t += warps_total)
    router_grad_token(dgp, dest, idx, w, t, k, E, ntu, dg, dlogits, lane);
}

// -----------------------------------------------------------------------------
// moe_get_routing helper: padded sorted rows -> unpadded rows.
// -----------------------------------------------------------------------------
__global__ void unpad_routing_kernel(RoutingPtrs rp, int R, int32_t* __restrict__ perm_out,
                                     int32_t* __restrict__ dest_out) {
  for (int p = blockIdx.x * blockDim.x + threadIdx.x; p < R; p += gridDim.x * blockDim.x) {
    const int e = rp.idx[p];
    const int u = rp.dest[p] - rp.poff[e] + rp.offsets[e];
    if (dest_out) dest_out[p] = u;
    if (perm_out) perm_out[u] = p;
  }
}

// ============================================================================ launchers
cudaError_t launch_router(const float* logits, int T, int E, int k, int32_t* chunk_hist, const RoutingPtrs& rp,
                          cudaStream_t st) {
  router_kernel<<<route_chunks(T), kRouteThreads, 0, st>>>(logits, T, E, k, rp.idx, rp.w, chunk_hist);
  return cudaGetLastError();
}
cudaError_t launch_scan(int T, int E, const int32_t* chunk_hist, int32_t* chunk_base, const RoutingPtrs& rp,
                        cudaStream_t st) {
  scan_kernel<<<1, 1024, 0, st>>>(chunk_hist, chunk_base, route_chunks(T), E, rp);
  return cudaGetLastError();
}
cudaError_t launch_permute(int T, int E, int k, const int32_t* chunk_base, const RoutingPtrs& rp, cudaStream_t st) {
  permute_kernel<<<route_chunks(T), 32, E * sizeof(int), st>>>(chunk_base, T, E, k, rp);
  return cudaGetLastError();
}

int route_chunks(int T) { return (T + kRouteChunk - 1) / kRouteChunk; }

cudaError_t launch_gather(const void* X0, const void* X1, const int32_t* perm_src, const int32_t* dest,
                          const int32_t* totals, int T, int k, int d, void* G0, void* G1, int grid, cudaStream_t st) {
  gather_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4*>(X0), reinterpret_cast<const uint4*>(X1),
                                      perm_src, dest, totals, T, k, d, reinterpret_cast<uint4*>(G0),
                                      reinterpret_cast<uint4*>(G1));
  return cudaGetLastError();
}

cudaError_t launch_combine(const void* S, const int32_t* dest, const float* w, int T, int k, int d, void* Y,
                           int grid, cudaStream_t st) {
  combine_kernel<<<grid, 128, 0, st>>>(reinterpret_cast<const uint4*>(S), dest, w, T, k, d,
                                       reinterpret_cast<uint4*>(Y));
  return cudaGetLastError();
}

cudaError_t launch_router_grad(const float* dgp, const int32_t* dest, const int32_t* idx, const float* w, int T,
                               int k, int E, int ntu, float* dg, float* dlogits, int grid, cudaStream_t st) {
  router_grad_kernel<<<grid, 256, 0, st>>>(dgp, dest, idx, w, T, k, E, ntu, dg, dlogits);
  return cudaGetLastError();
}

cudaError_t launch_unpad_routing(const RoutingPtrs& rp, int R, int32_t* perm_out, int32_t* dest_out,
                                 cudaStream_t st) {
  unpad_routing_kernel<<<(R + 255) / 256, 256, 0, st>>>(rp, R, perm_out, dest_out);
  return cudaGetLastError();
}

}  // namespace moe
