// megakernel_common.cuh -- the one-launch pieces shared by the BF16 and MXFP8
// forward megakernels (megakernel.cu, megakernel_mx.cu): a bounded grid
// barrier, the exit count that resets it, routing + layout + minibatch plan
// inside the kernel, and the last-arriver combine.  A is the kernel's
// argument block (MegaArgs or MegaMxArgs: both carry the fields used here).
#pragma once
#include "gemm.cuh"
#include "megakernel.cuh"
#include "routing.cuh"

namespace moe {

// ----------------------------------------------------------------------------
// One-launch forward, phase A: routing, layout and the minibatch plan, run by
// every CTA of the cooperative launch before any of them takes a role.
// Grid barrier b (1..3) waits (bounded) until gbar[0] reaches b * gridDim.x.
// Every CTA counts itself out in gbar[1] on each way out of the kernel
// (fused_exit), and the last one zeroes both counters, so every launch --
// also a replayed CUDA graph -- starts from zero.  The stage ring's shared
// memory is scratch here (histograms, scan, placement cursors).
// ----------------------------------------------------------------------------
template <class A>
__device__ __forceinline__ bool grid_sync(const A& g, int b, const WaitCtl& wc, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(g.gbar, 1ull);
    *flag = wait_counter64_geq(g.gbar, (unsigned long long)b * gridDim.x, wc) ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

// Called once by thread 0 of every CTA after its last access to any counter.
template <class A>
__device__ __forceinline__ void fused_exit(const A& g) {
  __threadfence();
  if (atomicAdd(g.gbar + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
    g.gbar[0] = 0;
    g.gbar[1] = 0;
    __threadfence();
  }
}

template <class A>
__device__ bool route_in_kernel(const A& g, int* scratch, const WaitCtl& wc, int* flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  const int gtid = blockIdx.x * blockDim.x + threadIdx.x, gthreads = gridDim.x * blockDim.x;
  const int nt2 = g.d / BN;
  for (int i = gtid; i < g.counters_len; i += gthreads) g.counters[i] = 0;
  for (int i = gtid; i < g.T * nt2; i += gthreads) g.tok_cnt[i] = 0;
  // S1 + per-chunk histograms
  const int nch = (g.T + kRouteChunk - 1) / kRouteChunk;
  for (int c = blockIdx.x; c < nch; c += gridDim.x) {
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) scratch[e] = 0;
    __syncthreads();
    for (int tt = warp; tt < kRouteChunk; tt += nwarps) {
      const int t = c * kRouteChunk + tt;
      if (t >= g.T) break;
      route_token(g.logits, t, g.E, g.k, lane, g.rp.idx, g.rp.w, scratch);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) g.chunk_hist[(size_t)c * g.E + e] = scratch[e];
    __syncthreads();
  }
  if (!grid_sync(g, 1, wc, flag)) return false;
  // S2a + minibatch plan (one CTA)
  if (blockIdx.x == 0) {
    scan_experts(g.chunk_hist, g.chunk_base, nch, g.E, g.rp, scratch);
    int* tiles = scratch + g.E;    // scan_experts leaves the counts in scratch[0, E)
    for (int e = threadIdx.x; e < g.E; e += blockDim.x) tiles[e] = (scratch[e] + BM - 1) / BM;
    __syncthreads();
    if (threadIdx.x == 0)
      cut_minibatches(tiles, g.E, g.mbt, g.cap, g.F / 128, nt2, g.mb_start, g.phase_start, g.n_mb);
  }
  if (!grid_sync(g, 2, wc, flag)) return false;
  // S2b: one warp per chunk
  for (int c = blockIdx.x * nwarps + warp; c < nch; c += gridDim.x * nwarps)
    permute_chunk(g.chunk_base, g.T, g.E, g.k, c, g.rp, scratch + warp * g.E, lane);
  if (!grid_sync(g, 3, wc, flag)) return false;
  fence_proxy_async_smem();  // scratch writes before TMA reuses the stage ring
  __syncthreads();
  return true;
}

// One-launch forward, combine (S7) as "last arriver reduces": after a down
// tile's y rows are stored (complete and fenced), each row counts one arrival
// for (its token, the tile's 256-column block).  The lane that brings a count
// to k makes its warp sum that block of the token's k slot rows in slot order
// -- the same fmaf chain as combine_vec / combine_kernel -- and write it to Y.
template <class A>
__device__ __forceinline__ void combine_arrivals(const A& g, int srow, int nt, int lane) {
  const int nt2 = g.d / BN;
  const int src = g.rp.perm_src[srow + lane];
  int t = -1, last = 0;
  if (src >= 0) {
    t = src / g.k;
    __threadfence();
    // two warps store each row's 256-column block (one half each): the
    // block is complete at 2k arrivals
    last = atom_add_acq_rel_gpu(g.tok_cnt + (size_t)t * nt2 + nt, 1) == 2 * g.k - 1;
  }
  unsigned m = __ballot_sync(0xffffffffu, last);
  const int nvec = g.d / 8;
  const int i = nt * (BN / 8) + lane;  // 32 lanes x 8 columns = the 256-column block
  while (m) {
    const int l = __ffs(m) - 1;
    m &= m - 1;
    const int tt = __shfl_sync(0xffffffffu, t, l);
    // lanes 0..k-1 fetch the slot rows and weights at once; then every lane
    // loads its 16 bytes of up to 8 slot rows at a time before the fmaf
    // chain, which runs in slot order exactly as in combine_vec
    const int rl = lane < g.k ? g.rp.dest[(size_t)tt * g.k + lane] : 0;
    const float wl = lane < g.k ? g.rp.w[(size_t)tt * g.k + lane] : 0.0f;
    float acc[8];
#pragma unroll
    for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
    for (int j0 = 0; j0 < g.k; j0 += 8) {
      uint4 v[8];
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const int r = __shfl_sync(0xffffffffu, rl, (j0 + jj) & 31);
        if (j0 + jj < g.k) v[jj] = g.Ys[(size_t)r * nvec + i];
      }
#pragma unroll
      for (int jj = 0; jj < 8; ++jj) {
        const float wj = __shfl_sync(0xffffffffu, wl, (j0 + jj) & 31);
        if (j0 + jj < g.k) {
          const uint32_t u[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
            acc[2 * q] = fmaf(wj, f.x, acc[2 * q]);
            acc[2 * q + 1] = fmaf(wj, f.y, acc[2 * q + 1]);
          }
        }
      }
    }
    uint4 o;
    __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
    __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
    __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4], acc[5]);
    __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[6], acc[7]);
    o.x = *reinterpret_cast<uint32_t*>(&b0);
    o.y = *reinterpret_cast<uint32_t*>(&b1);
    o.z = *reinterpret_cast<uint32_t*>(&b2);
    o.w = *reinterpret_cast<uint32_t*>(&b3);
    g.Y[(size_t)tt * nvec + i] = o;
  }
}

}  // namespace moe
