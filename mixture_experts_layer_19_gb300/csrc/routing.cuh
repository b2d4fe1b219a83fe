// routing.cuh -- device-side pieces of routing, layout and combine, shared by
// the stand-alone kernels (routing.cu) and the one-launch forward megakernel
// (megakernel.cu), so that both compute bit-identical results.
//
// Mixture-of-Kittens pages: the router re-decides each token's experts at
// every step, and the layout step counts tokens per expert and places each
// expert's tokens contiguously (kucoin page "Cursor's MoK réalise une
// amélioration des performances de 2,37x sur NVIDIA GB300 NVL72", section
// 01).  The final weighted fusion (same page, section 03) uses one fixed
// order (laura-martel.com blog, section "Le déterminisme est la partie
// sous-estimée").
#pragma once
#include <cuda_bf16.h>
#include <math.h>
#include <stdint.h>

#include "kernels.h"

namespace moe {

constexpr int kRouteChunk = 64;  // tokens per router block / permutation chunk

// S1 for token t, one warp (lane = its lane).  Lane l holds logits l, l+32, ...;
// k rounds of a warp arg-max (larger logit wins, lower id on ties) pick the
// experts in descending order.  The weights are the softmax over the k picked
// logits, taken relative to the first (largest) one.  Each pick adds one to
// hist[expert] (shared memory).
__device__ __forceinline__ void route_token(const float* __restrict__ logits, int t, int E, int k, int lane,
                                            int32_t* __restrict__ idx, float* __restrict__ w, int* hist) {
  const int nper = (E + 31) >> 5;
  const float* row = logits + (size_t)t * E;
  float v[32];
#pragma unroll
  for (int i = 0; i < 32; ++i) {
    const int e = lane + 32 * i;
    v[i] = (i < nper && e < E) ? __ldg(row + e) : -INFINITY;
  }
  uint32_t taken = 0;
  int my_id = 0;
  float my_val = 0.0f;
  for (int j = 0; j < k; ++j) {
    float best = -INFINITY;
    int bid = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < 32; ++i) {
      const int e = lane + 32 * i;
      if (i < nper && e < E && !((taken >> i) & 1u)) {
        if (v[i] > best || (v[i] == best && e < bid)) {
          best = v[i];
          bid = e;
        }
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) {
      const float ob = __shfl_xor_sync(0xffffffffu, best, off);
      const int oi = __shfl_xor_sync(0xffffffffu, bid, off);
      if (ob > best || (ob == best && oi < bid)) {
        best = ob;
        bid = oi;
      }
    }
    if (bid == 0x7fffffff) bid = 0;  // only reachable with NaN logits (outside the contract)
    if ((bid & 31) == lane) taken |= 1u << (bid >> 5);
    if (lane == j) {
      my_id = bid;
      my_val = best;
    }
  }
  const float vmax = __shfl_sync(0xffffffffu, my_val, 0);
  const float z = lane < k ? expf(my_val - vmax) : 0.0f;
  float sum = z;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, off);
  if (lane < k) {
    idx[(size_t)t * k + lane] = my_id;
    w[(size_t)t * k + lane] = z / sum;
    atomicAdd(&hist[my_id], 1);
  }
}

// S2a for any block size: per-expert running sums over chunks (chunk bases)
// and counts, exclusive scans of the counts (unpadded offsets) and of the
// counts rounded up to the 128-row tile (padded segment starts), tile
// prefix, totals, padding markers.  s_cnt: E ints of shared memory.  The
// integers equal those of scan_kernel (routing.cu).
__device__ __forceinline__ void scan_experts(const int32_t* chunk_hist, int32_t* chunk_base, int nchunks, int E,
                                             const RoutingPtrs& rp, int* s_cnt) {
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    int cnt = 0;
    // eight chunk counts loaded before any running sum is stored, so the
    // loads overlap instead of each waiting behind the previous store
    for (int c0 = 0; c0 < nchunks; c0 += 8) {
      int h[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) h[u] = c0 + u < nchunks ? chunk_hist[(size_t)(c0 + u) * E + e] : 0;
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        if (c0 + u < nchunks) chunk_base[(size_t)(c0 + u) * E + e] = cnt;
        cnt += h[u];
      }
    }
    s_cnt[e] = cnt;
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    int off = 0, poff = 0;
    for (int e = 0; e < E; ++e) {
      const int c = s_cnt[e];
      rp.counts[e] = c;
      rp.offsets[e] = off;
      rp.poff[e] = poff;
      rp.mtile_off[e] = poff / kTileRows;
      off += c;
      poff += (c + kTileRows - 1) / kTileRows * kTileRows;
    }
    rp.offsets[E] = off;
    rp.poff[E] = poff;
    rp.mtile_off[E] = poff / kTileRows;
    rp.totals[0] = poff;  // padded rows in use
    rp.totals[1] = off;   // routed pairs
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) {
    const int c = s_cnt[e];
    const int p = rp.poff[e];
    const int padded = (c + kTileRows - 1) / kTileRows * kTileRows;
    for (int r = p + c; r < p + padded; ++r) rp.perm_src[r] = -1;
  }
}

// S2b: stable placement of chunk c by one warp.  The warp walks the chunk's
// pairs in flat order, 32 at a time; lanes with the same expert get
// consecutive slots in lane order (match_any + popc), so within an expert
// the flat index increases.  cursor: E ints of shared memory owned by the warp.
__device__ __forceinline__ void permute_chunk(const int32_t* chunk_base, int T, int E, int k, int c,
                                              const RoutingPtrs& rp, int* cursor, int lane) {
  for (int e = lane; e < E; e += 32) cursor[e] = rp.poff[e] + chunk_base[(size_t)c * E + e];
  __syncwarp();
  const int p0 = c * kRouteChunk * k;
  const int p1 = min(T, (c + 1) * kRouteChunk) * k;
  for (int base = p0; base < p1; base += 32) {
    const int p = base + lane;
    const bool valid = p < p1;
    const int e = valid ? rp.idx[p] : -1;
    const unsigned grp = __match_any_sync(0xffffffffu, e);
    const int rank = __popc(grp & ((1u << lane) - 1u));
    int slot = 0;
    if (valid) slot = cursor[e];
    __syncwarp();
    if (valid && rank == 0) cursor[e] = slot + __popc(grp);
    __syncwarp();
    if (valid) {
      const int dst = slot + rank;
      rp.dest[p] = dst;
      rp.perm_src[dst] = p;
    }
  }
  __syncwarp();
}

// B6 for token t, one warp: dg[t,j] = sum over the ntu N tiles of the
// partial <u, h> of pair j's sorted row (tile order), then
// dlogits[t, idx[t,j]] = w_j (dg_j - sum_i w_i dg_i) (warp-tree sum), zero
// elsewhere; dlogits may be null.
__device__ __forceinline__ void router_grad_token(const float* dgp, const int32_t* dest, const int32_t* idx,
                                                  const float* w, int t, int k, int E, int ntu, float* dg,
                                                  float* dlogits, int lane) {
  float g = 0.0f, wj = 0.0f;
  int e = 0;
  if (lane < k) {
    const int r = dest[(size_t)t * k + lane];
    for (int n = 0; n < ntu; ++n) g += dgp[(size_t)r * ntu + n];
    wj = w[(size_t)t * k + lane];
    e = idx[(size_t)t * k + lane];
    dg[(size_t)t * k + lane] = g;
  }
  float s = wj * g;
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
  if (dlogits) {
    float* row = dlogits + (size_t)t * E;
    for (int i = lane; i < E; i += 32) row[i] = 0.0f;
    __syncwarp();
    if (lane < k) row[e] = wj * (g - s);
  }
}

// S7 for token t, 8 columns starting at vector i (16 bytes): fp32 fmaf chain
// over the slots j = 0..k-1 (weights w, or 1 when w is null), one bf16
// rounding.  NC: the slot rows were written before this kernel started
// (read-only loads allowed); otherwise plain loads.
template <bool NC>
__device__ __forceinline__ uint4 combine_vec(const uint4* S, const int32_t* dest, const float* w, int t, int k,
                                             int nvec, int i) {
  float acc[8];
#pragma unroll
  for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
  for (int j = 0; j < k; ++j) {
    const int r = NC ? __ldg(dest + (size_t)t * k + j) : dest[(size_t)t * k + j];
    const float wj = w ? (NC ? __ldg(w + (size_t)t * k + j) : w[(size_t)t * k + j]) : 1.0f;
    const uint4 v = NC ? __ldg(S + (size_t)r * nvec + i) : S[(size_t)r * nvec + i];
    const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
      acc[2 * q] = fmaf(wj, f.x, acc[2 * q]);
      acc[2 * q + 1] = fmaf(wj, f.y, acc[2 * q + 1]);
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
  return o;
}

}  // namespace moe
