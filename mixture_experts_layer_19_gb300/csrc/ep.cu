// ep.cu -- expert parallelism over R virtual ranks on one GPU: pull dispatch,
// push combine, pull reverse-combine and push reverse-dispatch with GPU-local
// flag signalling.
//
// Mixture-of-Kittens pages (kucoin page "Cursor's MoK réalise une
// amélioration des performances de 2,37x sur NVIDIA GB300 NVL72", section 02):
//  * dispatch is a pull: the rank that owns an expert fetches the tokens it
//    needs, knowing only which source rank holds each token and where; it
//    decides itself where the rows go locally, so no sender has to reserve
//    space in the receiver, and the rows land grouped by local expert;
//  * combine is a push: each result goes straight back to its token's home;
//  * backward mirrors them: pull reverse-combine, push reverse-dispatch;
//  * a receiver learns that its data is ready from signals, not from a
//    host-side barrier.
//
// Here the R ranks are CTA groups of one cooperative launch (G CTAs each):
// rank r owns the 64-token chunks [r C / R, (r+1) C / R) and the experts
// [r E / R, (r+1) E / R).  Its pulled rows form the region of the sorted row
// space that holds its experts, so the grouped GEMMs between the exchanges
// are the single-GPU ones, and every result equals the single-GPU path bit
// for bit.  Flags (ctr) are GPU-scope counters with release/acquire and
// bounded waits; the last CTA out of each launch zeroes them.
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"
#include "ptx.cuh"
#include "routing.cuh"

namespace moe {

constexpr int kEpThreads = 256;

struct EpRange {
  int t0, t1;        // own tokens
  int e0, e1;        // own experts
};

__device__ __forceinline__ EpRange ep_range(const EpArgs& a, int r) {
  const int c0 = r * a.nch / a.R, c1 = (r + 1) * a.nch / a.R;
  EpRange q;
  q.t0 = min(a.T, c0 * kRouteChunk);
  q.t1 = min(a.T, c1 * kRouteChunk);
  q.e0 = r * (a.E / a.R);
  q.e1 = (r + 1) * (a.E / a.R);
  return q;
}

// thread 0 waits (bounded) for ctr[i] >= target; the CTA learns the outcome
__device__ __forceinline__ bool ep_wait(const EpArgs& a, int i, int target, const WaitCtl& wc, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) *flag = wait_counter_geq(a.ctr + i, target, wc) ? 1 : 0;
  __syncthreads();
  return *flag != 0;
}
__device__ __forceinline__ void ep_signal(const EpArgs& a, int i) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    red_release_gpu_add(a.ctr + i, 1);
  }
}
// the last CTA to leave zeroes every flag for the next launch
__device__ __forceinline__ void ep_exit(const EpArgs& a) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    if (atomicAdd(a.ctr + 3 * a.R, 1) == (int)gridDim.x - 1) {
      for (int i = 0; i <= 3 * a.R; ++i) a.ctr[i] = 0;
      __threadfence();
    }
  }
}

// copy one row of d bf16 (or zeros) with a warp, 16-byte vectors, four
// loads in flight per lane
__device__ __forceinline__ void warp_copy_row(uint4* dst, const uint4* src, int nvec, int lane) {
  if (src) {
    for (int v = lane; v < nvec; v += 128) {
      uint4 t[4];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v + 32 * u < nvec) t[u] = src[v + 32 * u];
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (v + 32 * u < nvec) dst[v + 32 * u] = t[u];
    }
  } else {
    for (int v = lane; v < nvec; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
  }
}

// ----------------------------------------------------------------------------
// Forward dispatch.  Source role: rank r routes its own tokens (top-k, gate
// weights, per-chunk expert counts) and signals ctr[r].  Destination role:
// once every source has signalled, rank q lays out its own experts from the
// sources' counts (segment starts, chunk bases), places every pair routed to
// its experts (flat order within an expert: the stable layout), signals its
// own CTAs through ctr[R + q] and ctr[2R + q], and pulls the token rows into
// its region of the sorted buffer.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kEpThreads) ep_dispatch_kernel(const EpArgs a) {
  extern __shared__ int sm[];
  __shared__ int flag;
  __shared__ int abort_flag;
  const int r = blockIdx.x / a.G, lb = blockIdx.x % a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  WaitCtl wc{a.status, &abort_flag, a.timeout_ns};
  const EpRange me = ep_range(a, r);
  const int c_beg = r * a.nch / a.R, c_end = (r + 1) * a.nch / a.R;
  // --- source role: route own chunks
  for (int c = c_beg + lb; c < c_end; c += a.G) {
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) sm[e] = 0;
    __syncthreads();
    for (int tt = warp; tt < kRouteChunk; tt += nwarps) {
      const int t = c * kRouteChunk + tt;
      if (t >= a.T) break;
      route_token(a.logits, t, a.E, a.k, lane, a.rp.idx, a.rp.w, sm);
    }
    __syncthreads();
    for (int e = threadIdx.x; e < a.E; e += blockDim.x) a.chunk_hist[(size_t)c * a.E + e] = sm[e];
    __syncthreads();
  }
  ep_signal(a, r);
  // --- destination role: every source's counts are needed to lay out
  bool ok = true;
  for (int s = 0; s < a.R && ok; ++s) ok = ep_wait(a, s, a.G, wc, &flag);
  if (ok && lb == 0) {
    // counts of experts [0, e1): the lower experts only fix where this rank's
    // region starts; own experts also get their chunk bases
    int* cnt = sm;
    for (int e = threadIdx.x; e < me.e1; e += blockDim.x) {
      int n = 0;
      const bool own = e >= me.e0;
      for (int c = 0; c < a.nch; ++c) {
        if (own) a.chunk_base[(size_t)c * a.E + e] = n;
        n += a.chunk_hist[(size_t)c * a.E + e];
      }
      cnt[e] = n;
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      int off = 0, poff = 0;
      for (int e = 0; e < me.e1; ++e) {
        if (e >= me.e0) {
          a.rp.counts[e] = cnt[e];
          a.rp.offsets[e] = off;
          a.rp.poff[e] = poff;
          a.rp.mtile_off[e] = poff / kTileRows;
        }
        off += cnt[e];
        poff += (cnt[e] + kTileRows - 1) / kTileRows * kTileRows;
      }
      if (me.e1 == a.E) {  // the last rank closes the tables
        a.rp.offsets[a.E] = off;
        a.rp.poff[a.E] = poff;
        a.rp.mtile_off[a.E] = poff / kTileRows;
        a.rp.totals[0] = poff;
        a.rp.totals[1] = off;
      }
    }
    __syncthreads();
    for (int e = me.e0 + threadIdx.x; e < me.e1; e += blockDim.x) {
      const int p = a.rp.poff[e], c = cnt[e];
      for (int row = p + c; row < p + (c + kTileRows - 1) / kTileRows * kTileRows; ++row) a.rp.perm_src[row] = -1;
    }
    ep_signal(a, a.R + r);  // only the CTA that built the layout signals it
  }
  if (ok) ok = ep_wait(a, a.R + r, 1, wc, &flag);
  // place the pairs routed to own experts: one warp per chunk, flat order
  if (ok) {
    const int ne = me.e1 - me.e0;
    int* cursor = sm + warp * ne;
    for (int c = lb * nwarps + warp; c < a.nch; c += a.G * nwarps) {
      for (int i = lane; i < ne; i += 32)
        cursor[i] = a.rp.poff[me.e0 + i] + a.chunk_base[(size_t)c * a.E + me.e0 + i];
      __syncwarp();
      const int p0 = c * kRouteChunk * a.k, p1 = min(a.T, (c + 1) * kRouteChunk) * a.k;
      for (int base = p0; base < p1; base += 32) {
        const int p = base + lane;
        const int e = p < p1 ? a.rp.idx[p] : -1;
        const bool mine = e >= me.e0 && e < me.e1;
        const unsigned grp = __match_any_sync(0xffffffffu, mine ? e : -1);
        const int rank = __popc(grp & ((1u << lane) - 1u));
        int slot = 0;
        if (mine) slot = cursor[e - me.e0];
        __syncwarp();
        if (mine && rank == 0) cursor[e - me.e0] = slot + __popc(grp);
        __syncwarp();
        if (mine) {
          a.rp.dest[p] = slot + rank;
          a.rp.perm_src[slot + rank] = p;
        }
      }
      __syncwarp();
    }
    ep_signal(a, 2 * a.R + r);
    ok = ep_wait(a, 2 * a.R + r, a.G, wc, &flag);
  }
  // pull: own region of the sorted buffer <- token rows of any source rank.
  // The region ends where this rank's last expert segment ends (poff[e1]
  // belongs to the next rank, which may not have written it yet).
  if (ok) {
    const int nvec = a.d / 8;
    const int row0 = a.rp.poff[me.e0];
    const int row1 = a.rp.poff[me.e1 - 1] + (a.rp.counts[me.e1 - 1] + kTileRows - 1) / kTileRows * kTileRows;
    for (int row = row0 + lb * nwarps + warp; row < row1; row += a.G * nwarps) {
      const int p = a.rp.perm_src[row];
      warp_copy_row(a.Xg + (size_t)row * nvec, p >= 0 ? a.X + (size_t)(p / a.k) * nvec : nullptr, nvec, lane);
    }
  }
  ep_exit(a);
}

// ----------------------------------------------------------------------------
// Backward pull (reverse combine): home ranks signal that their tokens' dY is
// available; each expert rank then pulls the dY and X rows of its region.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kEpThreads) ep_pull_kernel(const EpArgs a) {
  __shared__ int flag;
  __shared__ int abort_flag;
  const int r = blockIdx.x / a.G, lb = blockIdx.x % a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  WaitCtl wc{a.status, &abort_flag, a.timeout_ns};
  ep_signal(a, r);
  bool ok = true;
  for (int s = 0; s < a.R && ok; ++s) ok = ep_wait(a, s, a.G, wc, &flag);
  if (ok) {
    const EpRange me = ep_range(a, r);
    const int nvec = a.d / 8;
    const int row0 = a.rp.poff[me.e0], row1 = a.rp.poff[me.e1];
    for (int row = row0 + lb * nwarps + warp; row < row1; row += a.G * nwarps) {
      const int p = a.rp.perm_src[row];
      const size_t tok = p >= 0 ? (size_t)(p / a.k) : 0;
      warp_copy_row(a.dYg + (size_t)row * nvec, p >= 0 ? a.dY + tok * nvec : nullptr, nvec, lane);
      warp_copy_row(a.Xg + (size_t)row * nvec, p >= 0 ? a.X + tok * nvec : nullptr, nvec, lane);
    }
  }
  ep_exit(a);
}

// ----------------------------------------------------------------------------
// Push (combine, or reverse dispatch) and the home-side reduction.  Expert
// role: rank q writes each sorted row of its region to the home slot of its
// pair (slot[p], p = t k + j), with the pair's <u, h> partials in the
// backward, then signals every home.  Home role: once all pushes have landed,
// rank r reduces its tokens' k slots in slot order -- the same arithmetic as
// combine_kernel (weights w, or a plain sum for dX) -- and, in the backward,
// forms dg and dlogits as router_grad_kernel does.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(kEpThreads) ep_push_kernel(const EpArgs a) {
  __shared__ int flag;
  __shared__ int abort_flag;
  const int r = blockIdx.x / a.G, lb = blockIdx.x % a.G;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, nwarps = blockDim.x >> 5;
  if (threadIdx.x == 0) abort_flag = 0;
  __syncthreads();
  WaitCtl wc{a.status, &abort_flag, a.timeout_ns};
  const EpRange me = ep_range(a, r);
  const int nvec = a.d / 8;
  {
    const int row0 = a.rp.poff[me.e0], row1 = a.rp.poff[me.e1];
    for (int row = row0 + lb * nwarps + warp; row < row1; row += a.G * nwarps) {
      const int p = a.rp.perm_src[row];
      if (p < 0) continue;
      warp_copy_row(a.slot + (size_t)p * nvec, a.Ys + (size_t)row * nvec, nvec, lane);
      if (a.dgp)
        for (int n = lane; n < a.ntu; n += 32) a.dgslot[(size_t)p * a.ntu + n] = a.dgp[(size_t)row * a.ntu + n];
    }
  }
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    for (int h = 0; h < a.R; ++h) red_release_gpu_add(a.ctr + h, 1);
  }
  if (ep_wait(a, r, a.R * a.G, wc, &flag)) {
    for (int t = me.t0 + lb * nwarps + warp; t < me.t1; t += a.G * nwarps) {
      // combine / dX reduce: lane i covers 16-byte vectors i, i+32, ...
      for (int i = lane; i < nvec; i += 32) {
        float acc[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) acc[q] = 0.0f;
        for (int j = 0; j < a.k; ++j) {
          const float wj = a.w_out ? a.w_out[(size_t)t * a.k + j] : 1.0f;
          const uint4 v = a.slot[((size_t)t * a.k + j) * nvec + i];
          const uint32_t u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
            acc[2 * q] = fmaf(wj, f.x, acc[2 * q]);
            acc[2 * q + 1] = fmaf(wj, f.y, acc[2 * q + 1]);
          }
        }
        __nv_bfloat162 b0 = __floats2bfloat162_rn(acc[0], acc[1]);
        __nv_bfloat162 b1 = __floats2bfloat162_rn(acc[2], acc[3]);
        __nv_bfloat162 b2 = __floats2bfloat162_rn(acc[4], acc[5]);
        __nv_bfloat162 b3 = __floats2bfloat162_rn(acc[6], acc[7]);
        a.out[(size_t)t * nvec + i] = make_uint4(*reinterpret_cast<uint32_t*>(&b0), *reinterpret_cast<uint32_t*>(&b1),
                                                 *reinterpret_cast<uint32_t*>(&b2), *reinterpret_cast<uint32_t*>(&b3));
      }
      if (a.dgp) {  // router gradient of token t
        float g = 0.0f, wj = 0.0f;
        int e = 0;
        if (lane < a.k) {
          const size_t p = (size_t)t * a.k + lane;
          for (int n = 0; n < a.ntu; ++n) g += a.dgslot[p * a.ntu + n];
          wj = a.rp.w[p];
          e = a.rp.idx[p];
          a.dg[p] = g;
        }
        float s = wj * g;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
        if (a.dlogits) {
          float* row = a.dlogits + (size_t)t * a.E;
          for (int i = lane; i < a.E; i += 32) row[i] = 0.0f;
          __syncwarp();
          if (lane < a.k) row[e] = wj * (g - s);
        }
      }
    }
  }
  ep_exit(a);
}

// ============================================================================ launchers
static cudaError_t ep_launch(const void* fn, const EpArgs& a, size_t smem, cudaStream_t st) {
  void* args[] = {const_cast<EpArgs*>(&a)};
  return cudaLaunchCooperativeKernel(fn, dim3(a.R * a.G), dim3(kEpThreads), args, smem, st);
}

cudaError_t launch_ep_dispatch(const EpArgs& a, cudaStream_t st) {
  // shared memory: max(E histogram ints, 8 warps x own-expert cursors, E counts)
  const size_t smem = (size_t)4 * max(a.E, (kEpThreads / 32) * (a.E / a.R));
  return ep_launch(reinterpret_cast<const void*>(ep_dispatch_kernel), a, smem, st);
}
cudaError_t launch_ep_pull(const EpArgs& a, cudaStream_t st) {
  return ep_launch(reinterpret_cast<const void*>(ep_pull_kernel), a, 0, st);
}
cudaError_t launch_ep_push(const EpArgs& a, cudaStream_t st) {
  return ep_launch(reinterpret_cast<const void*>(ep_push_kernel), a, 0, st);
}
cudaError_t prepare_ep() {
  return cudaFuncSetAttribute(ep_dispatch_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, 48 * 1024);
}

}  // namespace moe
