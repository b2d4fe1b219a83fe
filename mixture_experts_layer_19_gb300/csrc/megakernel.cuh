// megakernel.cuh -- argument block of the ring-buffer forward megakernel
// (megakernel.cu), shared with the host code that fills it (api.cu).
#pragma once
#include <cuda.h>
#include <cuda_bf16.h>
#include <stdint.h>

#include "kernels.h"

namespace moe {

struct MegaArgs {
  CUtensorMap mapXr;    // sorted X rows (Xg), K-major loads {d, rows}, box 64 x 128
  CUtensorMap mapWg;    // Wg K-major {d, E*F}, box 64 x 128
  CUtensorMap mapWu;
  CUtensorMap mapWd;    // Wd K-major {F, E*d}, box 64 x 256
  CUtensorMap mapHr;    // ring h rows, K-major loads {F, ring rows}, box 64 x 128
  CUtensorMap mapHrSt;  // ring h rows, stores, box 32 x 32
  CUtensorMap mapABSt;  // saved a|b {2F, rows}, stores
  CUtensorMap mapYsSt;  // sorted y rows {d, rows}, stores
  const uint4* X;       // [T, d] bf16 tokens
  uint4* xg;            // [rows, d] bf16 sorted X rows (the weight gradients read them too)
  const int32_t* perm_src;
  const int32_t* mtile_off;   // [E+1]
  int32_t* mb_start;          // [n_mb+1] first 128-row tile of each minibatch
  int32_t* phase_start;       // [2 n_mb + 1] first claim index of each phase
  int32_t* n_mb;              // (written by the plan step, or in-kernel by the one-launch forward)
  int* claim;
  int* gathered;
  int* g1_done;
  int* mb_done;
  int32_t* status;
  uint64_t timeout_ns;
  int E, d, F, k, movers, slots, slot_rows;
  // One-launch forward (fwd_megakernel<true>): routing, minibatch planning
  // and the combine run inside the kernel.
  const float* logits;        // [T, E] router logits
  RoutingPtrs rp;             // routing state, written into the saved context
  int32_t* chunk_hist;        // [ceil(T/64), E] per-chunk expert counts
  int32_t* chunk_base;        // [ceil(T/64), E] per-chunk running sums
  int* counters;              // claim, gathered, g1_done, mb_done (zeroed in the kernel)
  int counters_len;
  const uint4* Ys;            // sorted y rows (what mapYsSt stores), read back by the combine
  uint4* Y;                   // [T, d] bf16 layer output
  int* tok_cnt;               // [T * d/256] y blocks stored per (token, 256-column block)
  unsigned long long* gbar;   // [2] grid-barrier arrivals, CTA exits (both zero between launches)
  int T, mbt, cap;
};

// One claimed unit of work of a ring megakernel.
struct Item {
  int kind;   // 0 = G1 ([a|b] + SwiGLU tile), 1 = G2 (down tile), -1 = stop
  int mb, gt, nt, e, ring_row0;
};

#ifdef __CUDACC__
// One thread: cut the 128-row tiles into minibatches on expert boundaries
// (>= mbt tiles when possible, <= cap tiles always; an expert larger than cap
// is split into cap-sized pieces) and lay out the claim order's phase
// boundaries.
// tiles[e]: the expert's 128-row tiles (shared memory, so the serial walk
// does not wait on global loads).
__device__ __forceinline__ void cut_minibatches(const int* tiles, int E, int mbt, int cap, int nt1, int nt2,
                                int32_t* mb_start, int32_t* phase_start, int32_t* n_mb) {
  int nb = 0, cur = 0, g = 0;
  mb_start[0] = 0;
  for (int e = 0; e < E; ++e) {
    int t = tiles[e];
    while (t > 0) {
      if (cur + t <= cap) {
        cur += t;
        g += t;
        t = 0;
        if (cur >= mbt) {
          mb_start[++nb] = g;
          cur = 0;
        }
      } else if (cur > 0) {
        mb_start[++nb] = g;
        cur = 0;
      } else {
        g += cap;
        t -= cap;
        mb_start[++nb] = g;
      }
    }
  }
  if (cur > 0) mb_start[++nb] = g;
  *n_mb = nb;
  // phases: G1(0), [G1(i), G2(i-1)] for i = 1..nb-1, G2(nb-1)
  int acc = 0, p = 0;
  phase_start[p++] = 0;
  for (int i = 0; i <= nb; ++i) {
    if (i < nb) {  // G1(i)
      acc += (mb_start[i + 1] - mb_start[i]) * nt1;
      phase_start[p++] = acc;
    }
    if (i >= 1) {  // G2(i-1)
      acc += (mb_start[i] - mb_start[i - 1]) * nt2;
      phase_start[p++] = acc;
    }
  }
}

__device__ __forceinline__ int find_last_le(const int32_t* a, int n, int v) {  // last i in [0,n) with a[i] <= v
  int lo = 0, hi = n;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (a[mid] <= v) lo = mid; else hi = mid;
  }
  return lo;
}

// Claim index -> work item.  Claim order: phases G1(0), G1(1), G2(0), G1(2),
// G2(1), ..., G2(n-1) (phase_start holds their first claim indices); inside a
// phase the N tile is the slow index and the minibatch's 128-row tile the
// fast one.  A is any argument block with phase_start, mb_start, mtile_off,
// E, slots, slot_rows.
template <class A>
__device__ __forceinline__ Item decode_claim(const A& g, int nmb, int c) {
  Item it;
  const int p = find_last_le(g.phase_start, 2 * nmb, c);
  const int local = c - g.phase_start[p];
  if (p == 0) { it.kind = 0; it.mb = 0; }
  else if (p == 2 * nmb - 1) { it.kind = 1; it.mb = nmb - 1; }
  else if (p & 1) { it.kind = 0; it.mb = (p + 1) >> 1; }
  else { it.kind = 1; it.mb = (p >> 1) - 1; }
  const int m0 = g.mb_start[it.mb];
  const int mts = g.mb_start[it.mb + 1] - m0;
  it.nt = local / mts;
  const int mt = local - it.nt * mts;
  it.gt = m0 + mt;
  it.e = find_last_le(g.mtile_off, g.E + 1, it.gt);
  while (it.e < g.E && g.mtile_off[it.e + 1] <= it.gt) ++it.e;  // skip empty experts
  it.ring_row0 = (it.mb % g.slots) * g.slot_rows + mt * 128;
  return it;
}
#endif

// Argument block of the BF16 backward megakernel (megakernel_bwd.cu): the
// expert FFNs' backward (B1-B4, B6) as one launch over the saved layout.
struct BwdMegaArgs {
  CUtensorMap mapU_A;   // dYg K-major {d, rows}, box 64 x 128
  CUtensorMap mapU_B;   // Wd MN-major {F, E*d}, box 64 x 64
  CUtensorMap mapX_A;   // dA|dB K-major {2F, rows}, box 64 x 128
  CUtensorMap mapX_Bg;  // Wg MN-major {d, E*F}, box 64 x 64
  CUtensorMap mapX_Bu;  // Wu MN-major
  CUtensorMap mapDabSt; // dA|dB stores {2F, rows}, box 32 x 32
  CUtensorMap mapWhSt;  // w h stores {F, rows}
  CUtensorMap mapYsSt;  // dx per sorted row {d, rows}
  const uint4* dY;      // [T, d] upstream gradient
  const uint4* X;       // [T, d] tokens
  uint4* dYg;           // [rows, d] sorted dY rows (written: the weight gradients read them)
  uint4* Xg;            // [rows, d] sorted X rows, or null when they are already in place
  const __nv_bfloat16* ab;   // saved a|b [rows, 2F]
  RoutingPtrs rp;            // saved routing (read only)
  float* dgp;                // [rows, F/256] partial <u, h>
  float* dg;                 // [T, k]
  float* dlogits;            // [T, E] or null
  const uint4* Ys;           // dx per sorted row, read back by the dX reduce
  uint4* dX;                 // [T, d]
  const int32_t* mtile_off;  // = rp.mtile_off
  int32_t* mb_start;
  int32_t* phase_start;
  int32_t* n_mb;
  int* counters;             // claim | gathered[nm] | u_done[nm]   (zeroed in the kernel)
  int counters_len;
  int* tok_dx;               // [T * d/256] dx blocks stored per (token, 256-column block)
  int* tok_u;                // [T] <u, h> partials stored per token
  unsigned long long* gbar;  // [2] grid barrier, CTA exits (zero between launches)
  int32_t* status;
  uint64_t timeout_ns;
  int E, d, F, k, T, mbt, cap, nm_max;
  int slots, slot_rows;      // 1, 0: the sorted buffers are not recycled
};

// Argument block of the MXFP8 ring megakernel (megakernel_mx.cu): the ring
// holds E4M3 X and h rows with their scale atoms (rows = ring rows).
struct MegaMxArgs {
  CUtensorMap mapXr;    // ring Xq, K-major {d bytes, ring rows}, box 128 x 128
  CUtensorMap mapWg;    // Wgq {d, E*F}, box 128 x 128
  CUtensorMap mapWu;
  CUtensorMap mapWd;    // Wdq {F, E*d}, box 128 x 256
  CUtensorMap mapHr;    // ring Hq loads {F, ring rows}, box 128 x 128
  CUtensorMap mapHrSt;  // ring Hq stores, box 32 x 32 bytes
  CUtensorMap mapABSt;  // saved a|b bf16 stores
  CUtensorMap mapYsSt;  // sorted y rows bf16 stores
  uint8_t* xq;          // [T, d] E4M3 tokens, quantised once per token along d
  uint8_t* xs;          // their scale atoms (rows = tokens, K = d)
  uint8_t* ring_xq;     // [ring rows, d] E4M3
  uint8_t* ring_xs;     // scale atoms of ring_xq (K = d)
  uint8_t* ring_hs;     // scale atoms of the ring Hq rows (K = F)
  const uint8_t* wgs;
  const uint8_t* wus;
  const uint8_t* wds;
  const int32_t* perm_src;
  const int32_t* mtile_off;
  int32_t* mb_start;
  int32_t* phase_start;
  int32_t* n_mb;
  int* claim;
  int* gathered;
  int* g1_done;
  int* mb_done;
  int32_t* status;
  uint64_t timeout_ns;
  int E, d, F, k, movers, slots, slot_rows;
  // One-launch forward (fwd_megakernel_mx<true>): token quantisation, routing,
  // minibatch planning and the combine run inside the kernel.
  const __nv_bfloat16* Xtok;  // [T, d] bf16 tokens (quantised into xq / xs in the kernel)
  const float* logits;
  RoutingPtrs rp;
  int32_t* chunk_hist;
  int32_t* chunk_base;
  int* counters;
  int counters_len;
  const uint4* Ys;
  uint4* Y;
  int* tok_cnt;
  unsigned long long* gbar;
  int T, mbt, cap;
};

}  // namespace moe
