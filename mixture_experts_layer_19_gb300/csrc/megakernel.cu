// megakernel.cu -- the forward expert pipeline as one persistent, device-driven
// kernel over a fixed ring token buffer.
//
// Mixture-of-Kittens pages (kucoin page "Cursor's MoK réalise une
// amélioration des performances de 2,37x sur NVIDIA GB300 NVL72", section 02;
// fluidifia page "Cursor ouvre MoK, un mégakernel qui accélère l'entraînement
// MoE", section "Comment MoK tente de gratter des millisecondes partout";
// laura-martel.com blog, section "Ce qu'il fait réellement"):
//  * the SMs are split into data movers and compute; GPU-local counters hand
//    work over in both directions;
//  * tokens are processed in tunable minibatches of at least two full waves
//    of the expert-grouped GEMM;
//  * a fixed ring of slots (the "macrobatch" buffer) is filled by dispatch and
//    reused as soon as a minibatch's results have gone back, so the combine
//    side of minibatch i overlaps the dispatch of minibatch i+1, with no CPU
//    in the loop and no allocation inside the layer.
//
// Here (one GPU): movers pull the routed token rows of minibatch i into their
// sorted rows (the local form of pull dispatch; the backward's weight
// gradients read the same rows, so they are not recycled), and ring slot
// i % S holds the minibatch's h rows between its two GEMMs.  Compute CTAs claim tiles
// from one global order -- G1(0), G1(1), G2(0), G1(2), G2(1), ... -- where
// G1(i) are the [a|b] = x [Wg;Wu]^T + SwiGLU tiles of minibatch i (h goes back
// into the slot, a|b to the saved context) and G2(i) the y = h Wd^T tiles (y to
// its sorted row: the push-combine residue).  Counters:
//   gathered[i] : mover CTAs done with minibatch i      (movers  -> G1 tiles)
//   g1_done[m]  : G1 warps done with 128-row tile m      (G1      -> G2 tiles)
//   mb_done[i]  : G1 + G2 warps done with minibatch i    (compute -> movers)
// Every tile only waits on work claimed before it (or on movers that wait on
// such work), and the launch is cooperative (all CTAs resident), so progress
// is guaranteed; every wait is also bounded in time (status word + abort).
// Each tile still reduces its K range in one fixed order: results are
// bitwise identical to the separate-kernel path.
//
// Minibatches are cut on expert boundaries (see plan_minibatches_kernel), so an
// expert's weights are streamed once unless it alone exceeds a slot.
#include "gemm.cuh"
#include "kernels.h"
#include "megakernel.cuh"
#include "megakernel_common.cuh"
#include "routing.cuh"

namespace moe {

constexpr int kQueue = 4;          // tiles in flight between producer and consumers
// warp 0 claimer + producer, warp 1 MMA, warps 2..9 epilogue, warps 10..11
// movers (when the ring has no dedicated mover CTAs).  A G1 tile's
// SwiGLU epilogue (three stores per element) runs on warps 2..5, one per TMEM
// lane quarter; a G2 tile's plain store is split over all eight, two per lane
// quarter, each on half of the columns (the store-bound kind gets the most
// store bandwidth, as in the separate down GEMM).
constexpr int kMegaThreads = 384;
constexpr int kMoverWarps = 2;              // mover warps of a compute CTA (warps 10, 11)
constexpr int kMegaStagingA = 3 * kStageChunk;  // warps 2..5: a, b, h (G1); double buffer (G2)
constexpr int kMegaStagingB = kStageChunk;      // warps 6..9: one buffer (G2 only)
constexpr int kMegaSmem = kStages * kStageBytes + 4 * kMegaStagingA + 4 * kMegaStagingB + 1024 + 512;
static_assert(kMegaSmem <= 232448, "shared memory per CTA");
constexpr int kG1Warps = 4, kG2Warps = 8;   // epilogue warps that finish one G1 / G2 tile

// ----------------------------------------------------------------------------
// Plan: zero the counters, cut minibatches on expert boundaries (>= mbt tiles
// when possible, <= cap tiles always; an expert larger than cap is split into
// cap-sized pieces), and lay out the claim order's phase boundaries.
// ----------------------------------------------------------------------------
__global__ void __launch_bounds__(1024) plan_minibatches_kernel(const int32_t* __restrict__ mtile_off, int E,
                                                                  int mbt, int cap, int nt1, int nt2,
                                                                  int counters_len, int* counters,
                                                                  int32_t* mb_start, int32_t* phase_start,
                                                                  int32_t* n_mb) {
  __shared__ int tiles[1024];
  for (int i = threadIdx.x; i < counters_len; i += blockDim.x) counters[i] = 0;
  for (int e = threadIdx.x; e < E; e += blockDim.x) tiles[e] = mtile_off[e + 1] - mtile_off[e];
  __syncthreads();
  if (threadIdx.x != 0) return;
  cut_minibatches(tiles, E, mbt, cap, nt1, nt2, mb_start, phase_start, n_mb);
}

// ----------------------------------------------------------------------------
// Mover CTA: pull minibatch rows into their ring slot.  Token rows travel as
// whole-row bulk copies (cp.async.bulk) through shared-memory buffers: warps
// 0..kMoverPipes-1 each run one pipeline (its lane 0 keeps up to nbuf - 1 row
// loads in flight, storing each row into the slot as it lands); the other
// warps write the slot's padding rows as zeros with plain stores.
// ----------------------------------------------------------------------------
constexpr int kMoverPipes = 3;
constexpr int kMoverBufMax = 5;   // buffers per pipeline at most

__device__ void mover_loop(const MegaArgs& g, int nmb, int* abort_flag, uint8_t* buf_base, uint64_t* mbar) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int nvec = g.d / 8;
  const uint32_t row_bytes = (uint32_t)g.d * 2;
  const int nt1 = g.F / 128, nt2 = g.d / BN;
  // buffers per pipeline: the stage ring and staging area (kMegaSmem less the
  // barrier block) hold kMoverPipes * nbuf rows
  const int nbuf = min(kMoverBufMax, (int)((kStages * kStageBytes + 4 * kMegaStagingA + 4 * kMegaStagingB) /
                                           (row_bytes * kMoverPipes)));
  WaitCtl wc{g.status, abort_flag, g.timeout_ns};
  const bool pipe = warp < kMoverPipes && lane == 0;
  uint8_t* bufs = buf_base + (size_t)warp * nbuf * row_bytes;
  uint64_t* bar = mbar + warp * kMoverBufMax;
  uint32_t phase = 0;   // bit b: parity of buffer b's next completion
  if (pipe)
    for (int b = 0; b < nbuf; ++b) mbar_init(&bar[b], 1);
  fence_mbar_init();
  __syncthreads();
  const int npipes = g.movers * kMoverPipes, pid = blockIdx.x * kMoverPipes + warp;
  const int nzw = g.movers * (nwarps - kMoverPipes), zid = blockIdx.x * (nwarps - kMoverPipes) + (warp - kMoverPipes);
  for (int mb = 0; mb < nmb; ++mb) {
    __syncthreads();
    if (*abort_flag) return;
    const int row_base = g.mb_start[mb] * BM;
    const int nrows = (g.mb_start[mb + 1] - g.mb_start[mb]) * BM;
    const size_t slot_base = (size_t)row_base;   // sorted rows of the minibatch
    if (pipe) {
      // step j stores this pipeline's row j - (nbuf - 1) (if any) and loads its
      // row j into buffer j % nbuf; that buffer's previous row was stored one
      // step earlier, so at most one younger store may still be reading
      int ld_i = pid, st_i = pid;          // next candidate row (slot-relative) to load / store
      int dst[kMoverBufMax];
      bool ok = true;
      for (int j = 0;; ++j) {
        const int s = j - (nbuf - 1);
        bool any = false;
        if (s >= 0) {
          while (st_i < nrows && g.perm_src[row_base + st_i] < 0) st_i += npipes;
          if (st_i < nrows) {
            const int b = s % nbuf;
            if (!mbar_wait(&bar[b], (phase >> b) & 1u, wc)) { ok = false; break; }
            phase ^= 1u << b;
            bulk_store_1d(g.xg + (slot_base + dst[b]) * nvec, bufs + (size_t)b * row_bytes, row_bytes);
            bulk_commit();
            st_i += npipes;
            any = true;
          }
        }
        while (ld_i < nrows && g.perm_src[row_base + ld_i] < 0) ld_i += npipes;
        if (ld_i < nrows) {
          const int b = j % nbuf;
          bulk_wait_read<1>();
          const int src = g.perm_src[row_base + ld_i];
          dst[b] = ld_i;
          mbar_arrive_expect_tx(&bar[b], row_bytes);
          bulk_load_1d(bufs + (size_t)b * row_bytes, g.X + (size_t)(src / g.k) * nvec, row_bytes, &bar[b]);
          ld_i += npipes;
          any = true;
        }
        if (!any && s >= 0) break;
      }
      if (!ok) {
        // abort: let every issued load land before the CTA may exit
        for (int b = 0; b < nbuf; ++b)
          for (uint64_t t0 = globaltimer_ns(); !mbar_try_wait(&bar[b], (phase >> b) & 1u);)
            if (globaltimer_ns() - t0 > 50000000ull) break;
      }
      bulk_wait<0>();   // the slot rows are written, not only read out of shared memory
    } else if (warp >= kMoverPipes) {
      for (int i = zid; i < nrows; i += nzw) {
        if (g.perm_src[row_base + i] >= 0) continue;
        uint4* d = g.xg + (slot_base + i) * nvec;
        for (int v = lane; v < nvec; v += 32) d[v] = make_uint4(0, 0, 0, 0);
      }
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      fence_proxy_async_global();
      red_release_gpu_add(g.gathered + mb, 1);
    }
  }
}

// ----------------------------------------------------------------------------
// The default: no mover CTAs; warps 10..11 of every compute CTA pull the rows
// (the pull-dispatch residue), so every SM also computes.  Mover warp w of
// CTA c copies the minibatch's rows i = (2c + w) + j * 2 * gridDim.x, each
// row by the whole warp with kCopyUnroll 16-byte loads in flight per lane;
// padding rows are written as zeros.
// ----------------------------------------------------------------------------
constexpr int kCopyUnroll = 8;

__device__ void mover_warps(const MegaArgs& g, int nmb, int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = g.d / 8;
  const int nt1 = g.F / 128, nt2 = g.d / BN;
  WaitCtl wc{g.status, abort_flag, g.timeout_ns};
  const int nw = gridDim.x * kMoverWarps, wid = blockIdx.x * kMoverWarps + (warp - 10);
  for (int mb = 0; mb < nmb; ++mb) {
    if (*reinterpret_cast<volatile int*>(abort_flag)) return;
    const int row_base = g.mb_start[mb] * BM;
    const int nrows = (g.mb_start[mb + 1] - g.mb_start[mb]) * BM;
    for (int i = wid; i < nrows; i += nw) {
      const int src = g.perm_src[row_base + i];
      uint4* dst = g.xg + (size_t)(row_base + i) * nvec;
      if (src < 0) {
        for (int v = lane; v < nvec; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
        continue;
      }
      const uint4* sp = g.X + (size_t)(src / g.k) * nvec;
      for (int v0 = 0; v0 < nvec; v0 += 32 * kCopyUnroll) {
        uint4 r[kCopyUnroll];
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) r[u] = __ldg(sp + v);
        }
#pragma unroll
        for (int u = 0; u < kCopyUnroll; ++u) {
          const int v = v0 + u * 32 + lane;
          if (v < nvec) dst[v] = r[u];
        }
      }
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      fence_proxy_async_global();
      red_release_gpu_add(g.gathered + mb, 1);
    }
  }
}

// FUSED: the one-launch forward (phase A above, combine in the down-tile
// epilogue); otherwise routing, plan and combine are separate launches.
template <bool FUSED>
__global__ void __launch_bounds__(kMegaThreads, 1) fwd_megakernel(const __grid_constant__ MegaArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* staging_base = smem + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging_base + 4 * kMegaStagingA + 4 * kMegaStagingB);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* qfull = tempty + 2;
  uint64_t* qempty = qfull + kQueue;
  Item* queue = reinterpret_cast<Item*>(qempty + kQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(queue + kQueue);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* sync_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();
  if (FUSED) {
    WaitCtl wca{g.status, abort_flag, g.timeout_ns};
    if (!route_in_kernel(g, reinterpret_cast<int*>(stage_base), wca, sync_flag)) {
      if (threadIdx.x == 0) fused_exit(g);
      return;
    }
  }
  const int nmb = *g.n_mb;
  if ((int)blockIdx.x < g.movers) {
    mover_loop(g, nmb, abort_flag, stage_base, bars);
    if (FUSED) {
      __syncthreads();
      if (threadIdx.x == 0) fused_exit(g);
    }
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kG2Warps);   // every epilogue warp arrives once per tile
    }
    for (int q = 0; q < kQueue; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], 1 + kG2Warps);  // MMA thread + 8 epilogue warps
    }
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
    tc_fence_before();
  }
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  WaitCtl wc{g.status, abort_flag, g.timeout_ns};
  const int nt1 = g.F / 128, nt2 = g.d / BN;
  const int total = g.phase_start[2 * nmb];
  // a minibatch is gathered once every mover CTA, or every mover warp, has
  // signalled it
  const int gathered_target = g.movers > 0 ? g.movers : (int)gridDim.x * kMoverWarps;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- claimer + producer
      // weights evict_last: the M tiles of a minibatch re-read each weight
      // tile, from CTAs that claim them at slightly different times
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      uint32_t s = 0, ph = 0, qi = 0, qph = 0, issued_mask = 0, last_par = 0;
      bool ok = true;
      // the next claim is taken while the current item's stages load, and
      // decoded right after them, so neither sits between two items' stages
      // the next claim is taken while the current item's stages load, and
      // decoded right after them, so neither sits between two items' stages
      int c = atomicAdd(g.claim, 1);
      Item nxt;
      nxt.kind = -1;
      if (c < total) nxt = decode_claim(g, nmb, c);
      while (ok) {
        Item it = nxt;
        const int c_next = c < total ? atomicAdd(g.claim, 1) : total;
        if (c < total) {
          if (it.kind == 0) {
            // the minibatch's X rows are gathered, and its ring slot's h rows
            // have been read by every G2 tile of minibatch mb - slots
            ok = wait_counter_geq(g.gathered + it.mb, gathered_target, wc);
            if (ok && it.mb >= g.slots) {
              const int prev = it.mb - g.slots;
              ok = wait_counter_geq(g.mb_done + prev,
                                    (g.mb_start[prev + 1] - g.mb_start[prev]) * (kG1Warps * nt1 + kG2Warps * nt2),
                                    wc);
            }
          } else {
            ok = wait_counter_geq(g.g1_done + it.gt, kG1Warps * nt1, wc);
          }
          fence_proxy_async_global();
          if (!ok) it.kind = -1;
        } else {
          it.kind = -1;
        }
        if (!mbar_wait(&qempty[qi], qph ^ 1, wc)) break;
        queue[qi] = it;
        mbar_arrive(&qfull[qi]);
        if (++qi == kQueue) { qi = 0; qph ^= 1; }
        if (it.kind < 0) break;
        const int nkb = it.kind == 0 ? g.d / BK : g.F / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          uint8_t* sa = stage_base + s * kStageBytes;
          uint8_t* sb = sa + kABytes;
          const int k0 = kb * BK;
          if (it.kind == 0) {
            tma_load_2d(sa, &g.mapXr, k0, it.gt * BM, &full[s], pol_a);
            tma_load_2d(sb, &g.mapWg, k0, it.e * g.F + it.nt * 128, &full[s], pol_w);
            tma_load_2d(sb + kBBytes / 2, &g.mapWu, k0, it.e * g.F + it.nt * 128, &full[s], pol_w);
          } else {
            tma_load_2d(sa, &g.mapHr, k0, it.ring_row0, &full[s], pol_a);
            tma_load_2d(sb, &g.mapWd, k0, it.e * g.d + it.nt * BN, &full[s], pol_w);
          }
          issued_mask |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
        c = c_next;
        if (c < total) nxt = decode_claim(g, nmb, c);
      }
      if (!ok) {
        for (int st = 0; st < kStages; ++st) {
          if (!(issued_mask & (1u << st))) continue;
          const uint32_t par = (last_par >> st) & 1u;
          for (uint64_t t0 = globaltimer_ns(); !mbar_try_wait(&full[st], par);)
            if (globaltimer_ns() - t0 > 50000000ull) break;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16(BM, BN, 0, 0);
      uint32_t s = 0, ph = 0, acc = 0, aph = 0, qi = 0, qph = 0;
      for (;;) {
        if (!mbar_wait(&qfull[qi], qph, wc)) break;
        const Item it = queue[qi];
        mbar_arrive(&qempty[qi]);
        if (++qi == kQueue) { qi = 0; qph ^= 1; }
        if (it.kind < 0) break;
        if (!mbar_wait(&tempty[acc], aph ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int nkb = it.kind == 0 ? g.d / BK : g.F / BK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024), idesc,
                      (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) aph ^= 1;
      }
    }
  } else if (warp >= 10) {
    // ------------------------------------------------- movers (no mover CTAs)
    if (g.movers == 0) mover_warps(g, nmb, abort_flag);
  } else {
    // ------------------------------------------------- epilogue
    const int q = warp & 3;                    // TMEM lane quarter this warp may access
    const bool g1_warp = warp < 2 + kG1Warps;  // warps 2..5 also run the SwiGLU epilogue
    const int c0 = ((warp - 2) >> 2) * 4;      // G2: this warp's four 32-column chunks
    uint8_t* stg = g1_warp ? staging_base + (warp - 2) * kMegaStagingA
                           : staging_base + kG1Warps * kMegaStagingA + (warp - 2 - kG1Warps) * kMegaStagingB;
    uint32_t acc = 0, aph = 0, qi = 0, qph = 0;
    int chunk_ctr = 0;
    for (;;) {
      if (!mbar_wait(&qfull[qi], qph, wc)) break;
      const Item it = queue[qi];
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qi]);
      if (++qi == kQueue) { qi = 0; qph ^= 1; }
      if (it.kind < 0) break;
      if (!mbar_wait(&tfull[acc], aph, wc)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + acc * BN;
      const int srow = it.gt * BM + 32 * q;        // sorted padded row of this warp's slab
      const int rrow = it.ring_row0 + 32 * q;      // ring row of this warp's slab
      if (it.kind == 0 && !g1_warp) {
        // a G1 tile is drained by warps 2..5; the others only release it
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      } else if (it.kind == 0) {
#pragma unroll 1
        for (int c = 0; c < 4; ++c) {
          uint32_t ra[32], rb[32];
          tmem_ld32(tbase + c * 32, ra);
          tmem_ld32(tbase + 128 + c * 32, rb);
          tmem_ld_wait();
          if (c == 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          float a[32], b[32], h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = __uint_as_float(ra[i]);
            b[i] = __uint_as_float(rb[i]);
            h[i] = a[i] * sigmoidf_(a[i]) * b[i];
          }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row(stg, lane, a);
          stage_row(stg + kStageChunk, lane, b);
          stage_row(stg + 2 * kStageChunk, lane, h);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int col = it.nt * 128 + c * 32;
            tma_store_2d(&g.mapABSt, stg, col, srow);
            tma_store_2d(&g.mapABSt, stg + kStageChunk, g.F + col, srow);
            tma_store_2d(&g.mapHrSt, stg + 2 * kStageChunk, col, rrow);
            bulk_commit();
          }
        }
      } else {
#pragma unroll 1
        for (int c = c0; c < c0 + 4; ++c) {
          uint32_t rv[32];
          tmem_ld32(tbase + c * 32, rv);
          tmem_ld_wait();
          if (c == c0 + 3) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rv[i]);
          uint8_t* buf = stg;
          if (g1_warp) {                 // double buffer
            buf += (chunk_ctr & 1) * kStageChunk;
            if (lane == 0) bulk_wait_read<1>();
          } else if (lane == 0) {
            bulk_wait_read<0>();
          }
          __syncwarp();
          stage_row(buf, lane, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&g.mapYsSt, buf, it.nt * BN + c * 32, srow);
            bulk_commit();
          }
          ++chunk_ctr;
        }
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      // hand-off counters.  A G1 tile's h rows must be complete before a G2
      // tile reads them, and a G2 tile's y rows before the in-kernel combine
      // reads them; a ring slot is free once every tile of its minibatch has
      // been drained (their MMAs have read the slot).
      if (it.kind == 0 && g1_warp) {
        if (lane == 0) {
          bulk_wait<0>();
          fence_proxy_async_global();
          red_release_gpu_add(g.g1_done + it.gt, 1);
          red_release_gpu_add(g.mb_done + it.mb, 1);
        }
      } else if (it.kind == 1) {
        if (lane == 0) {
          if (FUSED) {
            bulk_wait<0>();
            fence_proxy_async_global();
          }
          red_release_gpu_add(g.mb_done + it.mb, 1);
        }
      }
      __syncwarp();
      if (FUSED && it.kind == 1) combine_arrivals(g, srow, it.nt, lane);
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (FUSED && threadIdx.x == 0) fused_exit(g);
}

// ============================================================================ launchers
cudaError_t launch_plan_minibatches(const int32_t* mtile_off, int E, int mbt, int cap, int nt1, int nt2,
                                    int counters_len, int* counters, int32_t* mb_start, int32_t* phase_start,
                                    int32_t* n_mb, cudaStream_t st) {
  plan_minibatches_kernel<<<1, 1024, 0, st>>>(mtile_off, E, mbt, cap, nt1, nt2, counters_len, counters, mb_start,
                                               phase_start, n_mb);
  return cudaGetLastError();
}

cudaError_t launch_fwd_megakernel(const MegaArgs& a, int grid, bool fused, cudaStream_t st) {
  void* args[] = {const_cast<MegaArgs*>(&a)};
  const void* fn = fused ? reinterpret_cast<const void*>(fwd_megakernel<true>)
                         : reinterpret_cast<const void*>(fwd_megakernel<false>);
  return cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kMegaThreads), args, kMegaSmem, st);
}

cudaError_t prepare_fwd_megakernel() {
  cudaError_t e = cudaFuncSetAttribute(fwd_megakernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMegaSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fwd_megakernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMegaSmem);
}

size_t mega_args_size() { return sizeof(MegaArgs); }

}  // namespace moe
