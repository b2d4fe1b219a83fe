// megakernel_bwd.cu -- the expert FFNs' backward (BF16) as one persistent,
// device-driven launch: the reverse of the ring forward.
//
// Mixture-of-Kittens pages: the backward adds the two communication steps in
// reverse -- a pull of the upstream gradient rows to the experts (reverse
// combine) and a push of the input-gradient rows back to their tokens
// (reverse dispatch) (kucoin page "Cursor's MoK réalise une amélioration des
// performances de 2,37x sur NVIDIA GB300 NVL72", sections 01 and 02); one
// kernel, one launch, no host round trip (laura-martel.com blog, section "Ce
// qu'il fait réellement"); every reduction in one fixed order (same blog,
// section "Le déterminisme est la partie sous-estimée").
//
// Here, on one GPU:
//  * phase A (all CTAs): zero the hand-off counters; CTA 0 cuts the saved
//    layout's 128-row tiles into minibatches (the forward's two-wave floor);
//    one bounded grid barrier;
//  * movers (warps 10..11 of every CTA) pull each minibatch's dY rows -- and
//    X rows when they are not in place already -- into the sorted buffers
//    (B1).  The weight gradients read those buffers after this launch, so
//    the rows stay where they land rather than in recycled slots;
//  * compute CTAs claim tiles in the order U(0), U(1), DX(0), U(2), DX(1), ...:
//      U(i)  u = dYg Wd (K = d) with the SwiGLU-backward epilogue: dA|dB,
//            w h and the per-tile partials <u, h> (B2).  When a token's last
//            partial lands, that warp forms its dg and dlogits (B6);
//      DX(i) dx = dA|dB [Wg; Wu] (K = 2F), one row per (token, slot) pair
//            (B3).  When the k rows of a token's 256-column block are all
//            stored, that warp sums them in slot order into dX (B4).
// Counters: gathered[i] (movers -> U tiles of minibatch i), u_done[m] (the
// eight U tiles of 128-row block m -> its DX tiles), tok_dx / tok_u
// (arrivals for the two in-kernel reductions).  Every tile waits only on work
// claimed before it, the launch is cooperative, and every wait is bounded.
// Each tile reduces its K range in one fixed order and the reductions use the
// separate kernels' arithmetic, so results are bitwise identical to them.
#include "gemm.cuh"
#include "kernels.h"
#include "megakernel.cuh"
#include "routing.cuh"

namespace moe {

namespace {

constexpr int kBQueue = 4;
constexpr int kBThreads = 384;             // producer, MMA, 8 epilogue warps, 2 mover warps
constexpr int kBMoverWarps = 2;
constexpr int kBStagingA = 3 * kStageChunk;   // warps 2..5: dA, dB, w h (U); double buffer (DX)
constexpr int kBStagingB = kStageChunk;       // warps 6..9: one buffer (DX only)
constexpr int kBSmem = kStages * kStageBytes + 4 * kBStagingA + 4 * kBStagingB + 1024 + 512;
static_assert(kBSmem <= 232448, "shared memory per CTA");
constexpr int kUWarps = 4, kXWarps = 8;    // epilogue warps that finish one U / DX tile
constexpr int kCopyUnrollB = 8;

__device__ __forceinline__ bool grid_sync_b(unsigned long long* gbar, int b, const WaitCtl& wc, int* flag) {
  __syncthreads();
  if (threadIdx.x == 0) {
    __threadfence();
    atomicAdd(gbar, 1ull);
    *flag = wait_counter64_geq(gbar, (unsigned long long)b * gridDim.x, wc) ? 1 : 0;
  }
  __syncthreads();
  return *flag != 0;
}

// Called once by thread 0 of every CTA after its last access to any counter;
// the last CTA out zeroes the barrier, so every launch starts from zero.
__device__ __forceinline__ void exit_b(unsigned long long* gbar) {
  __threadfence();
  if (atomicAdd(gbar + 1, 1ull) == (unsigned long long)gridDim.x - 1) {
    gbar[0] = 0;
    gbar[1] = 0;
    __threadfence();
  }
}

// One sorted row by the whole warp: dst <- src's token row, or zeros.
__device__ __forceinline__ void copy_row_b(uint4* dst, const uint4* src_rows, int src, int k, int nvec, int lane) {
  if (src < 0) {
    for (int v = lane; v < nvec; v += 32) dst[v] = make_uint4(0, 0, 0, 0);
    return;
  }
  const uint4* sp = src_rows + (size_t)(src / k) * nvec;
  for (int v0 = 0; v0 < nvec; v0 += 32 * kCopyUnrollB) {
    uint4 q[kCopyUnrollB];
#pragma unroll
    for (int u = 0; u < kCopyUnrollB; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < nvec) q[u] = __ldg(sp + v);
    }
#pragma unroll
    for (int u = 0; u < kCopyUnrollB; ++u) {
      const int v = v0 + u * 32 + lane;
      if (v < nvec) dst[v] = q[u];
    }
  }
}

// B1: mover warp w of CTA c copies the minibatch's rows (2c + w) + j * 2 * grid
// of dY, minibatch by minibatch (the U tiles wait on them); then, when they
// are not in place already (a forward of another plan or another input ran
// in between), the X rows of every minibatch, which only the weight
// gradients read after this launch.
__device__ void mover_warps_b(const BwdMegaArgs& g, int nmb, int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nvec = g.d / 8;
  const int nw = gridDim.x * kBMoverWarps, wid = blockIdx.x * kBMoverWarps + (warp - 10);
  for (int mb = 0; mb < nmb; ++mb) {
    if (*reinterpret_cast<volatile int*>(abort_flag)) return;
    const int row_base = g.mb_start[mb] * BM;
    const int nrows = (g.mb_start[mb + 1] - g.mb_start[mb]) * BM;
    for (int i = wid; i < nrows; i += nw) {
      const int r = row_base + i;
      copy_row_b(g.dYg + (size_t)r * nvec, g.dY, g.rp.perm_src[r], g.k, nvec, lane);
    }
    __syncwarp();
    if (lane == 0) {
      __threadfence();
      fence_proxy_async_global();
      red_release_gpu_add(g.counters + 1 + mb, 1);   // gathered[mb]
    }
  }
  if (g.Xg) {
    const int nrows = g.mb_start[nmb] * BM;
    for (int r = wid; r < nrows; r += nw) copy_row_b(g.Xg + (size_t)r * nvec, g.X, g.rp.perm_src[r], g.k, nvec, lane);
  }
}

// B4 in the DX epilogue: each of the warp's 32 rows counts one arrival for
// (its token, the tile's 256-column block); two warps store each block (one
// half each), so the block is complete at 2k arrivals.  The warp then sums
// that block of the token's k rows in slot order -- combine_vec's chain with
// unit weights -- into dX.
__device__ __forceinline__ void dx_arrivals(const BwdMegaArgs& g, int srow, int nt, int lane) {
  const int nt2 = g.d / BN;
  const int src = g.rp.perm_src[srow + lane];
  int t = -1, last = 0;
  if (src >= 0) {
    t = src / g.k;
    __threadfence();
    last = atom_add_acq_rel_gpu(g.tok_dx + (size_t)t * nt2 + nt, 1) == 2 * g.k - 1;
  }
  unsigned m = __ballot_sync(0xffffffffu, last);
  const int nvec = g.d / 8;
  const int i = nt * (BN / 8) + lane;
  while (m) {
    const int l = __ffs(m) - 1;
    m &= m - 1;
    const int tt = __shfl_sync(0xffffffffu, t, l);
    const int rl = lane < g.k ? g.rp.dest[(size_t)tt * g.k + lane] : 0;
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
        if (j0 + jj < g.k) {
          const uint32_t u[4] = {v[jj].x, v[jj].y, v[jj].z, v[jj].w};
#pragma unroll
          for (int q = 0; q < 4; ++q) {
            const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[q]));
            acc[2 * q] = fmaf(1.0f, f.x, acc[2 * q]);
            acc[2 * q + 1] = fmaf(1.0f, f.y, acc[2 * q + 1]);
          }
        }
      }
    }
    uint4 o;
    o.x = pack_bf16(acc[0], acc[1]);
    o.y = pack_bf16(acc[2], acc[3]);
    o.z = pack_bf16(acc[4], acc[5]);
    o.w = pack_bf16(acc[6], acc[7]);
    g.dX[(size_t)tt * nvec + i] = o;
  }
}

// B6 in the U epilogue: each of the warp's 32 rows counts one arrival for its
// token (after its partial <u, h> is written); a token is complete after k
// pairs x F/256 tiles, and the warp then runs router_grad_token for it.
__device__ __forceinline__ void u_arrivals(const BwdMegaArgs& g, int srow, int lane) {
  const int ntu = g.F / BN;
  const int src = g.rp.perm_src[srow + lane];
  int t = -1, last = 0;
  if (src >= 0) {
    t = src / g.k;
    __threadfence();
    last = atom_add_acq_rel_gpu(g.tok_u + t, 1) == g.k * ntu - 1;
  }
  unsigned m = __ballot_sync(0xffffffffu, last);
  while (m) {
    const int l = __ffs(m) - 1;
    m &= m - 1;
    const int tt = __shfl_sync(0xffffffffu, t, l);
    router_grad_token(g.dgp, g.rp.dest, g.rp.idx, g.rp.w, tt, g.k, g.E, ntu, g.dg, g.dlogits, lane);
  }
}

}  // namespace

__global__ void __launch_bounds__(kBThreads, 1) bwd_megakernel(const __grid_constant__ BwdMegaArgs g) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* staging_base = smem + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging_base + 4 * kBStagingA + 4 * kBStagingB);
  uint64_t* full = bars;
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* qfull = tempty + 2;
  uint64_t* qempty = qfull + kBQueue;
  Item* queue = reinterpret_cast<Item*>(qempty + kBQueue);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(queue + kBQueue);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* sync_flag = abort_flag + 1;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int ntu = g.F / BN, ntx = g.d / BN;

  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();
  // ---------------------------------------------------------------- phase A
  {
    WaitCtl wca{g.status, abort_flag, g.timeout_ns};
    const int gtid = blockIdx.x * blockDim.x + threadIdx.x, gthreads = gridDim.x * blockDim.x;
    for (int i = gtid; i < g.counters_len; i += gthreads) g.counters[i] = 0;
    for (int i = gtid; i < g.T * ntx; i += gthreads) g.tok_dx[i] = 0;
    for (int i = gtid; i < g.T; i += gthreads) g.tok_u[i] = 0;
    if (blockIdx.x == 0) {
      int* tiles = reinterpret_cast<int*>(stage_base);
      for (int e = threadIdx.x; e < g.E; e += blockDim.x) tiles[e] = g.mtile_off[e + 1] - g.mtile_off[e];
      __syncthreads();
      if (threadIdx.x == 0) cut_minibatches(tiles, g.E, g.mbt, g.cap, ntu, ntx, g.mb_start, g.phase_start, g.n_mb);
    }
    if (!grid_sync_b(g.gbar, 1, wca, sync_flag)) {
      if (threadIdx.x == 0) exit_b(g.gbar);
      return;
    }
  }
  const int nmb = *g.n_mb;
  int* gathered = g.counters + 1;
  int* u_done = g.counters + 1 + g.nm_max;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], kXWarps);
    }
    for (int q = 0; q < kBQueue; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], 1 + kXWarps);
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
  const int total = g.phase_start[2 * nmb];
  const int gathered_target = (int)gridDim.x * kBMoverWarps;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- claimer + producer
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      uint32_t s = 0, ph = 0, qi = 0, qph = 0, issued_mask = 0, last_par = 0;
      bool ok = true;
      // the next claim is taken while the current item's stages load
      int c = atomicAdd(g.counters, 1);
      Item nxt;
      nxt.kind = -1;
      if (c < total) nxt = decode_claim(g, nmb, c);
      while (ok) {
        Item it = nxt;
        const int c_next = c < total ? atomicAdd(g.counters, 1) : total;
        if (c < total) {
          ok = it.kind == 0 ? wait_counter_geq(gathered + it.mb, gathered_target, wc)
                            : wait_counter_geq(u_done + it.gt, kUWarps * ntu, wc);
          fence_proxy_async_global();
          if (!ok) it.kind = -1;
        } else {
          it.kind = -1;
        }
        if (!mbar_wait(&qempty[qi], qph ^ 1, wc)) break;
        queue[qi] = it;
        mbar_arrive(&qfull[qi]);
        if (++qi == kBQueue) { qi = 0; qph ^= 1; }
        if (it.kind < 0) break;
        const int nkb = it.kind == 0 ? g.d / BK : (2 * g.F) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          uint8_t* sa = stage_base + s * kStageBytes;
          uint8_t* sb = sa + kABytes;
          const int k0 = kb * BK;
          if (it.kind == 0) {
            tma_load_2d(sa, &g.mapU_A, k0, it.gt * BM, &full[s], pol_a);
#pragma unroll
            for (int j = 0; j < 4; ++j)
              tma_load_2d(sb + j * 8192, &g.mapU_B, it.nt * BN + j * 64, it.e * g.d + k0, &full[s], pol_w);
          } else {
            tma_load_2d(sa, &g.mapX_A, k0, it.gt * BM, &full[s], pol_a);
            const bool up = k0 >= g.F;
            const CUtensorMap* mb = up ? &g.mapX_Bu : &g.mapX_Bg;
            const int krow = it.e * g.F + (up ? k0 - g.F : k0);
#pragma unroll
            for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, mb, it.nt * BN + j * 64, krow, &full[s], pol_w);
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
      // ------------------------------------------------- MMA issuer (A K-major, B MN-major)
      constexpr uint32_t idesc = idesc_bf16(BM, BN, 0, 1);
      uint32_t s = 0, ph = 0, acc = 0, aph = 0, qi = 0, qph = 0;
      for (;;) {
        if (!mbar_wait(&qfull[qi], qph, wc)) break;
        const Item it = queue[qi];
        mbar_arrive(&qempty[qi]);
        if (++qi == kBQueue) { qi = 0; qph ^= 1; }
        if (it.kind < 0) break;
        if (!mbar_wait(&tempty[acc], aph ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        const int nkb = it.kind == 0 ? g.d / BK : (2 * g.F) / BK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            umma_bf16(d_tmem, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 2048, 8192, 1024), idesc,
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
    mover_warps_b(g, nmb, abort_flag);
  } else {
    // ------------------------------------------------- epilogue
    const int q = warp & 3;
    const bool u_warp = warp < 2 + kUWarps;
    const int c0 = ((warp - 2) >> 2) * 4;
    uint8_t* stg = u_warp ? staging_base + (warp - 2) * kBStagingA
                          : staging_base + kUWarps * kBStagingA + (warp - 2 - kUWarps) * kBStagingB;
    uint32_t acc = 0, aph = 0, qi = 0, qph = 0;
    int chunk_ctr = 0;
    for (;;) {
      if (!mbar_wait(&qfull[qi], qph, wc)) break;
      const Item it = queue[qi];
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qi]);
      if (++qi == kBQueue) { qi = 0; qph ^= 1; }
      if (it.kind < 0) break;
      if (!mbar_wait(&tfull[acc], aph, wc)) break;
      tc_fence_after();
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + acc * BN;
      const int rowq = it.gt * BM + 32 * q;
      if (it.kind == 0 && !u_warp) {
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[acc]);
      } else if (it.kind == 0) {
        // B2 epilogue: the arithmetic of the separate u GEMM's epilogue
        const int r = rowq + lane;
        const int src = g.rp.perm_src[r];
        const float wr = src >= 0 ? g.rp.w[src] : 0.0f;
        const __nv_bfloat16* abrow = g.ab + (size_t)r * (2 * g.F);
        float dgacc = 0.0f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t ru[32];
          tmem_ld32(tbase + c * 32, ru);
          const int col = it.nt * BN + c * 32;
          float a[32], b[32];
          load_bf16x32(abrow + col, a);
          load_bf16x32(abrow + g.F + col, b);
          tmem_ld_wait();
          if (c == 7) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          // dA, dB, w h packed to bf16 pairs as they are formed (the same
          // rounding stage_row applies)
          uint32_t pda[16], pdb[16], pwh[16];
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            float da2[2], db2[2], wh2[2];
#pragma unroll
            for (int h2 = 0; h2 < 2; ++h2) {
              const int i = 2 * i2 + h2;
              const float u = __uint_as_float(ru[i]);
              const float sa = sigmoidf_(a[i]);
              const float sl = a[i] * sa;
              const float hh = sl * b[i];
              dgacc = fmaf(u, hh, dgacc);
              const float dh = wr * u;
              da2[h2] = dh * b[i] * sa * (1.0f + a[i] * (1.0f - sa));
              db2[h2] = dh * sl;
              wh2[h2] = wr * hh;
            }
            pda[i2] = pack_bf16(da2[0], da2[1]);
            pdb[i2] = pack_bf16(db2[0], db2[1]);
            pwh[i2] = pack_bf16(wh2[0], wh2[1]);
          }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row_packed(stg, lane, pda);
          stage_row_packed(stg + kStageChunk, lane, pdb);
          stage_row_packed(stg + 2 * kStageChunk, lane, pwh);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&g.mapDabSt, stg, col, rowq);
            tma_store_2d(&g.mapDabSt, stg + kStageChunk, g.F + col, rowq);
            tma_store_2d(&g.mapWhSt, stg + 2 * kStageChunk, col, rowq);
            bulk_commit();
          }
        }
        g.dgp[(size_t)r * ntu + it.nt] = dgacc;
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
          if (u_warp) {
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
            tma_store_2d(&g.mapYsSt, buf, it.nt * BN + c * 32, rowq);
            bulk_commit();
          }
          ++chunk_ctr;
        }
      }
      acc ^= 1;
      if (acc == 0) aph ^= 1;
      // hand-offs: dA|dB rows complete before a DX tile loads them; dx rows
      // complete before the dX reduce reads them
      if ((it.kind == 0 && u_warp) || it.kind == 1) {
        if (lane == 0) {
          bulk_wait<0>();
          fence_proxy_async_global();
          if (it.kind == 0) red_release_gpu_add(u_done + it.gt, 1);
        }
        __syncwarp();
        if (it.kind == 0) u_arrivals(g, rowq, lane);
        else dx_arrivals(g, rowq, it.nt, lane);
      }
    }
    if (lane == 0) bulk_wait<0>();
    __syncwarp();
  }

  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, 512);
  }
  if (threadIdx.x == 0) exit_b(g.gbar);
}

cudaError_t launch_bwd_megakernel(const BwdMegaArgs& a, int grid, cudaStream_t st) {
  void* args[] = {const_cast<BwdMegaArgs*>(&a)};
  return cudaLaunchCooperativeKernel(reinterpret_cast<const void*>(bwd_megakernel), dim3(grid), dim3(kBThreads), args,
                                     kBSmem, st);
}

cudaError_t prepare_bwd_megakernel() {
  return cudaFuncSetAttribute(bwd_megakernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kBSmem);
}

}  // namespace moe
