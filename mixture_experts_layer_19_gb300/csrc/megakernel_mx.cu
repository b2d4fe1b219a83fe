// megakernel_mx.cu -- the MXFP8 forward expert pipeline as one persistent,
// device-driven kernel over the ring token buffer: same schedule and hand-off
// counters as the bf16 megakernel (megakernel.cu), with the MXFP8 datapath of
// gemm_mx.cuh.
//
// The tokens are quantised along d once per token (all SMs, just before this
// kernel); mover CTAs then pull each routed row's E4M3 bytes and scale words
// into its ring slot -- MXFP8 activation quantisation in the dispatch datapath
// (kucoin page "Cursor's MoK réalise une amélioration des performances de
// 2,37x sur NVIDIA GB300 NVL72", section 02), done k times less often than a
// per-row quantisation and leaving the movers plain copies.
// G1 tiles run the block-scaled [a|b] GEMM, SwiGLU, and re-quantise h along F
// straight into the slot; G2 tiles run the block-scaled down GEMM from the
// slot.  Eight epilogue warps per compute CTA each bump the hand-off counters
// once per tile (targets are 8 x tiles).
// FUSED (the one-launch forward): the kernel also quantises the tokens,
// routes them, lays out the sorted rows and cuts the minibatches (three
// bounded grid barriers; megakernel_common.cuh) and combines each token's
// 256-column blocks as their last rows land, so the whole MXFP8 forward is
// one launch.
#include "gemm_mx.cuh"
#include "kernels.h"
#include "megakernel.cuh"
#include "megakernel_common.cuh"
#include "mx.cuh"

#include <cstdio>
#include <cstring>

namespace moe {

constexpr int kMxMegaStages = 3;
constexpr int kQueueMx = 4;
constexpr int kMxMegaThreads = 64 + 32 * 8;
constexpr int kMxMegaStaging = 2 * kStageChunk + 1024;  // a, b (bf16) and h (E4M3) chunks per warp
constexpr int kMxMegaSfStage = 1536;
constexpr int kMxMegaStagingOff = (kMxMegaStages * (kStageBytes + kMxMegaSfStage) + 1023) / 1024 * 1024;
constexpr int kMxMegaSmem = kMxMegaStagingOff + 8 * kMxMegaStaging + 1024 + 512;

__device__ void mx_mover_loop(const MegaMxArgs& g, int nmb, int* abort_flag) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int nwarps = blockDim.x >> 5;
  const int nt1 = g.F / 128, nt2 = g.d / BN;
  const int kblocks = g.d / 32;
  WaitCtl wc{g.status, abort_flag, g.timeout_ns};
  for (int mb = 0; mb < nmb; ++mb) {
    if (threadIdx.x == 0 && mb >= g.slots) {
      const int prev = mb - g.slots;
      const int target = 8 * (g.mb_start[prev + 1] - g.mb_start[prev]) * (nt1 + nt2);
      wait_counter_geq(g.mb_done + prev, target, wc);
    }
    __syncthreads();
    if (*abort_flag) return;
    const int row_base = g.mb_start[mb] * BM;
    const int nrows = (g.mb_start[mb + 1] - g.mb_start[mb]) * BM;
    const int slot_base = (mb % g.slots) * g.slot_rows;
    // copy the token's E4M3 row (16-byte vectors) and its scale words (4
    // consecutive blocks share one 32-bit word of an atom) into the ring row
    const int nvec = g.d / 16, nwords = kblocks / 4;
    for (int i = blockIdx.x * nwarps + warp; i < nrows; i += g.movers * nwarps) {
      const int src = g.perm_src[row_base + i];
      const int rr = slot_base + i;   // ring row
      uint4* qdst = reinterpret_cast<uint4*>(g.ring_xq + (size_t)rr * g.d);
      const size_t rw = (size_t)(rr & 31) * 16 + (size_t)((rr >> 5) & 3) * 4;
      if (src < 0) {
        for (int v = lane; v < nvec; v += 32) qdst[v] = make_uint4(0, 0, 0, 0);
        for (int j = lane; j < nwords; j += 32)
          *reinterpret_cast<uint32_t*>(g.ring_xs + ((size_t)(rr >> 7) * nwords + j) * 512 + rw) = 0u;
        continue;
      }
      const int t = src / g.k;
      const uint4* qsrc = reinterpret_cast<const uint4*>(g.xq + (size_t)t * g.d);
      for (int v = lane; v < nvec; v += 32) qdst[v] = __ldg(qsrc + v);
      const size_t tw = (size_t)(t & 31) * 16 + (size_t)((t >> 5) & 3) * 4;
      for (int j = lane; j < nwords; j += 32)
        *reinterpret_cast<uint32_t*>(g.ring_xs + ((size_t)(rr >> 7) * nwords + j) * 512 + rw) =
            __ldg(reinterpret_cast<const uint32_t*>(g.xs + ((size_t)(t >> 7) * nwords + j) * 512 + tw));
    }
    __syncthreads();
    if (threadIdx.x == 0) {
      __threadfence();
      fence_proxy_async_global();
      red_release_gpu_add(g.gathered + mb, 1);
    }
  }
}

template <bool FUSED>
__global__ void __launch_bounds__(kMxMegaThreads, 1) fwd_megakernel_mx(const __grid_constant__ MegaMxArgs g) {
  constexpr int S = kMxMegaStages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* sf_base = smem + S * kStageBytes;
  uint8_t* staging_base = smem + kMxMegaStagingOff;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging_base + 8 * kMxMegaStaging);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = tfull + 1;
  uint64_t* qfull = tempty + 1;
  uint64_t* qempty = qfull + kQueueMx;
  Item* queue = reinterpret_cast<Item*>(qempty + kQueueMx);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(queue + kQueueMx);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);
  int* sync_flag = abort_flag + 1;

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) *abort_flag = 0;
  __syncthreads();
  if (FUSED) {
    // every token quantised along d once (the quant_rows_kernel arithmetic),
    // then routing, layout and the minibatch plan
    const int kblocks = g.d >> 5;
    const int64_t nblk = (int64_t)g.T * kblocks;
    for (int64_t i = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; i < nblk; i += (int64_t)gridDim.x * blockDim.x) {
      const int64_t r = i / kblocks;
      const int kb = (int)(i - r * kblocks);
      float v[32];
      load_bf16x32_f(g.Xtok + r * g.d + kb * 32, v);
      quant_block_store(v, g.xq + r * g.d + kb * 32, g.xs + sf_atom_offset(r, kb, kblocks));
    }
    WaitCtl wca{g.status, abort_flag, g.timeout_ns};
    if (!route_in_kernel(g, reinterpret_cast<int*>(stage_base), wca, sync_flag)) {
      if (threadIdx.x == 0) fused_exit(g);
      return;
    }
  }
  const int nmb = *g.n_mb;
  if ((int)blockIdx.x < g.movers) {
    mx_mover_loop(g, nmb, abort_flag);
    if (FUSED) {
      __syncthreads();
      if (threadIdx.x == 0) fused_exit(g);
    }
    return;
  }
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 8);
    for (int q = 0; q < kQueueMx; ++q) {
      mbar_init(&qfull[q], 1);
      mbar_init(&qempty[q], 9);  // MMA thread + 8 epilogue warps
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
  const int nt1 = g.F / 128;
  const int total = g.phase_start[2 * nmb];

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------- claimer + producer
      const uint64_t pol_w = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      uint32_t s = 0, ph = 0, qi = 0, qph = 0, issued_mask = 0, last_par = 0;
      bool ok = true;
      while (ok) {
        const int c = atomicAdd(g.claim, 1);
        Item it;
        if (c >= total) {
          it.kind = -1;
        } else {
          it = decode_claim(g, nmb, c);
          ok = it.kind == 0 ? wait_counter_geq(g.gathered + it.mb, g.movers, wc)
                            : wait_counter_geq(g.g1_done + it.gt, 8 * nt1, wc);
          fence_proxy_async_global();
          if (!ok) it.kind = -1;
        }
        if (!mbar_wait(&qempty[qi], qph ^ 1, wc)) break;
        queue[qi] = it;
        mbar_arrive(&qfull[qi]);
        if (++qi == kQueueMx) { qi = 0; qph ^= 1; }
        if (it.kind < 0) break;
        const int K = it.kind == 0 ? g.d : g.F;
        const int kg = K / kMxBK;
        const int nkb = kg;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kStageBytes + kMxMegaSfStage);
          uint8_t* sa = stage_base + s * kStageBytes;
          uint8_t* sb = sa + kABytes;
          uint8_t* ssf = sf_base + s * kMxMegaSfStage;
          const int k0 = kb * kMxBK;
          const uint8_t* asf = (it.kind == 0 ? g.ring_xs : g.ring_hs) +
                               ((size_t)(it.ring_row0 >> 7) * kg + kb) * 512;
          if (it.kind == 0) {
            const int brow = it.e * g.F + it.nt * 128;
            tma_load_2d(sa, &g.mapXr, k0, it.ring_row0, &full[s], pol_a);
            tma_load_2d(sb, &g.mapWg, k0, brow, &full[s], pol_w);
            tma_load_2d(sb + kBBytes / 2, &g.mapWu, k0, brow, &full[s], pol_w);
            bulk_load_1d(ssf, asf, 512, &full[s]);
            bulk_load_1d(ssf + 512, g.wgs + ((size_t)(brow >> 7) * kg + kb) * 512, 512, &full[s]);
            bulk_load_1d(ssf + 1024, g.wus + ((size_t)(brow >> 7) * kg + kb) * 512, 512, &full[s]);
          } else {
            const int brow = it.e * g.d + it.nt * BN;
            tma_load_2d(sa, &g.mapHr, k0, it.ring_row0, &full[s], pol_a);
            tma_load_2d(sb, &g.mapWd, k0, brow, &full[s], pol_w);
            bulk_load_1d(ssf, asf, 512, &full[s]);
            bulk_load_1d(ssf + 512, g.wds + ((size_t)(brow >> 7) * kg + kb) * 512, 512, &full[s]);
            bulk_load_1d(ssf + 1024, g.wds + ((size_t)((brow >> 7) + 1) * kg + kb) * 512, 512, &full[s]);
          }
          issued_mask |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == S) { s = 0; ph ^= 1; }
        }
      }
      if (!ok) {
        for (int st = 0; st < S; ++st) {
          if (!(issued_mask & (1u << st))) continue;
          const uint32_t par = (last_par >> st) & 1u;
          for (uint64_t t0 = globaltimer_ns(); !mbar_try_wait(&full[st], par);)
            if (globaltimer_ns() - t0 > 50000000ull) break;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------- MMA issuer (one accumulator)
      uint32_t s = 0, ph = 0, aph = 0, qi = 0, qph = 0;
      for (;;) {
        if (!mbar_wait(&qfull[qi], qph, wc)) break;
        const Item it = queue[qi];
        mbar_arrive(&qempty[qi]);
        if (++qi == kQueueMx) { qi = 0; qph ^= 1; }
        if (it.kind < 0) break;
        if (!mbar_wait(tempty, aph ^ 1, wc)) break;
        tc_fence_after();
        const int nkb = (it.kind == 0 ? g.d : g.F) / kMxBK;
        bool ok = true;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
          const uint32_t ssf = smem_u32(sf_base + s * kMxMegaSfStage);
          const uint32_t sfa_t = tmem_base + BN + s * 16;
          const uint32_t sfb_t = sfa_t + 8;
          tmem_cp_32x128_x4(sfa_t, sdesc_plain(ssf));
          tmem_cp_32x128_x4(sfb_t, sdesc_plain(ssf + 512));
          tmem_cp_32x128_x4(sfb_t + 4, sdesc_plain(ssf + 1024));
#pragma unroll
          for (int kk = 0; kk < kMxBK / 32; ++kk)
            umma_mxf8(tmem_base, sdesc_sw128(sa + kk * 32, 16, 1024), sdesc_sw128(sb + kk * 32, 16, 1024),
                      idesc_mxf8(BM, BN, 0, 0, kk), sfa_t, sfb_t, (kb | kk) != 0 ? 1u : 0u);
          umma_commit(&empty[s]);
          if (++s == S) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        umma_commit(tfull);
        aph ^= 1;
      }
    }
  } else {
    // ------------------------------------------------- epilogue (8 warps)
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    uint8_t* stg = staging_base + (warp - 2) * kMxMegaStaging;
    uint32_t aph = 0, qi = 0, qph = 0;
    for (;;) {
      if (!mbar_wait(&qfull[qi], qph, wc)) break;
      const Item it = queue[qi];
      __syncwarp();
      if (lane == 0) mbar_arrive(&qempty[qi]);
      if (++qi == kQueueMx) { qi = 0; qph ^= 1; }
      if (it.kind < 0) break;
      if (!mbar_wait(tfull, aph, wc)) break;
      tc_fence_after();
      const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16);
      const int srow = it.gt * BM + 32 * q;
      const int rrow = it.ring_row0 + 32 * q;
      uint32_t acc[4][32];
      if (it.kind == 0) {
        tmem_ld32(tb + half * 64, acc[0]);
        tmem_ld32(tb + half * 64 + 32, acc[1]);
        tmem_ld32(tb + 128 + half * 64, acc[2]);
        tmem_ld32(tb + 128 + half * 64 + 32, acc[3]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tb + half * 128 + c * 32, acc[c]);
      }
      tmem_ld_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(tempty);
      aph ^= 1;
      if (it.kind == 0) {
        uint32_t sfw = 0;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float a[32], b[32], h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = __uint_as_float(acc[c2][i]);
            b[i] = __uint_as_float(acc[2 + c2][i]);
            h[i] = a[i] * sigmoidf_(a[i]) * b[i];
          }
          const int X = mx_block_exponent(amax32(h));
          uint32_t hq[8];
          mx_encode32(h, X, hq);
          sfw |= (uint32_t)(X + 127) << (8 * c2);
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row(stg, lane, a);
          stage_row(stg + kStageChunk, lane, b);
          stage_row_fp8(stg + 2 * kStageChunk, lane, hq);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int col = it.nt * 128 + half * 64 + c2 * 32;
            tma_store_2d(&g.mapABSt, stg, col, srow);
            tma_store_2d(&g.mapABSt, stg + kStageChunk, g.F + col, srow);
            tma_store_2d(&g.mapHrSt, stg + 2 * kStageChunk, col, rrow);
            bulk_commit();
          }
        }
        const int kb = it.nt * 4 + half * 2;  // this warp's two scale blocks of h (K = F)
        *reinterpret_cast<uint16_t*>(g.ring_hs + sf_atom_offset(rrow + lane, kb, g.F / 32)) = (uint16_t)sfw;
        __threadfence();
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(acc[c][i]);
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row(stg, lane, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&g.mapYsSt, stg, it.nt * BN + half * 128 + c * 32, srow);
            bulk_commit();
          }
        }
      }
      __syncwarp();
      if (lane == 0) {
        bulk_wait<0>();
        fence_proxy_async_global();
        if (it.kind == 0) red_release_gpu_add(g.g1_done + it.gt, 1);
        red_release_gpu_add(g.mb_done + it.mb, 1);
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

cudaError_t launch_fwd_megakernel_mx(const MegaMxArgs& a, int grid, bool fused, cudaStream_t st) {
  void* args[] = {const_cast<MegaMxArgs*>(&a)};
  const void* fn = fused ? reinterpret_cast<const void*>(fwd_megakernel_mx<true>)
                         : reinterpret_cast<const void*>(fwd_megakernel_mx<false>);
  const cudaError_t e = cudaLaunchCooperativeKernel(fn, dim3(grid), dim3(kMxMegaThreads), args, kMxMegaSmem, st);
  if (e == cudaErrorCooperativeLaunchTooLarge) {
    // say why the grid cannot be co-resident
    int per_sm = -1;
    cudaFuncAttributes fa;
    memset(&fa, 0, sizeof(fa));
    cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, fn, kMxMegaThreads, kMxMegaSmem);
    cudaFuncGetAttributes(&fa, fn);
    char buf[256];
    snprintf(buf, sizeof(buf),
             "cooperative grid %d: %d CTA(s) per SM fit (registers %d, static smem %zu, dynamic smem %d of max %d, "
             "local %zu B, max threads %d)",
             grid, per_sm, fa.numRegs, fa.sharedSizeBytes, kMxMegaSmem, fa.maxDynamicSharedSizeBytes,
             fa.localSizeBytes, fa.maxThreadsPerBlock);
    set_error_detail(buf);
  }
  return e;
}

cudaError_t prepare_fwd_megakernel_mx() {
  cudaError_t e =
      cudaFuncSetAttribute(fwd_megakernel_mx<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxMegaSmem);
  if (e != cudaSuccess) return e;
  return cudaFuncSetAttribute(fwd_megakernel_mx<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, kMxMegaSmem);
}

}  // namespace moe
