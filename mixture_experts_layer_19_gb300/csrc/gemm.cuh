// gemm.cuh -- persistent tcgen05 grouped GEMM for the MoE expert contractions.
//
// One CTA per SM (192 or 320 threads):
//   warp 0      TMA producer: streams 64-deep K slices of A and B into a
//               4-stage shared-memory ring (128-byte swizzle).
//   warp 1      TMEM owner + single-thread UMMA issuer (tcgen05.mma
//               kind::f16, M=128, N=256, K=16, fp32 accumulate in TMEM).
//   warps 2..   epilogue (4 warps, or 8 for single-output kinds: two per TMEM
//               lane quadrant, each on half the columns): TMEM -> registers
//               -> fused math -> bf16 -> 64-byte-swizzled staging -> TMA store.
// Two 256-column TMEM accumulators let the epilogue of tile i overlap the
// main loop of tile i+1.  Tiles are handed out statically (tile = CTA id +
// j * gridDim.x).  Every tile accumulates its K range in one fixed order, so
// the result does not depend on scheduling: bitwise deterministic.
//
// The six contractions of the layer (sorted/padded row space, 128-row expert
// segments; "rows" are (token, slot) pairs sorted by expert):
//   kUp     [a|b] = Xg . [Wg;Wu]^T      A K-major, B K-major   (+ SwiGLU epilogue)
//   kDown   Ys    = H . Wd^T            A K-major, B K-major
//   kBwdU   u     = dYg . Wd            A K-major, B MN-major  (+ SwiGLU backward epilogue)
//   kBwdX   dXs   = dAB . [Wg;Wu]       A K-major, B MN-major
//   kWgradD dWd   = dYg^T . (w h)       A MN-major, B MN-major (K = expert's rows)
//   kWgradGU [dWg;dWu] = dAB^T . Xg     A MN-major, B MN-major (K = expert's rows)
// and the dense router GEMM in front of the layer (tiles over T or E, no experts):
//   kRouter   logits = X . Wr^T         A K-major, B K-major   (fp32 output)
//   kRouterDX dX    += dlogits . Wr     A K-major, B MN-major  (adds into bf16 dX)
//   kRouterDW dWr    = dlogits^T . X    A MN-major, B MN-major (K = T tokens)
#pragma once
#include "ptx.cuh"

namespace moe {

constexpr int BM = 128;           // tile rows (UMMA M)
constexpr int BN = 256;           // tile cols (UMMA N)
constexpr int BK = 64;            // K slice per pipeline stage (128 bytes of bf16)
constexpr int kStages = 4;
constexpr int kGemmThreadsMax = 320;  // 2 control warps + up to 8 epilogue warps
constexpr int kABytes = BM * BK * 2;             // 16 KB
constexpr int kBBytes = BN * BK * 2;             // 32 KB
constexpr int kStageBytes = kABytes + kBBytes;   // 48 KB
constexpr int kStageChunk = 32 * 32 * 2;         // one epilogue staging tile: 32 rows x 32 bf16

enum GemmKind { kUp = 0, kDown = 1, kBwdU = 2, kBwdX = 3, kWgradD = 4, kWgradGU = 5,
                kRouter = 6, kRouterDX = 7, kRouterDW = 8 };

template <int KIND>
struct KindTraits {
  static constexpr bool a_mn = (KIND == kWgradD || KIND == kWgradGU || KIND == kRouterDW);
  static constexpr bool b_mn = (KIND != kUp && KIND != kDown && KIND != kRouter);
  static constexpr bool grouped = (KIND <= kBwdX);          // tiles follow expert segments
  static constexpr bool dense = (KIND >= kRouter);          // plain M x N tiles (router GEMM)
  static constexpr int n_out = (KIND == kUp || KIND == kBwdU) ? 3 : 1;
  // staging buffers per epilogue warp: the weight gradients keep one, so each
  // warp has at most one dW store reading shared memory (measured: more dW
  // store bytes in flight slow the operand loads more than they gain)
  static constexpr bool wgrad = (KIND == kWgradD || KIND == kWgradGU);
  static constexpr int n_buf = (n_out == 3 || wgrad) ? 1 : 2;
  // single-output epilogues are store-bound (weight gradients write 64 KB per
  // tile): two warps per TMEM lane quadrant, each taking half of the columns
  static constexpr int epi_warps = (n_out == 1) ? 8 : 4;
  static constexpr int threads = 64 + 32 * epi_warps;
  static constexpr int staging_per_warp = n_out * n_buf * kStageChunk;
  static constexpr int smem_bytes =
      kStages * kStageBytes + epi_warps * staging_per_warp + 1024 /*align*/ + 256 /*bars*/;
};

struct GemmArgs {
  CUtensorMap mapA;    // operand A loads
  CUtensorMap mapB0;   // operand B loads (Wg / Wd / wH / Xg)
  CUtensorMap mapB1;   // second B source (Wu) where the B operand is [Wg;Wu]
  CUtensorMap mapO0;   // output stores
  CUtensorMap mapO1;
  CUtensorMap mapO2;
  const int32_t* poff;       // [E+1] padded segment starts (rows)
  const int32_t* mtile_off;  // [E+1] prefix sum of 128-row tiles per expert
  const __nv_bfloat16* ab;   // kBwdU: saved [R, 2F] pre-activations a|b
  const int32_t* perm_src;   // kBwdU: flat pair of each sorted row (-1 = padding)
  const float* wts;          // kBwdU: gate weights [T*k]
  float* dgp;                // kBwdU: [R, F/256] partial <u, h> per N tile
  float* out_f32;            // kRouter: logits [T, E] (with ksplit > 1: partials [ksplit, T, E])
  float* part_f32;           // kRouterDW with ksplit > 1: fp32 partials [ksplit, E, d]
  int ksplit;                // router kinds kRouter / kRouterDW: K range split over this many tiles (0 / 1: none)
  __nv_bfloat16* io_bf16;    // kRouterDX: dX [T, d], read and written
  int32_t* status;
  uint64_t timeout_ns;
  int E, d, F;
  int T;                     // dense kinds: tokens
  int stall;                 // fault-injection test hook: the producer issues nothing, so the
                             //   consumers' bounded waits expire (MOE_DEBUG_STALL_TEST)
};

struct Tile {
  int e, mt, nt;   // expert, M tile, N tile
  int row0;        // first sorted row (grouped) / first output row inside the expert (wgrad)
  int nkb;         // K slices
  int kbase;       // first sorted row of the K range (wgrad); first K of the split (router kinds)
  int split;       // router kinds: which K split this tile's partial sums belong to
};

// The helpers below take any argument struct with E, d, F, poff, mtile_off
// (GemmArgs here, MxArgs for the MXFP8 kernel).
template <int KIND, class G>
__device__ __forceinline__ int n_tiles_n(const G& g) {
  if (KIND == kUp) return g.F / 128;
  if (KIND == kDown || KIND == kBwdX) return g.d / BN;
  if (KIND == kBwdU) return g.F / BN;
  if (KIND == kWgradD) return g.F / BN;
  return g.d / BN;  // kWgradGU
}
template <int KIND, class G>
__device__ __forceinline__ int n_tiles_m_wgrad(const G& g) {
  return KIND == kWgradD ? g.d / BM : (2 * g.F) / BM;
}
template <int KIND, class G>
__device__ __forceinline__ int k_blocks_grouped(const G& g) {
  if (KIND == kUp || KIND == kBwdU) return g.d / BK;
  if (KIND == kDown) return g.F / BK;
  return (2 * g.F) / BK;  // kBwdX
}

// Dense (router) kinds: M = T (kRouter, kRouterDX) or E (kRouterDW); N = E
// (kRouter) or d; K = d (kRouter), E (kRouterDX) or T (kRouterDW).  Ragged
// edges read as zeros (TMA out-of-bounds fill) and are not stored.
template <int KIND, class G>
__device__ __forceinline__ int dense_mt(const G& g) {
  return ((KIND == kRouterDW ? g.E : g.T) + BM - 1) / BM;
}
template <int KIND, class G>
__device__ __forceinline__ int dense_nt(const G& g) {
  return KIND == kRouter ? (g.E + BN - 1) / BN : g.d / BN;
}
template <int KIND, class G>
__device__ __forceinline__ int dense_nkb(const G& g) {
  return ((KIND == kRouter ? g.d : KIND == kRouterDX ? g.E : g.T) + BK - 1) / BK;
}

template <int KIND, class G>
__device__ __forceinline__ int total_tiles(const G& g) {
  if constexpr (KindTraits<KIND>::dense) return dense_mt<KIND>(g) * dense_nt<KIND>(g) * max(1, g.ksplit);
  if (KindTraits<KIND>::grouped) return g.mtile_off[g.E] * n_tiles_n<KIND>(g);
  return g.E * n_tiles_m_wgrad<KIND>(g) * n_tiles_n<KIND>(g);
}

template <int KIND, class G>
__device__ __forceinline__ Tile decode_tile(const G& g, int tile) {
  Tile t;
  t.split = 0;
  if constexpr (KindTraits<KIND>::dense) {  // (split, n, m) with m fastest, split slowest
    const int MT = dense_mt<KIND>(g), NT = dense_nt<KIND>(g);
    const int S = max(1, g.ksplit);
    t.split = tile / (MT * NT);
    const int local = tile - t.split * MT * NT;
    t.e = 0;
    t.nt = local / MT;
    t.mt = local - t.nt * MT;
    t.row0 = t.mt * BM;
    const int nkb = dense_nkb<KIND>(g), base = nkb / S, rem = nkb % S;
    t.nkb = base + (t.split < rem ? 1 : 0);
    t.kbase = (t.split * base + min(t.split, rem)) * BK;
    return t;
  }
  const int NT = n_tiles_n<KIND>(g);
  if (KindTraits<KIND>::grouped) {
    // expert e owns tiles [mtile_off[e]*NT, mtile_off[e+1]*NT), ordered (n, m) with m fastest
    const int gidx = tile / NT;
    int lo = 0, hi = g.E;  // find last e with mtile_off[e] <= gidx
    while (hi - lo > 1) {
      int mid = (lo + hi) >> 1;
      if (__ldg(g.mtile_off + mid) <= gidx) lo = mid; else hi = mid;
    }
    t.e = lo;
    const int m0 = __ldg(g.mtile_off + lo);
    const int mte = __ldg(g.mtile_off + lo + 1) - m0;
    const int local = tile - m0 * NT;
    t.nt = local / mte;
    t.mt = local - t.nt * mte;
    t.row0 = __ldg(g.poff + lo) + t.mt * BM;
    t.nkb = k_blocks_grouped<KIND>(g);
    t.kbase = 0;
  } else {
    const int MT = n_tiles_m_wgrad<KIND>(g);
    const int per = MT * NT;
    t.e = tile / per;
    const int local = tile - t.e * per;
    t.nt = local / MT;
    t.mt = local - t.nt * MT;
    t.row0 = t.mt * BM;
    t.kbase = __ldg(g.poff + t.e);
    t.nkb = (__ldg(g.poff + t.e + 1) - t.kbase) / BK;
  }
  return t;
}

// ----------------------------------------------------------------------------
// Producer: TMA loads of one K slice of A and B into a stage.
// ----------------------------------------------------------------------------
template <int KIND>
__device__ __forceinline__ void load_stage(const GemmArgs& g, const Tile& t, int kb, uint8_t* sa, uint8_t* sb,
                                           uint64_t* bar, uint64_t pol_w, uint64_t pol_a) {
  const int k0 = kb * BK + (KindTraits<KIND>::dense ? t.kbase : 0);
  if (KIND == kUp) {
    tma_load_2d(sa, &g.mapA, k0, t.row0, bar, pol_a);
    tma_load_2d(sb, &g.mapB0, k0, t.e * g.F + t.nt * 128, bar, pol_w);
    tma_load_2d(sb + kBBytes / 2, &g.mapB1, k0, t.e * g.F + t.nt * 128, bar, pol_w);
  } else if (KIND == kDown) {
    tma_load_2d(sa, &g.mapA, k0, t.row0, bar, pol_a);
    tma_load_2d(sb, &g.mapB0, k0, t.e * g.d + t.nt * BN, bar, pol_w);
  } else if (KIND == kBwdU) {
    tma_load_2d(sa, &g.mapA, k0, t.row0, bar, pol_a);
#pragma unroll
    for (int j = 0; j < 4; ++j)
      tma_load_2d(sb + j * 8192, &g.mapB0, t.nt * BN + j * 64, t.e * g.d + k0, bar, pol_w);
  } else if (KIND == kBwdX) {
    tma_load_2d(sa, &g.mapA, k0, t.row0, bar, pol_a);
    const bool up = k0 >= g.F;
    const CUtensorMap* mb = up ? &g.mapB1 : &g.mapB0;
    const int krow = t.e * g.F + (up ? k0 - g.F : k0);
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, mb, t.nt * BN + j * 64, krow, bar, pol_w);
  } else if (KIND == kRouter) {
    tma_load_2d(sa, &g.mapA, k0, t.row0, bar, pol_a);         // X rows
    tma_load_2d(sb, &g.mapB0, k0, t.nt * BN, bar, pol_w);     // Wr rows
  } else if (KIND == kRouterDX) {
    tma_load_2d(sa, &g.mapA, k0, t.row0, bar, pol_a);         // dlogits rows (bf16), K = E
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &g.mapB0, t.nt * BN + j * 64, k0, bar, pol_w);  // Wr
  } else if (KIND == kRouterDW) {                              // K = tokens
#pragma unroll
    for (int j = 0; j < 2; ++j) tma_load_2d(sa + j * 8192, &g.mapA, t.row0 + j * 64, k0, bar, pol_a);     // dlogits
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &g.mapB0, t.nt * BN + j * 64, k0, bar, pol_a);  // X
  } else {  // wgrad: both operands MN-major, K = sorted rows of expert e
    const int kr = t.kbase + k0;
#pragma unroll
    for (int j = 0; j < 2; ++j) tma_load_2d(sa + j * 8192, &g.mapA, t.row0 + j * 64, kr, bar, pol_a);
#pragma unroll
    for (int j = 0; j < 4; ++j) tma_load_2d(sb + j * 8192, &g.mapB0, t.nt * BN + j * 64, kr, bar, pol_a);
  }
}

// ----------------------------------------------------------------------------
// Epilogue helpers.
// ----------------------------------------------------------------------------
// Write 32 fp32 values of this lane's row into a 32x32 bf16 staging tile laid
// out for a 64-byte-swizzled TMA store (16-byte chunk c of row r lives at
// chunk c ^ ((r >> 1) & 3)).
__device__ __forceinline__ void stage_row(uint8_t* buf, int lane, const float* v) {
  uint32_t p[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) p[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 q = make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
    *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ sw) << 4)) = q;
  }
}

// The same for 32 values already packed as 16 bf16 pairs.
__device__ __forceinline__ void stage_row_packed(uint8_t* buf, int lane, const uint32_t* p) {
  const int sw = (lane >> 1) & 3;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 q = make_uint4(p[4 * c], p[4 * c + 1], p[4 * c + 2], p[4 * c + 3]);
    *reinterpret_cast<uint4*>(buf + lane * 64 + ((c ^ sw) << 4)) = q;
  }
}

__device__ __forceinline__ void load_bf16x32(const __nv_bfloat16* src, float* v) {
  const uint4* s = reinterpret_cast<const uint4*>(src);
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    uint4 q = __ldg(s + c);
    const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&w[i]);
      float2 f = __bfloat1622float2(b);
      v[8 * c + 2 * i] = f.x;
      v[8 * c + 2 * i + 1] = f.y;
    }
  }
}

__device__ __forceinline__ float sigmoidf_(float a) { return 1.0f / (1.0f + __expf(-a)); }

// ----------------------------------------------------------------------------
// The kernel.
// ----------------------------------------------------------------------------
template <int KIND>
__global__ void __launch_bounds__(KindTraits<KIND>::threads, 1) gemm_kernel(const __grid_constant__ GemmArgs g) {
  using TR = KindTraits<KIND>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* staging_base = smem + kStages * kStageBytes;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging_base + TR::epi_warps * TR::staging_per_warp);
  uint64_t* full = bars;
  uint64_t* empty = bars + kStages;
  uint64_t* tfull = bars + 2 * kStages;
  uint64_t* tempty = bars + 2 * kStages + 2;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * kStages + 4);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(&tfull[a], 1);
      mbar_init(&tempty[a], TR::epi_warps);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&g.mapA);
    tma_prefetch_desc(&g.mapB0);
    if (KIND == kUp || KIND == kBwdX) tma_prefetch_desc(&g.mapB1);
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
  // static schedule: tile w = blockIdx.x + j * gridDim.x
  const int nwork = total_tiles<KIND>(g);
  const int w0 = (int)blockIdx.x;
  const int wstep = (int)gridDim.x;

  if (warp == 0) {
    if (lane == 0) {
      // ---------------------------------------------------------- producer
      // L2 policies, chosen by measurement at d=7168, F=2048, E=256, top-8.
      // Grouped GEMMs: a weight tile is read by every M tile of its expert,
      // by CTAs that drift apart in time; evict_last keeps it for the late
      // ones (evict_first cost ~1 GB of DRAM re-reads and ~0.1 ms per launch).
      // Weight-gradient GEMMs read two activation operands, both re-read by
      // every output tile of the expert (pol_a, evict_last).
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_a = policy_evict_last();
      uint32_t s = 0, ph = 0;
      uint32_t issued_mask = 0, last_par = 0;
      bool ok = true;
      for (int w = w0; w < nwork && ok && !g.stall; w += wstep) {
        const Tile t = decode_tile<KIND>(g, w);
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kStageBytes);
          uint8_t* sa = stage_base + s * kStageBytes;
          load_stage<KIND>(g, t, kb, sa, sa + kABytes, &full[s], pol_w, pol_a);
          issued_mask |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
      }
      if (!ok) {
        // abort: let every issued copy land before the CTA may exit
        WaitCtl drain{nullptr, abort_flag, 50000000ull};
        for (int st = 0; st < kStages; ++st) {
          if (!(issued_mask & (1u << st))) continue;
          const uint32_t par = (last_par >> st) & 1u;
          for (uint64_t t0 = globaltimer_ns(); !mbar_try_wait(&full[st], par);)
            if (globaltimer_ns() - t0 > drain.timeout_ns) break;
        }
      }
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ---------------------------------------------------------- MMA issuer
      constexpr uint32_t idesc = idesc_bf16(BM, BN, TR::a_mn ? 1 : 0, TR::b_mn ? 1 : 0);
      uint32_t s = 0, ph = 0, acc = 0, aph = 0;
      bool ok = true;
      for (int w = w0; w < nwork && ok; w += wstep) {
        const Tile t = decode_tile<KIND>(g, w);
        if (t.nkb == 0) continue;
        if (!mbar_wait(&tempty[acc], aph ^ 1, wc)) break;
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + acc * BN;
        for (int kb = 0; kb < t.nkb; ++kb) {
          if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk) {
            const uint64_t ad = TR::a_mn ? sdesc_sw128(sa + kk * 2048, 8192, 1024) : sdesc_sw128(sa + kk * 32, 16, 1024);
            const uint64_t bd = TR::b_mn ? sdesc_sw128(sb + kk * 2048, 8192, 1024) : sdesc_sw128(sb + kk * 32, 16, 1024);
            umma_bf16(d_tmem, ad, bd, idesc, (kb | kk) != 0 ? 1u : 0u);
          }
          umma_commit(&empty[s]);
          if (++s == kStages) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        umma_commit(&tfull[acc]);
        acc ^= 1;
        if (acc == 0) aph ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint8_t* stg = staging_base + (warp - 2) * TR::staging_per_warp;
    uint32_t acc = 0, aph = 0;
    int chunk_ctr = 0;
    for (int w = w0; w < nwork; w += wstep) {
      const Tile t = decode_tile<KIND>(g, w);
      const bool has_acc = t.nkb > 0;
      if (has_acc) {
        if (!mbar_wait(&tfull[acc], aph, wc)) break;
        tc_fence_after();
      }
      const uint32_t tbase = tmem_base + ((uint32_t)(32 * q) << 16) + acc * BN;
      const int rowq = t.row0 + 32 * q;   // first row of this warp's 32-row slab
      if (KIND == kUp) {
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
            const int col = t.nt * 128 + c * 32;
            tma_store_2d(&g.mapO0, stg, col, rowq);
            tma_store_2d(&g.mapO0, stg + kStageChunk, g.F + col, rowq);
            tma_store_2d(&g.mapO1, stg + 2 * kStageChunk, col, rowq);
            bulk_commit();
          }
        }
      } else if (KIND == kBwdU) {
        const int r = rowq + lane;
        const int src = __ldg(g.perm_src + r);
        const float wr = src >= 0 ? __ldg(g.wts + src) : 0.0f;
        const __nv_bfloat16* abrow = g.ab + (size_t)r * (2 * g.F);
        float dgacc = 0.0f;
#pragma unroll 1
        for (int c = 0; c < 8; ++c) {
          uint32_t ru[32];
          tmem_ld32(tbase + c * 32, ru);
          const int col = t.nt * BN + c * 32;
          float a[32], b[32];
          load_bf16x32(abrow + col, a);
          load_bf16x32(abrow + g.F + col, b);
          tmem_ld_wait();
          if (c == 7) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          float da[32], db[32], wh[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float u = __uint_as_float(ru[i]);
            const float sa = sigmoidf_(a[i]);
            const float sl = a[i] * sa;              // silu(a)
            const float hh = sl * b[i];              // h
            dgacc = fmaf(u, hh, dgacc);              // <u, h> in column order
            const float dh = wr * u;
            da[i] = dh * b[i] * sa * (1.0f + a[i] * (1.0f - sa));
            db[i] = dh * sl;
            wh[i] = wr * hh;
          }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row(stg, lane, da);
          stage_row(stg + kStageChunk, lane, db);
          stage_row(stg + 2 * kStageChunk, lane, wh);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&g.mapO0, stg, col, rowq);
            tma_store_2d(&g.mapO0, stg + kStageChunk, g.F + col, rowq);
            tma_store_2d(&g.mapO1, stg + 2 * kStageChunk, col, rowq);
            bulk_commit();
          }
        }
        g.dgp[(size_t)r * (g.F / BN) + t.nt] = dgacc;
      } else if (KIND == kRouter || KIND == kRouterDX) {
        // one token row per lane: logits stored as fp32, or dX += tile (fp32
        // add, one bf16 rounding); rows past T and columns past E are skipped
        constexpr int kChunks = 8 / (TR::epi_warps / 4);
        const int c0 = ((warp - 2) >> 2) * kChunks;
        const int row = rowq + lane;
#pragma unroll 1
        for (int c = c0; c < c0 + kChunks; ++c) {
          uint32_t rv[32];
          tmem_ld32(tbase + c * 32, rv);
          tmem_ld_wait();
          if (c == c0 + kChunks - 1) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&tempty[acc]);
          }
          const int col0 = t.nt * BN + c * 32;
          if (row < g.T) {
            if (KIND == kRouter) {
              float4* dst = reinterpret_cast<float4*>(g.out_f32 + ((size_t)t.split * g.T + row) * g.E + col0);
              const int nv = min(32, g.E - col0) / 4;  // E % 8 == 0: whole 16-byte vectors
              for (int v = 0; v < nv; ++v)
                dst[v] = make_float4(__uint_as_float(rv[4 * v]), __uint_as_float(rv[4 * v + 1]),
                                     __uint_as_float(rv[4 * v + 2]), __uint_as_float(rv[4 * v + 3]));
            } else {
              uint4* dst = reinterpret_cast<uint4*>(g.io_bf16 + (size_t)row * g.d + col0);
#pragma unroll
              for (int v = 0; v < 4; ++v) {
                uint4 o = dst[v];
                uint32_t w[4] = {o.x, o.y, o.z, o.w};
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                  const float2 f = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&w[i]));
                  w[i] = pack_bf16(f.x + __uint_as_float(rv[8 * v + 2 * i]), f.y + __uint_as_float(rv[8 * v + 2 * i + 1]));
                }
                dst[v] = make_uint4(w[0], w[1], w[2], w[3]);
              }
            }
          }
        }
      } else {
        // plain bf16 store of the 128 x 256 tile: kDown, kBwdX, kWgradD, kWgradGU, kRouterDW
        const CUtensorMap* om = &g.mapO0;
        int orow = rowq;
        if (KIND == kWgradD) {
          orow = t.e * g.d + t.row0 + 32 * q;
        } else if (KIND == kWgradGU) {
          const bool up = t.row0 >= g.F;
          om = up ? &g.mapO1 : &g.mapO0;
          orow = t.e * g.F + (up ? t.row0 - g.F : t.row0) + 32 * q;
        }
        constexpr int kChunks = 8 / (TR::epi_warps / 4);   // 32-column chunks per warp
        const int c0 = ((warp - 2) >> 2) * kChunks;
#pragma unroll 1
        for (int c = c0; c < c0 + kChunks; ++c) {
          float v[32];
          if (has_acc) {
            uint32_t rv[32];
            tmem_ld32(tbase + c * 32, rv);
            tmem_ld_wait();
            if (c == c0 + kChunks - 1) {
              tc_fence_before();
              __syncwarp();
              if (lane == 0) mbar_arrive(&tempty[acc]);
            }
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(rv[i]);
          } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) v[i] = 0.0f;
          }
          if constexpr (KIND == kRouterDW) {
            if (g.ksplit > 1) {
              // split K: this split's fp32 partial sums, one row per lane
              if (rowq + lane < g.E) {
                float4* dst = reinterpret_cast<float4*>(g.part_f32 + ((size_t)t.split * g.E + rowq + lane) * g.d +
                                                        t.nt * BN + c * 32);
#pragma unroll
                for (int v4 = 0; v4 < 8; ++v4) dst[v4] = make_float4(v[4 * v4], v[4 * v4 + 1], v[4 * v4 + 2], v[4 * v4 + 3]);
              }
              ++chunk_ctr;
              continue;
            }
          }
          uint8_t* buf = stg + (TR::n_buf == 2 ? (chunk_ctr & 1) : 0) * kStageChunk;
          if (lane == 0) {
            if constexpr (TR::n_buf == 2) bulk_wait_read<1>();
            else bulk_wait_read<0>();
          }
          __syncwarp();
          stage_row(buf, lane, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            // kRouterDW: a 32-row slab wholly past the last expert is not stored
            if (KIND != kRouterDW || orow < g.E) tma_store_2d(om, buf, t.nt * BN + c * 32, orow);
            bulk_commit();
          }
          ++chunk_ctr;
        }
      }
      if (has_acc) {
        acc ^= 1;
        if (acc == 0) aph ^= 1;
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
}

// ---------------------------------------------------------------- host side
template <int KIND>
cudaError_t gemm_launch(const GemmArgs& a, int grid, cudaStream_t st) {
  gemm_kernel<KIND><<<grid, KindTraits<KIND>::threads, KindTraits<KIND>::smem_bytes, st>>>(a);
  return cudaGetLastError();
}

template <int KIND>
cudaError_t gemm_prepare() {
  return cudaFuncSetAttribute(gemm_kernel<KIND>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              KindTraits<KIND>::smem_bytes);
}

}  // namespace moe
