// gemm_mx.cuh -- persistent block-scaled (MXFP8) grouped GEMM for the
// forward expert contractions:
//   kUp    [a|b] = Xq . [Wgq;Wuq]^T   epilogue: a|b bf16 (saved), h = silu(a) b
//                                     re-quantised to MXFP8 along F (fused)
//   kDown  Ys    = Hq . Wdq^T         epilogue: bf16 rows
// (MXFP8 quantisation fused into the grouped-GEMM and SwiGLU datapaths:
// kucoin page "Cursor's MoK réalise une amélioration des performances de
// 2,37x sur NVIDIA GB300 NVL72", section 02.)
//
// Same structure as the bf16 kernel (gemm.cuh): warp 0 streams 128-byte K
// slices (128 E4M3 values = 4 scale blocks) of A and B with TMA plus their
// scale atoms with 1-D bulk copies; one thread of warp 1 copies the stage's
// scale atoms into TMEM (tcgen05.cp 32x128b.warpx4) and issues four
// tcgen05.mma.kind::mxf8f6f4.block_scale (M=128, N=256, K=32), the scale
// byte of each picked by the instruction's scale-factor id.  TMEM holds one
// 256-column fp32 accumulator plus a 16-column scale slot per stage, so the
// eight epilogue warps first drain the whole accumulator into registers
// (128 columns each), release it, and only then do the math and the stores.
// The u kind, which also reads a|b, parks the last of its four 32-column
// chunks in the TMEM columns left past the scale slots instead (three for
// MXFP8; two for NVFP4, whose u kind keeps two stages to make room).
// NVFP4 variant (NV = true): the same pipeline over packed E2M1 operands
// (128 bytes = 256 values of K per stage) with one E4M3 scale per 16 values:
// a 512-byte scale atom then covers one MMA's K = 64, so a stage brings four
// atoms per 128 rows, copies each into its own four TMEM columns, and issues
// four tcgen05.mma.kind::mxf4nvf4.block_scale.scale_vec::4X (M=128, N=256,
// K=64).  The weights' fp32 tensor scale multiplies the accumulator in the
// epilogue; h and dA|dB are re-quantised to NVFP4 (tensor scale 1).
#pragma once
#include "gemm.cuh"
#include "mx.cuh"
#include "nv.cuh"

namespace moe {

constexpr int kMxBK = 128;  // bytes of K per stage (128 E4M3 or 256 E2M1 values)

// Kinds: kUp, kDown (forward); kBwdU  u = dYq . WdTq^T with the SwiGLU-backward
// epilogue (dA|dB re-quantised along F for the dx GEMM; [dA|dB]^T and (w h)^T
// quantised along the sorted rows for the weight gradients; <u, h> partials);
// kBwdX  dx = dABq . [WgTq;WuTq]^T.
// WdTq [E*F, d], WgTq / WuTq [E*d, F] are the weights' backward orientation,
// quantised along their K (the dgrad GEMMs' K), so every operand is K-major.
template <int KIND, bool NV = false>
struct MxTraits {
  // MXFP8 keeps four stages in every kind: its multi-output epilogues (up:
  // a, b, h; bwd-u: dA, dB, w h) stage their bf16 tiles one after another
  // through a single buffer (seq), which leaves room for the fourth stage.
  // NVFP4's 54 KB stages fit three in its weight-gradient kinds, and four in
  // the up, down and dx kinds when their bf16 outputs go out 16 columns at a
  // time through one 1 KB buffer per warp (half16).  Its bwd-u kind keeps
  // two stages: their 96 scale columns
  // leave TMEM room to park half of u, so the accumulator is free before the
  // SwiGLU backward runs.
  static constexpr bool wgrad = (KIND == kWgradD || KIND == kWgradGU);
  static constexpr bool seq = !NV;
  static constexpr bool half16 = NV && (KIND == kUp || KIND == kDown || KIND == kBwdX);
  static constexpr int stages = (NV && KIND == kBwdU) ? 2 : (NV && wgrad) ? 3 : 4;
  static constexpr int epi_warps = 8;
  static constexpr int threads = 64 + 32 * epi_warps;
  static constexpr int kelems = NV ? 256 : 128;         // K values per stage
  static constexpr int atom_k = NV ? 64 : 128;          // K values per scale atom
  static constexpr int sf_rows = NV ? 2048 : 512;       // scale bytes per 128 rows per stage
  static constexpr int sf_stage = 3 * sf_rows;          // A atoms + two B row blocks
  static constexpr int sf_cols = NV ? 48 : 16;          // TMEM columns of one stage's scales
  static constexpr int qout = NV ? 512 : 1024;          // one 32 x 32 quantised staging tile
  static constexpr int staging_per_warp =
      half16 ? 1024
      : (KIND == kUp) ? ((seq ? 1 : 2) * 2048 + qout)
      : (KIND == kBwdU) ? (seq ? 2048 + qout : 3 * 2048 + 2 * qout) : 2048;
  static constexpr int staging_off = (stages * (kStageBytes + sf_stage) + 1023) / 1024 * 1024;
  static constexpr int smem_bytes = staging_off + epi_warps * staging_per_warp + 1024 + 256;
  static_assert(smem_bytes <= 232448, "shared memory per CTA");
  static_assert(BN + stages * sf_cols <= 512, "TMEM columns");
};

struct MxArgs {
  CUtensorMap mapA;   // quantised activations [rows, K bytes]
  CUtensorMap mapB0;  // quantised weights (Wg / Wd)
  CUtensorMap mapB1;  // quantised weights (Wu) for kUp
  CUtensorMap mapO0;  // bf16 stores (a|b for kUp, Ys for kDown); NVFP4 up/down/dx: 16-column boxes
  CUtensorMap mapO1;  // quantised stores (kUp: h; kBwdU: dA|dB)
  CUtensorMap mapO2;  // kBwdU: bf16 w h stores
  const uint8_t* sfA;   // scale atoms of A (rows = sorted padded rows)
  const uint8_t* sfB0;  // scale atoms of B0
  const uint8_t* sfB1;  // scale atoms of B1
  uint8_t* sfO;         // scale atoms of the quantised output (kUp: h, K = F; kBwdU: dA|dB, K = 2F)
  const float* tsB;     // NVFP4: device fp32 tensor scale of the B operand (weights)
  const __nv_bfloat16* ab;   // kBwdU: saved a|b [rows, 2F]
  const int32_t* perm_src;   // kBwdU
  const float* wts;          // kBwdU
  float* dgp;                // kBwdU: [rows, F/128] partial <u, h> per 128 columns
  float* dbg;                // debug (or null): the fp32 values the epilogue quantises,
                             //   kUp h [rows, F], kBwdU dA|dB [rows, 2F]
  const int32_t* poff;
  const int32_t* mtile_off;
  int32_t* status;
  uint64_t timeout_ns;
  int E, d, F;
  int Kcap;                  // weight-gradient kinds and kBwdU: token capacity of the transposed operands
  // kBwdU: [dA|dB]^T and (w h)^T quantised along the sorted rows (the weight
  // gradients' operands), [2F, Kcap] and [F, Kcap] with their scale atoms
  uint8_t* qT0;
  uint8_t* sT0;
  uint8_t* qT1;
  uint8_t* sT1;
};

// Column `lane` of a staged 32 x 32 bf16 tile (stage_row's layout: 16-byte
// chunk c of row r at chunk c ^ ((r >> 1) & 3)), quantised along its 32 rows
// -- sorted rows rowq .. rowq + 31, one MXFP8 block or two NVFP4 blocks
// (tensor scale 1) -- into row `orow` of a transposed operand qT [C, P] at
// column rowq, its scale bytes into the atoms of the C rows with K = P.  A
// warp's 32 lanes read one 64-byte row per step: no bank conflicts.
template <bool NV>
__device__ __forceinline__ void store_col_q(const uint8_t* stg, int lane, uint8_t* __restrict__ qT,
                                            uint8_t* __restrict__ sT, int64_t orow, int rowq, int P, float rc1) {
  float v[32];
  const int ch = lane >> 3, el = lane & 7;
#pragma unroll
  for (int r = 0; r < 32; ++r)
    v[r] = __bfloat162float(
        *reinterpret_cast<const __nv_bfloat16*>(stg + r * 64 + ((ch ^ ((r >> 1) & 3)) << 4) + el * 2));
  if constexpr (NV) {
    uint4 o;
    const uint32_t s2 = nv_encode32(v, rc1, 1.0f, o);
    *reinterpret_cast<uint4*>(qT + orow * (P / 2) + rowq / 2) = o;
    *reinterpret_cast<uint16_t*>(sT + sf_atom_offset(orow, rowq / 16, P / 16)) = (uint16_t)s2;
  } else {
    const int xe = mx_block_exponent(amax32(v));
    uint32_t o[8];
    mx_encode32(v, xe, o);
    uint4* dq = reinterpret_cast<uint4*>(qT + orow * P + rowq);
    dq[0] = make_uint4(o[0], o[1], o[2], o[3]);
    dq[1] = make_uint4(o[4], o[5], o[6], o[7]);
    sT[sf_atom_offset(orow, rowq / 32, P / 32)] = (uint8_t)(xe + 127);
  }
}

// One stage: the A and B tiles (TMA; x coordinates in bytes) and their scale
// atoms (1-D bulk copies).  Atoms of consecutive K groups are adjacent, so the
// four NVFP4 atoms of a stage are one 2 KB copy per 128-row block.
template <int KIND, bool NV>
__device__ __forceinline__ void mx_load_stage(const MxArgs& g, const Tile& t, int kb, uint8_t* sa, uint8_t* sb,
                                              uint8_t* ssf, uint64_t* bar, uint64_t pol_w, uint64_t pol_a) {
  using TR = MxTraits<KIND, NV>;
  constexpr uint32_t SFB = TR::sf_rows;
  const int x0 = kb * kMxBK;          // byte coordinate along K
  const int ke = kb * TR::kelems;     // value coordinate along K
  if (KIND == kWgradD || KIND == kWgradGU) {
    // K = the expert's tokens from its segment start, in the transposed
    // operands [rows, Kcap]: A = dY^T (kWgradD) or [dA|dB]^T rows, B = (w h)^T
    // or X^T rows nt*256 ..; everything is an activation (pol_a)
    const int kt = t.kbase + ke;                  // first token of the stage
    const int xk = NV ? kt / 2 : kt;              // its byte coordinate
    const int kg = g.Kcap / TR::atom_k;
    const int ka = kt / TR::atom_k;
    const int brow = t.nt * BN;
    tma_load_2d(sa, &g.mapA, xk, t.row0, bar, pol_a);
    tma_load_2d(sb, &g.mapB0, xk, brow, bar, pol_a);
    bulk_load_1d(ssf, g.sfA + ((size_t)(t.row0 >> 7) * kg + ka) * 512, SFB, bar);
    bulk_load_1d(ssf + SFB, g.sfB0 + ((size_t)(brow >> 7) * kg + ka) * 512, SFB, bar);
    bulk_load_1d(ssf + 2 * SFB, g.sfB0 + ((size_t)((brow >> 7) + 1) * kg + ka) * 512, SFB, bar);
  } else if (KIND == kUp) {
    const int kg = g.d / TR::atom_k;  // scale atoms per 128-row block
    tma_load_2d(sa, &g.mapA, x0, t.row0, bar, pol_a);
    const int brow = t.e * g.F + t.nt * 128;
    tma_load_2d(sb, &g.mapB0, x0, brow, bar, pol_w);
    tma_load_2d(sb + kBBytes / 2, &g.mapB1, x0, brow, bar, pol_w);
    const int ka = ke / TR::atom_k;
    bulk_load_1d(ssf, g.sfA + ((size_t)(t.row0 >> 7) * kg + ka) * 512, SFB, bar);
    bulk_load_1d(ssf + SFB, g.sfB0 + ((size_t)(brow >> 7) * kg + ka) * 512, SFB, bar);
    bulk_load_1d(ssf + 2 * SFB, g.sfB1 + ((size_t)(brow >> 7) * kg + ka) * 512, SFB, bar);
  } else if (KIND == kDown || KIND == kBwdU) {
    // kDown: A = Hq (K = F), B = Wdq rows e*d + n;  kBwdU: A = dYq (K = d), B = WdTq rows e*F + n
    const int K = (KIND == kDown) ? g.F : g.d;
    const int kg = K / TR::atom_k;
    const int ka = ke / TR::atom_k;
    tma_load_2d(sa, &g.mapA, x0, t.row0, bar, pol_a);
    const int brow = (KIND == kDown ? t.e * g.d : t.e * g.F) + t.nt * BN;
    tma_load_2d(sb, &g.mapB0, x0, brow, bar, pol_w);
    bulk_load_1d(ssf, g.sfA + ((size_t)(t.row0 >> 7) * kg + ka) * 512, SFB, bar);
    bulk_load_1d(ssf + SFB, g.sfB0 + ((size_t)(brow >> 7) * kg + ka) * 512, SFB, bar);
    bulk_load_1d(ssf + 2 * SFB, g.sfB0 + ((size_t)((brow >> 7) + 1) * kg + ka) * 512, SFB, bar);
  } else {  // kBwdX: A = dABq (K = 2F); B = WgTq for k < F, WuTq for k >= F (rows e*d + n, K = F)
    const int kga = (2 * g.F) / TR::atom_k, kgb = g.F / TR::atom_k;
    tma_load_2d(sa, &g.mapA, x0, t.row0, bar, pol_a);
    const bool up = ke >= g.F;
    const int kw = up ? ke - g.F : ke;           // value coordinate inside Wg^T / Wu^T
    const int brow = t.e * g.d + t.nt * BN;
    tma_load_2d(sb, up ? &g.mapB1 : &g.mapB0, NV ? kw / 2 : kw, brow, bar, pol_w);
    const uint8_t* sfb = up ? g.sfB1 : g.sfB0;
    bulk_load_1d(ssf, g.sfA + ((size_t)(t.row0 >> 7) * kga + ke / TR::atom_k) * 512, SFB, bar);
    bulk_load_1d(ssf + SFB, sfb + ((size_t)(brow >> 7) * kgb + kw / TR::atom_k) * 512, SFB, bar);
    bulk_load_1d(ssf + 2 * SFB, sfb + ((size_t)((brow >> 7) + 1) * kgb + kw / TR::atom_k) * 512, SFB, bar);
  }
}

// K stages of a tile, and how many of the last stage's four MMAs carry K.
// Weight-gradient kinds take the expert's (128-row aligned) token segment: a
// stage holds 128 E4M3 or 256 E2M1 tokens, so an NVFP4 segment whose length
// is an odd multiple of 128 ends on a half stage (two of the four K=64 MMAs);
// an expert without rows has no stage.
template <int KIND, bool NV>
__device__ __forceinline__ int mx_tile_nkb(const MxArgs& g, const Tile& t, int& last_mmas) {
  using TR = MxTraits<KIND, NV>;
  last_mmas = 4;
  if (KIND == kWgradD || KIND == kWgradGU) {
    const int rows = __ldg(g.poff + t.e + 1) - t.kbase;
    if (NV && (rows % 256)) last_mmas = 2;
    return (rows + TR::kelems - 1) / TR::kelems;
  }
  return (KIND == kUp || KIND == kBwdU ? g.d : KIND == kDown ? g.F : 2 * g.F) / TR::kelems;
}

// 32 fp32 -> 32 E4M3 bytes of one row into an unswizzled 32x32-byte staging tile.
__device__ __forceinline__ void stage_row_fp8(uint8_t* buf, int lane, const uint32_t (&q)[8]) {
  uint4* p = reinterpret_cast<uint4*>(buf + lane * 32);
  p[0] = make_uint4(q[0], q[1], q[2], q[3]);
  p[1] = make_uint4(q[4], q[5], q[6], q[7]);
}

// 16 floats -> 16 bf16 of one row into an unswizzled 32-row x 32-byte staging tile.
__device__ __forceinline__ void stage_row16(uint8_t* buf, int lane, const float* v) {
  uint32_t p[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) p[i] = pack_bf16(v[2 * i], v[2 * i + 1]);
  uint4* d = reinterpret_cast<uint4*>(buf + lane * 32);
  d[0] = make_uint4(p[0], p[1], p[2], p[3]);
  d[1] = make_uint4(p[4], p[5], p[6], p[7]);
}

// 32 values -> 16 packed E2M1 bytes of one row into an unswizzled 32x16-byte staging tile.
__device__ __forceinline__ void stage_row_fp4(uint8_t* buf, int lane, const uint4& q) {
  *reinterpret_cast<uint4*>(buf + lane * 16) = q;
}

template <int KIND, bool NV = false>
__global__ void __launch_bounds__(MxTraits<KIND, NV>::threads, 1) gemm_mx_kernel(const __grid_constant__ MxArgs g) {
  using TR = MxTraits<KIND, NV>;
  constexpr int S = TR::stages;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* stage_base = smem;
  uint8_t* sf_base = smem + S * kStageBytes;
  uint8_t* staging_base = smem + TR::staging_off;
  uint64_t* bars = reinterpret_cast<uint64_t*>(staging_base + TR::epi_warps * TR::staging_per_warp);
  uint64_t* full = bars;
  uint64_t* empty = bars + S;
  uint64_t* tfull = bars + 2 * S;
  uint64_t* tempty = bars + 2 * S + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 2 * S + 2);
  int* abort_flag = reinterpret_cast<int*>(tmem_slot + 1);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, TR::epi_warps);
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
  const int ntiles = total_tiles<KIND>(g);

  if (warp == 0) {
    if (lane == 0) {
      // weight tiles are re-read by every M tile of their expert: evict_last,
      // as in the bf16 grouped GEMMs.  MXFP8: an expert with a single M tile
      // reads its weight tiles once, so they go evict_first and leave L2 to
      // the re-read activation rows (the four grouped kinds 0.04-0.07 ms
      // faster per fwd+bwd step at T=8192, E=256; neutral for bf16, and the
      // NVFP4 u kind got slower).
      const uint64_t pol_w = policy_evict_last();
      const uint64_t pol_once = policy_evict_first();
      const uint64_t pol_a = policy_evict_last();
      uint32_t s = 0, ph = 0, issued_mask = 0, last_par = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const Tile t = decode_tile<KIND>(g, tile);
        int last_mmas;
        const int nkb = mx_tile_nkb<KIND, NV>(g, t, last_mmas);
        bool once = false;
        if constexpr (!NV && KindTraits<KIND>::grouped)
          once = __ldg(g.mtile_off + t.e + 1) - __ldg(g.mtile_off + t.e) == 1;
        const uint64_t pw = once ? pol_once : pol_w;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait(&empty[s], ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(&full[s], kStageBytes + TR::sf_stage);
          uint8_t* sa = stage_base + s * kStageBytes;
          mx_load_stage<KIND, NV>(g, t, kb, sa, sa + kABytes, sf_base + s * TR::sf_stage, &full[s], pw, pol_a);
          issued_mask |= 1u << s;
          last_par = (last_par & ~(1u << s)) | (ph << s);
          if (++s == S) { s = 0; ph ^= 1; }
        }
      }
      if (!ok) {  // abort: let issued copies land before the CTA may exit
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
      uint32_t s = 0, ph = 0, aph = 0;
      bool ok = true;
      for (int tile = blockIdx.x; tile < ntiles && ok; tile += gridDim.x) {
        const Tile t = decode_tile<KIND>(g, tile);
        int last_mmas;
        const int nkb = mx_tile_nkb<KIND, NV>(g, t, last_mmas);
        if (nkb == 0) continue;  // an expert without rows: the epilogue writes zeros
        if (!mbar_wait(tempty, aph ^ 1, wc)) break;
        tc_fence_after();
        for (int kb = 0; kb < nkb; ++kb) {
          const int nmma = kb == nkb - 1 ? last_mmas : 4;  // MMAs of this stage that carry K
          if (!mbar_wait(&full[s], ph, wc)) { ok = false; break; }
          tc_fence_after();
          const uint32_t sa = smem_u32(stage_base + s * kStageBytes);
          const uint32_t sb = sa + kABytes;
          const uint32_t ssf = smem_u32(sf_base + s * TR::sf_stage);
          const uint32_t sfa_t = tmem_base + BN + s * TR::sf_cols;
          if constexpr (NV) {
            // atom kk of each 128-row block -> its own 4 TMEM columns: A at
            // sfa_t + 4 kk, B rows 0-127 at sfb_t + 8 kk, rows 128-255 at +4
            const uint32_t sfb_t = sfa_t + 16;
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              tmem_cp_32x128_x4(sfa_t + 4 * kk, sdesc_plain(ssf + 512 * kk));
              tmem_cp_32x128_x4(sfb_t + 8 * kk, sdesc_plain(ssf + TR::sf_rows + 512 * kk));
              tmem_cp_32x128_x4(sfb_t + 8 * kk + 4, sdesc_plain(ssf + 2 * TR::sf_rows + 512 * kk));
            }
#pragma unroll
            for (int kk = 0; kk < 4; ++kk) {
              if (kk >= nmma) break;
              const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(sb + kk * 32, 16, 1024);
              umma_nvf4(tmem_base, ad, bd, idesc_nvf4(BM, BN), sfa_t + 4 * kk, sfb_t + 8 * kk,
                        (kb | kk) != 0 ? 1u : 0u);
            }
          } else {
            const uint32_t sfb_t = sfa_t + 8;  // 8 columns
            tmem_cp_32x128_x4(sfa_t, sdesc_plain(ssf));
            tmem_cp_32x128_x4(sfb_t, sdesc_plain(ssf + 512));
            tmem_cp_32x128_x4(sfb_t + 4, sdesc_plain(ssf + 1024));
#pragma unroll
            for (int kk = 0; kk < kMxBK / 32; ++kk) {
              const uint64_t ad = sdesc_sw128(sa + kk * 32, 16, 1024);
              const uint64_t bd = sdesc_sw128(sb + kk * 32, 16, 1024);
              umma_mxf8(tmem_base, ad, bd, idesc_mxf8(BM, BN, 0, 0, kk), sfa_t, sfb_t, (kb | kk) != 0 ? 1u : 0u);
            }
          }
          umma_commit(&empty[s]);
          if (++s == S) { s = 0; ph ^= 1; }
        }
        if (!ok) break;
        umma_commit(tfull);
        aph ^= 1;
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;            // TMEM lane quadrant
    const int half = (warp - 2) >> 2;  // which half of the tile's columns
    uint8_t* stg = staging_base + (warp - 2) * TR::staging_per_warp;
    const float gs = (NV && g.tsB) ? __ldg(g.tsB) : 1.0f;   // weights' tensor scale (NVFP4)
    const float rc1 = nv_rc(1.0f);               // activations: tensor scale 1
    uint32_t aph = 0;
    for (int tile = blockIdx.x; tile < ntiles; tile += gridDim.x) {
      const Tile t = decode_tile<KIND>(g, tile);
      int last_mmas;
      const bool has_acc = mx_tile_nkb<KIND, NV>(g, t, last_mmas) > 0;
      if (has_acc) {
        if (!mbar_wait(tfull, aph, wc)) break;
        tc_fence_after();
      }
      const uint32_t tb = tmem_base + ((uint32_t)(32 * q) << 16);
      const int rowq = t.row0 + 32 * q;
      if (KIND == kBwdU) {
        // u in 32-column chunks: dh = w u, da = dh b s(a)(1 + a(1 - s(a))),
        // db = dh silu(a); outputs dA|dB quantised along F for the dx GEMM,
        // the bf16 dA, dB and w h staged 32 rows x 32 columns and quantised
        // column by column along the rows into the weight gradients'
        // transposed operands, and the row's <u, h> over this warp's 128
        // columns.
        const int r = rowq + lane;
        const int src = __ldg(g.perm_src + r);
        const float wr = src >= 0 ? __ldg(g.wts + src) : 0.0f;
        const __nv_bfloat16* abrow = g.ab + (size_t)r * (2 * g.F);
        float dgacc = 0.0f;
        uint32_t sfa[2] = {0u, 0u}, sfb[2] = {0u, 0u};
        // the bf16 dA|dB and w h are read only by the debug dump: the weight
        // gradients take their quantised transposes, made from the staged tiles
        const bool keep_bf16 = g.dbg != nullptr;
        // one 32-column chunk c of u, its TMEM load issued into ru: the SwiGLU
        // backward and the stores; `release` frees the accumulator as soon as
        // that load has landed
        auto chunk = [&](int c, uint32_t (&ru)[32], bool release) {
          const int col = t.nt * BN + half * 128 + c * 32;
          float a[32], b[32];
          load_bf16x32(abrow + col, a);
          load_bf16x32(abrow + g.F + col, b);
          tmem_ld_wait();
          if (release) {
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(tempty);
          }
          float da[32], db[32], wh[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            const float u = NV ? __uint_as_float(ru[i]) * gs : __uint_as_float(ru[i]);
            const float sa = sigmoidf_(a[i]);
            const float sl = a[i] * sa;
            const float hh = sl * b[i];
            dgacc = fmaf(u, hh, dgacc);
            const float dh = wr * u;
            da[i] = dh * b[i] * sa * (1.0f + a[i] * (1.0f - sa));
            db[i] = dh * sl;
            wh[i] = wr * hh;
          }
          if (g.dbg) {
            float4* pa = reinterpret_cast<float4*>(g.dbg + (size_t)r * (2 * g.F) + col);
            float4* pb = reinterpret_cast<float4*>(g.dbg + (size_t)r * (2 * g.F) + g.F + col);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              pa[i] = make_float4(da[4 * i], da[4 * i + 1], da[4 * i + 2], da[4 * i + 3]);
              pb[i] = make_float4(db[4 * i], db[4 * i + 1], db[4 * i + 2], db[4 * i + 3]);
            }
          }
          constexpr int qd = NV ? 2 : 1;   // values per quantised byte
          if constexpr (TR::seq) {
            // one bf16 and one quantised buffer, reused output by output
            uint32_t qa[8], qb[8];
            const int Xa = mx_block_exponent(amax32(da));
            const int Xb = mx_block_exponent(amax32(db));
            mx_encode32(da, Xa, qa);
            mx_encode32(db, Xb, qb);
            sfa[0] |= (uint32_t)(Xa + 127) << (8 * c);
            sfb[0] |= (uint32_t)(Xb + 127) << (8 * c);
            uint8_t* sq = stg + kStageChunk;
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            stage_row(stg, lane, da);
            stage_row_fp8(sq, lane, qa);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (keep_bf16) tma_store_2d(&g.mapO0, stg, col, rowq);
              tma_store_2d(&g.mapO1, sq, col / qd, rowq);
              bulk_commit();
            }
            store_col_q<NV>(stg, lane, g.qT0, g.sT0, col + lane, rowq, g.Kcap, rc1);
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            stage_row(stg, lane, db);
            stage_row_fp8(sq, lane, qb);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              if (keep_bf16) tma_store_2d(&g.mapO0, stg, g.F + col, rowq);
              tma_store_2d(&g.mapO1, sq, (g.F + col) / qd, rowq);
              bulk_commit();
            }
            store_col_q<NV>(stg, lane, g.qT0, g.sT0, g.F + col + lane, rowq, g.Kcap, rc1);
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            stage_row(stg, lane, wh);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0 && keep_bf16) {
              tma_store_2d(&g.mapO2, stg, col, rowq);
              bulk_commit();
            }
            store_col_q<NV>(stg, lane, g.qT1, g.sT1, col + lane, rowq, g.Kcap, rc1);
            return;
          }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row(stg, lane, da);
          stage_row(stg + kStageChunk, lane, db);
          stage_row(stg + 2 * kStageChunk, lane, wh);
          if constexpr (NV) {
            uint4 qa, qb;
            sfa[c >> 1] |= nv_encode32(da, rc1, 1.0f, qa) << (16 * (c & 1));
            sfb[c >> 1] |= nv_encode32(db, rc1, 1.0f, qb) << (16 * (c & 1));
            stage_row_fp4(stg + 3 * kStageChunk, lane, qa);
            stage_row_fp4(stg + 3 * kStageChunk + TR::qout, lane, qb);
          } else {
            const int Xa = mx_block_exponent(amax32(da));
            const int Xb = mx_block_exponent(amax32(db));
            uint32_t qa[8], qb[8];
            mx_encode32(da, Xa, qa);
            mx_encode32(db, Xb, qb);
            sfa[0] |= (uint32_t)(Xa + 127) << (8 * c);
            sfb[0] |= (uint32_t)(Xb + 127) << (8 * c);
            stage_row_fp8(stg + 3 * kStageChunk, lane, qa);
            stage_row_fp8(stg + 3 * kStageChunk + TR::qout, lane, qb);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            if (keep_bf16) {
              tma_store_2d(&g.mapO0, stg, col, rowq);
              tma_store_2d(&g.mapO0, stg + kStageChunk, g.F + col, rowq);
              tma_store_2d(&g.mapO2, stg + 2 * kStageChunk, col, rowq);
            }
            tma_store_2d(&g.mapO1, stg + 3 * kStageChunk, col / qd, rowq);
            tma_store_2d(&g.mapO1, stg + 3 * kStageChunk + TR::qout, (g.F + col) / qd, rowq);
            bulk_commit();
          }
          store_col_q<NV>(stg, lane, g.qT0, g.sT0, col + lane, rowq, g.Kcap, rc1);
          store_col_q<NV>(stg + kStageChunk, lane, g.qT0, g.sT0, g.F + col + lane, rowq, g.Kcap, rc1);
          store_col_q<NV>(stg + 2 * kStageChunk, lane, g.qT1, g.sT1, col + lane, rowq, g.Kcap, rc1);
        };
        {
          // All four chunks leave the accumulator before any math: the last
          // kPark of them into the TMEM columns past the stages' scale slots
          // (kPark * 32 per column half), the others into registers.  The next
          // tile's MMAs then run while this tile's SwiGLU backward and stores do.
          constexpr int kPark = NV ? 2 : 3;
          static_assert(KIND != kBwdU || BN + TR::stages * TR::sf_cols + 2 * 32 * kPark <= 512,
                        "TMEM columns for the parked u");
          const uint32_t park = tb + BN + TR::stages * TR::sf_cols + half * 32 * kPark;
          uint32_t ru0[32], ru1[32];
#pragma unroll 1
          for (int c = 4 - kPark; c < 4; ++c) {
            tmem_ld32(tb + half * 128 + c * 32, ru0);
            tmem_ld_wait();
            tmem_st32(park + (c - (4 - kPark)) * 32, ru0);
            tmem_st_wait();   // ru0 is reloaded next
          }
          tmem_ld32(tb + half * 128, ru0);
          if (kPark == 2) tmem_ld32(tb + half * 128 + 32, ru1);
          tmem_ld_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(tempty);
          chunk(0, ru0, false);
          if (kPark == 2) chunk(1, ru1, false);
#pragma unroll 1
          for (int c = 4 - kPark; c < 4; ++c) {
            tmem_ld32(park + (c - (4 - kPark)) * 32, ru0);
            chunk(c, ru0, false);
          }
        }
        aph ^= 1;
        if constexpr (NV) {
          // 8 blocks of 16 per operand: two scale words, in consecutive atoms
          const int kba = (t.nt * BN + half * 128) / 16;
          const int nb = (2 * g.F) / 16;
#pragma unroll
          for (int w2 = 0; w2 < 2; ++w2) {
            *reinterpret_cast<uint32_t*>(g.sfO + sf_atom_offset(r, kba + 4 * w2, nb)) = sfa[w2];
            *reinterpret_cast<uint32_t*>(g.sfO + sf_atom_offset(r, g.F / 16 + kba + 4 * w2, nb)) = sfb[w2];
          }
        } else {
          const int kba = (t.nt * BN + half * 128) / 32;  // first of this warp's 4 blocks (K = 2F)
          *reinterpret_cast<uint32_t*>(g.sfO + sf_atom_offset(r, kba, (2 * g.F) / 32)) = sfa[0];
          *reinterpret_cast<uint32_t*>(g.sfO + sf_atom_offset(r, g.F / 32 + kba, (2 * g.F) / 32)) = sfb[0];
        }
        g.dgp[(size_t)r * (g.F / 128) + t.nt * 2 + half] = dgacc;
        continue;
      }
      uint32_t acc[4][32];
      if (KIND == kUp) {  // a cols [64 half, +64), b cols 128 + [64 half, +64)
        tmem_ld32(tb + half * 64, acc[0]);
        tmem_ld32(tb + half * 64 + 32, acc[1]);
        tmem_ld32(tb + 128 + half * 64, acc[2]);
        tmem_ld32(tb + 128 + half * 64 + 32, acc[3]);
      } else if (has_acc) {
#pragma unroll
        for (int c = 0; c < 4; ++c) tmem_ld32(tb + half * 128 + c * 32, acc[c]);
      } else {
#pragma unroll
        for (int c = 0; c < 4; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i) acc[c][i] = 0u;   // dW of an expert without rows
      }
      if (has_acc) {
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty);
        aph ^= 1;
      }
      if (KIND == kUp) {
        uint32_t sfw = 0;
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2) {
          float a[32], b[32], h[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) {
            a[i] = NV ? __uint_as_float(acc[c2][i]) * gs : __uint_as_float(acc[c2][i]);
            b[i] = NV ? __uint_as_float(acc[2 + c2][i]) * gs : __uint_as_float(acc[2 + c2][i]);
            h[i] = a[i] * sigmoidf_(a[i]) * b[i];
          }
          if (g.dbg) {
            float4* ph = reinterpret_cast<float4*>(g.dbg + (size_t)(rowq + lane) * g.F + t.nt * 128 + half * 64 +
                                                   c2 * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i) ph[i] = make_float4(h[4 * i], h[4 * i + 1], h[4 * i + 2], h[4 * i + 3]);
          }
          if constexpr (TR::half16) {
            // a and b in 16-column halves, then h, through one 1 KB buffer
            uint4 hq;
            sfw |= nv_encode32(h, rc1, 1.0f, hq) << (16 * c2);
            const int col = t.nt * 128 + half * 64 + c2 * 32;
#pragma unroll
            for (int part = 0; part < 5; ++part) {
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              if (part < 2) stage_row16(stg, lane, a + 16 * part);
              else if (part < 4) stage_row16(stg, lane, b + 16 * (part - 2));
              else stage_row_fp4(stg, lane, hq);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                if (part < 2) tma_store_2d(&g.mapO0, stg, col + 16 * part, rowq);
                else if (part < 4) tma_store_2d(&g.mapO0, stg, g.F + col + 16 * (part - 2), rowq);
                else tma_store_2d(&g.mapO1, stg, col / 2, rowq);
                bulk_commit();
              }
            }
            continue;
          }
          if constexpr (TR::seq) {
            // a, then b with h, through one bf16 buffer and one E4M3 buffer
            const int X = mx_block_exponent(amax32(h));
            uint32_t hq[8];
            mx_encode32(h, X, hq);
            sfw |= (uint32_t)(X + 127) << (8 * c2);
            const int col = t.nt * 128 + half * 64 + c2 * 32;
            if (lane == 0) bulk_wait_read<0>();
            __syncwarp();
            stage_row(stg, lane, a);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&g.mapO0, stg, col, rowq);
              bulk_commit();
              bulk_wait_read<0>();
            }
            __syncwarp();
            stage_row(stg, lane, b);
            stage_row_fp8(stg + kStageChunk, lane, hq);
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&g.mapO0, stg, g.F + col, rowq);
              tma_store_2d(&g.mapO1, stg + kStageChunk, col, rowq);
              bulk_commit();
            }
            continue;
          }
          if (lane == 0) bulk_wait_read<0>();
          __syncwarp();
          stage_row(stg, lane, a);
          stage_row(stg + kStageChunk, lane, b);
          if constexpr (NV) {
            uint4 hq;
            sfw |= nv_encode32(h, rc1, 1.0f, hq) << (16 * c2);
            stage_row_fp4(stg + 2 * kStageChunk, lane, hq);
          } else {
            const int X = mx_block_exponent(amax32(h));
            uint32_t hq[8];
            mx_encode32(h, X, hq);
            sfw |= (uint32_t)(X + 127) << (8 * c2);
            stage_row_fp8(stg + 2 * kStageChunk, lane, hq);
          }
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            const int col = t.nt * 128 + half * 64 + c2 * 32;
            tma_store_2d(&g.mapO0, stg, col, rowq);
            tma_store_2d(&g.mapO0, stg + kStageChunk, g.F + col, rowq);
            tma_store_2d(&g.mapO1, stg + 2 * kStageChunk, NV ? col / 2 : col, rowq);
            bulk_commit();
          }
        }
        const int r = rowq + lane;
        if constexpr (NV) {
          // four scale bytes of this row (blocks 8 nt + 4 half .. +3): one word
          *reinterpret_cast<uint32_t*>(g.sfO + sf_atom_offset(r, t.nt * 8 + half * 4, g.F / 16)) = sfw;
        } else {
          // two consecutive scale bytes of this row (blocks 4 nt + 2 half, +1)
          const int kb = t.nt * 4 + half * 2;
          *reinterpret_cast<uint16_t*>(g.sfO + sf_atom_offset(r, kb, g.F / 32)) = (uint16_t)sfw;
        }
      } else {
        // output rows: kDown / kBwdX the sorted rows; weight gradients the
        // expert's dW rows (kWgradGU: rows below F are dWg, the rest dWu)
        const CUtensorMap* om = &g.mapO0;
        int orow = rowq;
        if (KIND == kWgradD) {
          orow = t.e * g.d + t.row0 + 32 * q;
        } else if (KIND == kWgradGU) {
          const bool up = t.row0 >= g.F;
          om = up ? &g.mapO1 : &g.mapO0;
          orow = t.e * g.F + (up ? t.row0 - g.F : t.row0) + 32 * q;
        }
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          float v[32];
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = NV ? __uint_as_float(acc[c][i]) * gs : __uint_as_float(acc[c][i]);
          if constexpr (TR::half16) {
#pragma unroll
            for (int part = 0; part < 2; ++part) {
              if (lane == 0) bulk_wait_read<0>();
              __syncwarp();
              stage_row16(stg, lane, v + 16 * part);
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&g.mapO0, stg, t.nt * BN + half * 128 + c * 32 + 16 * part, rowq);
                bulk_commit();
              }
            }
            continue;
          }
          if (lane == 0) {
            // MXFP8 weight gradients: the warp's previous dW store has left
            // for global memory, not only been read out of shared memory
            // (measured: throttling the dW stores this way lets the operand
            // loads through; 3.83 -> 3.41 ms for gate/up at T=8192.  NVFP4,
            // with three stages, loses with it)
            if constexpr (TR::wgrad && !NV) bulk_wait<0>();
            else bulk_wait_read<0>();
          }
          __syncwarp();
          stage_row(stg, lane, v);
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(om, stg, t.nt * BN + half * 128 + c * 32, orow);
            bulk_commit();
          }
        }
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

}  // namespace moe
