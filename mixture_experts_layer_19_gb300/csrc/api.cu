// api.cu -- the C ABI (include/moe.h): plan / workspace, argument checks,
// tensor-map encoding and the kernel sequence of forward and backward.
//
// Forward  (one stream, no host sync, no allocation):
//   router+histogram -> scan -> stable permute -> gather X into sorted rows
//   -> [a|b] GEMM + SwiGLU -> down GEMM -> fixed-order weighted combine.
// Backward:
//   gather dY and X -> u GEMM + SwiGLU backward -> dx GEMM -> per-token dx
//   reduce -> router gradient -> dWd GEMM -> dWg/dWu GEMM.
#include <cudaTypedefs.h>

#include <algorithm>
#include <cstdio>
#include <initializer_list>
#include <cstring>
#include <mutex>
#include <string>
#include <vector>

#include "gemm.cuh"
#include "gemm_mx.cuh"
#include "kernels.h"
#include "megakernel.cuh"
#include "moe.h"

using namespace moe;

namespace {

thread_local std::string g_last_error;
thread_local std::string g_encode_detail;  // last tensor-map encoding failure, appended by fail()

moe_status_t fail(moe_status_t s, const std::string& msg) {
  g_last_error = msg;
  if (!g_encode_detail.empty()) {
    g_last_error += " [" + g_encode_detail + "]";
    g_encode_detail.clear();
  }
  return s;
}
moe_status_t cuda_fail(cudaError_t e, const char* what) {
  g_last_error = std::string(what) + ": " + cudaGetErrorString(e);
  return MOE_ERR_CUDA;
}

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D tensor map over a row-major [outer, inner] buffer of bf16 (esize 2) or
// bytes (esize 1, E4M3 data).
bool encode_2d(CUtensorMap* m, const void* base, uint64_t inner, uint64_t outer, uint32_t box_in, uint32_t box_out,
               CUtensorMapSwizzle sw, int esize = 2) {
  auto enc = encode_fn();
  if (!enc) return false;
  cuuint64_t dims[2] = {inner, outer};
  cuuint64_t strides[1] = {inner * (uint64_t)esize};
  cuuint32_t box[2] = {box_in, box_out};
  cuuint32_t es[2] = {1, 1};
  CUresult r = enc(m, esize == 2 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_UINT8, 2,
                   const_cast<void*>(base), dims, strides, box, es, CU_TENSOR_MAP_INTERLEAVE_NONE, sw,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) {
    char buf[160];
    snprintf(buf, sizeof(buf), "cuTensorMapEncodeTiled error %d: base %p, %llu x %llu, box %u x %u", (int)r, base,
             (unsigned long long)outer, (unsigned long long)inner, box_out, box_in);
    g_encode_detail = buf;
  }
  return r == CUDA_SUCCESS;
}
// E4M3 operand loads: 128-byte K slices, 128 (or 256) rows, 128-byte swizzle.
bool map_fp8_kmajor(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer, uint32_t rows = BM) {
  return encode_2d(m, b, inner, outer, 128, rows, CU_TENSOR_MAP_SWIZZLE_128B, 1);
}
// Quantised stores of 32 rows x box_in bytes (32 E4M3 or 32 packed E2M1
// values: 32 or 16 bytes), no swizzle.
bool map_fp8_store(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer, uint32_t box_in = 32) {
  return encode_2d(m, b, inner, outer, box_in, 32, CU_TENSOR_MAP_SWIZZLE_NONE, 1);
}
// The three shapes the GEMMs use.
bool map_kmajor(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer, uint32_t rows = BM) {
  return encode_2d(m, b, inner, outer, 64, rows, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_mnmajor(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer) {
  return encode_2d(m, b, inner, outer, 64, 64, CU_TENSOR_MAP_SWIZZLE_128B);
}
bool map_store(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer) {
  return encode_2d(m, b, inner, outer, 32, 32, CU_TENSOR_MAP_SWIZZLE_64B);
}
// bf16 stores of 32 rows x 16 columns, no swizzle (the NVFP4 GEMMs' half-chunk staging).
bool map_store16(CUtensorMap* m, const void* b, uint64_t inner, uint64_t outer) {
  return encode_2d(m, b, inner, outer, 16, 32, CU_TENSOR_MAP_SWIZZLE_NONE);
}

struct SavedLayout {
  size_t idx, w, dest, counts, offsets, poff, mtile, totals, perm, ab, total;
  int64_t rows;  // padded sorted-row capacity for this T
};

SavedLayout saved_layout(const moe_config_t& c, int64_t T) {
  SavedLayout L{};
  const int64_t R = T * c.k;
  L.rows = ((R + (int64_t)c.E * (kTileRows - 1)) + kTileRows - 1) / kTileRows * kTileRows;
  size_t o = 0;
  L.idx = o;     o += align256(R * 4);
  L.w = o;       o += align256(R * 4);
  L.dest = o;    o += align256(R * 4);
  L.counts = o;  o += align256(c.E * 4);
  L.offsets = o; o += align256((c.E + 1) * 4);
  L.poff = o;    o += align256((c.E + 1) * 4);
  L.mtile = o;   o += align256((c.E + 1) * 4);
  L.totals = o;  o += align256(16);
  L.perm = o;    o += align256(L.rows * 4);
  L.ab = o;      o += align256((size_t)L.rows * 2 * c.F * 2);
  L.total = o;
  return L;
}

RoutingPtrs routing_ptrs(const SavedLayout& L, void* saved) {
  char* b = static_cast<char*>(saved);
  RoutingPtrs rp;
  rp.idx = reinterpret_cast<int32_t*>(b + L.idx);
  rp.w = reinterpret_cast<float*>(b + L.w);
  rp.dest = reinterpret_cast<int32_t*>(b + L.dest);
  rp.counts = reinterpret_cast<int32_t*>(b + L.counts);
  rp.offsets = reinterpret_cast<int32_t*>(b + L.offsets);
  rp.poff = reinterpret_cast<int32_t*>(b + L.poff);
  rp.mtile_off = reinterpret_cast<int32_t*>(b + L.mtile);
  rp.totals = reinterpret_cast<int32_t*>(b + L.totals);
  rp.perm_src = reinterpret_cast<int32_t*>(b + L.perm);
  return rp;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

// Makes the plan's device current for the call, and always binds its primary
// context to the calling thread: the tensor-map encoder is a driver call and
// fails on a thread (such as autograd's backward worker) that has not yet
// made a runtime call.
struct DeviceGuard {
  int old = -1;
  bool ok = true;
  explicit DeviceGuard(int dev) {
    if (cudaGetDevice(&old) != cudaSuccess) old = -1;
    ok = cudaSetDevice(dev) == cudaSuccess;
  }
  ~DeviceGuard() {
    int cur = -1;
    if (old >= 0 && cudaGetDevice(&cur) == cudaSuccess && cur != old) cudaSetDevice(old);
  }
};

struct TimedLaunch {
  const char* name;
  cudaEvent_t a, b;
};

}  // namespace

struct moe_plan_s {
  moe_config_t cfg;
  int num_sms = 0;
  int64_t Rpm = 0;  // padded row capacity at T_max
  void* ws = nullptr;
  int32_t* chunk_hist = nullptr;
  int32_t* chunk_base = nullptr;
  int32_t* status = nullptr;
  void *Xg = nullptr, *H = nullptr, *Ys = nullptr, *dYg = nullptr, *dAB = nullptr, *wH = nullptr;
  float* dgp = nullptr;
  // workspace tensor maps
  CUtensorMap m_Xg_k, m_Xg_mn, m_H_k, m_H_st, m_Ys_st, m_dYg_k, m_dYg_mn, m_dAB_k, m_dAB_mn, m_dAB_st, m_wH_mn,
      m_wH_st;
  // caller-pointer tensor maps, re-encoded when a pointer changes
  const void *p_wg = nullptr, *p_wu = nullptr, *p_wd = nullptr;
  CUtensorMap m_Wg_k, m_Wu_k, m_Wd_k, m_Wg_mn, m_Wu_mn, m_Wd_mn;
  const void *p_dwg = nullptr, *p_dwu = nullptr, *p_dwd = nullptr;
  CUtensorMap m_dWg_st, m_dWu_st, m_dWd_st;
  // MXFP8 (prec == MOE_MXFP8): E4M3 weights + scale atoms (filled by
  // moe_quantize_weights), E4M3 gathered activations and h with their scales
  void* mx_ws = nullptr;
  uint8_t *Wgq = nullptr, *Wuq = nullptr, *Wdq = nullptr, *Wgs = nullptr, *Wus = nullptr, *Wds = nullptr;
  uint8_t *Xq = nullptr, *Xs = nullptr, *Hq = nullptr, *Hs = nullptr;
  // backward orientation (quantised along the dgrad GEMMs' K) and E4M3 dA|dB
  uint8_t *WdTq = nullptr, *WgTq = nullptr, *WuTq = nullptr, *WdTs = nullptr, *WgTs = nullptr, *WuTs = nullptr;
  uint8_t *dABq = nullptr, *dABs = nullptr;
  // MXFP8 ring slots: E4M3 X and h rows with their scale atoms
  uint8_t *ring_xq = nullptr, *ring_xs = nullptr, *ring_hq = nullptr, *ring_hs = nullptr;
  uint8_t *Xtq = nullptr, *Xts = nullptr;  // tokens (X, or dY in the backward) quantised once per token
  CUtensorMap m_ring_xq, m_ring_hq, m_ring_hq_st;
  bool weights_quantized = false;
  CUtensorMap m_Wgq, m_Wuq, m_Wdq, m_Xq, m_Hq_k, m_Hq_st;
  CUtensorMap m_WdTq, m_WgTq, m_WuTq, m_dABq_k, m_dABq_st;
  CUtensorMap m_Ys_st16;  // NVFP4: Ys stores in 16-column boxes
  // block-scaled weight gradients: the backward's operands transposed and
  // quantised along the tokens, [rows, Rpm] (dY^T, X^T: d rows; [dA|dB]^T: 2F;
  // (w h)^T: F), with their scale atoms (K = Rpm)
  uint8_t *dYTq = nullptr, *dYTs = nullptr, *XTq = nullptr, *XTs = nullptr, *dABTq = nullptr, *dABTs = nullptr,
          *wHTq = nullptr, *wHTs = nullptr;
  CUtensorMap m_dYTq, m_XTq, m_dABTq, m_wHTq;
  // NVFP4 (prec == MOE_NVFP4) reuses the block-scaled buffers above with
  // packed E2M1 values and a scale per 16; its fp32 tensor scales: [0] Wg and
  // Wu together, [1] Wd
  float* nv_scale = nullptr;
  // The separate-kernel BF16 forward leaves the sorted X rows in Xg; the
  // backward of that same forward (same X, saved context and T, no forward
  // in between) reads them instead of gathering X again.
  const void* xg_X = nullptr;
  const void* xg_saved = nullptr;
  int64_t xg_T = -1;
  // MOE_DEBUG_DUMP_QUANT: fp32 values the fused epilogues quantise (h, dA|dB)
  float *dbg_h = nullptr, *dbg_dab = nullptr;
  // ring-buffer forward megakernel (BF16): ring slots of X and h rows, GPU-local
  // hand-off counters, minibatch table
  void* ring_ws = nullptr;
  void* ring_h = nullptr;   // BF16 ring: slots of h rows (X rows go to their sorted rows in Xg)
  int* counters = nullptr;  // claim | gathered[NM] | mb_done[NM] | g1_done[NM]
  int32_t *mb_start = nullptr, *phase_start = nullptr, *n_mb = nullptr;
  int movers = 0, slots = 0, mbt = 0, cap = 0, nm_max = 0;
  int mx_movers = 0;   // mover CTAs of the MXFP8 ring megakernel
  CUtensorMap m_ring_h, m_ring_h_st;
  // one-launch forward: per-(token, 256-column block) arrival counts of the
  // in-kernel combine; grid-barrier arrivals and CTA exits (zero between launches)
  int* tok_cnt = nullptr;
  int* tok_u = nullptr;   // backward megakernel: <u, h> partials stored per token
  unsigned long long* gbar = nullptr;
  // router GEMM backward: dlogits in bf16 [T_max, E]
  void* dlg_bf16 = nullptr;
  float* router_part = nullptr;   // split-K partial sums of the router GEMMs
  // virtual-rank expert parallelism (ep_ranks >= 2): home slots of the pushed
  // rows [T_max * k, d] bf16, of the pushed <u, h> partials, and the flags
  void* ep_ws = nullptr;
  void* ep_slot = nullptr;
  float* ep_dgslot = nullptr;
  int* ep_ctr = nullptr;
  // timing (MOE_DEBUG_TIMING)
  std::vector<TimedLaunch> timed;
  std::vector<cudaEvent_t> spare_events;
};

namespace {
// K splits for a router GEMM with `tiles` output tiles and nkb K blocks: enough
// to fill about one wave of the SMs, at most kRouterMaxSplit and nkb.
constexpr int kRouterMaxSplit = 8;
int router_splits(const moe_plan_s* p, int64_t tiles, int64_t nkb) {
  if (tiles >= p->num_sms) return 1;
  return (int)std::max<int64_t>(1, std::min<int64_t>({p->num_sms / tiles, nkb, (int64_t)kRouterMaxSplit}));
}
}  // namespace

namespace {

cudaEvent_t take_event(moe_plan_s* p) {
  if (!p->spare_events.empty()) {
    cudaEvent_t e = p->spare_events.back();
    p->spare_events.pop_back();
    return e;
  }
  cudaEvent_t e = nullptr;
  cudaEventCreate(&e);
  return e;
}

// Launch `fn` on `st`; in timing mode bracket it with a pair of events.
template <class Fn>
cudaError_t timed_launch(moe_plan_s* p, const char* name, cudaStream_t st, Fn&& fn) {
  if (!(p->cfg.debug_flags & MOE_DEBUG_TIMING)) return fn();
  TimedLaunch t{name, take_event(p), take_event(p)};
  cudaEventRecord(t.a, st);
  cudaError_t e = fn();
  cudaEventRecord(t.b, st);
  p->timed.push_back(t);
  return e;
}

bool ensure_weight_maps(moe_plan_s* p, const void* Wg, const void* Wu, const void* Wd) {
  const moe_config_t& c = p->cfg;
  const uint64_t EF = (uint64_t)c.E * c.F, Ed = (uint64_t)c.E * c.d;
  if (Wg != p->p_wg) {
    if (!map_kmajor(&p->m_Wg_k, Wg, c.d, EF) || !map_mnmajor(&p->m_Wg_mn, Wg, c.d, EF)) return false;
    p->p_wg = Wg;
  }
  if (Wu != p->p_wu) {
    if (!map_kmajor(&p->m_Wu_k, Wu, c.d, EF) || !map_mnmajor(&p->m_Wu_mn, Wu, c.d, EF)) return false;
    p->p_wu = Wu;
  }
  if (Wd != p->p_wd) {
    if (!map_kmajor(&p->m_Wd_k, Wd, c.F, Ed, BN) || !map_mnmajor(&p->m_Wd_mn, Wd, c.F, Ed)) return false;
    p->p_wd = Wd;
  }
  return true;
}

// Grid of the persistent expert GEMMs: one CTA per SM.
int gemm_grid(const moe_plan_s* p) { return p->num_sms; }

// Virtual-rank expert parallelism: the argument block shared by its three
// exchanges (R ranks of G CTAs each).
EpArgs ep_args(moe_plan_s* p, const RoutingPtrs& rp, int64_t T) {
  const moe_config_t& c = p->cfg;
  EpArgs a;
  memset(&a, 0, sizeof(a));
  a.R = c.ep_ranks;
  a.G = std::max(1, 2 * p->num_sms / c.ep_ranks);  // two CTAs per SM (all co-resident)
  a.T = (int)T;
  a.d = c.d;
  a.F = c.F;
  a.E = c.E;
  a.k = c.k;
  a.ntu = c.prec == MOE_BF16 ? c.F / BN : c.F / 128;   // <u, h> partials per row of the u GEMM kind
  a.nch = route_chunks((int)T);
  a.rp = rp;
  a.chunk_hist = p->chunk_hist;
  a.chunk_base = p->chunk_base;
  a.slot = static_cast<uint4*>(p->ep_slot);
  a.dgslot = p->ep_dgslot;
  a.ctr = p->ep_ctr;
  a.status = p->status;
  a.timeout_ns = (uint64_t)c.wait_timeout_ns;
  return a;
}

// Ring-pipeline fields of the BF16 forward megakernel's argument block.
MegaArgs mega_args(moe_plan_s* p, const RoutingPtrs& rp, const void* X, const CUtensorMap& m_ab_st) {
  const moe_config_t& c = p->cfg;
  MegaArgs m;
  memset(&m, 0, sizeof(m));
  m.mapXr = p->m_Xg_k;
  m.mapWg = p->m_Wg_k;
  m.mapWu = p->m_Wu_k;
  m.mapWd = p->m_Wd_k;
  m.mapHr = p->m_ring_h;
  m.mapHrSt = p->m_ring_h_st;
  m.mapABSt = m_ab_st;
  m.mapYsSt = p->m_Ys_st;
  m.X = reinterpret_cast<const uint4*>(X);
  m.xg = reinterpret_cast<uint4*>(p->Xg);
  m.perm_src = rp.perm_src;
  m.mtile_off = rp.mtile_off;
  m.mb_start = p->mb_start;
  m.phase_start = p->phase_start;
  m.n_mb = p->n_mb;
  m.claim = p->counters;
  m.gathered = p->counters + 1;
  m.mb_done = p->counters + 1 + p->nm_max;
  m.g1_done = p->counters + 1 + 2 * p->nm_max;
  m.status = p->status;
  m.timeout_ns = (uint64_t)c.wait_timeout_ns;
  m.E = c.E;
  m.d = c.d;
  m.F = c.F;
  m.k = c.k;
  m.movers = p->movers;
  m.slots = p->slots;
  m.slot_rows = p->cap * BM;
  return m;
}

// Argument block of the MXFP8 ring megakernel (both forms).
MegaMxArgs mx_mega_args(moe_plan_s* p, const RoutingPtrs& rp, const CUtensorMap& m_ab_st) {
  const moe_config_t& c = p->cfg;
  MegaMxArgs m;
  memset(&m, 0, sizeof(m));
  m.mapXr = p->m_ring_xq;
  m.mapWg = p->m_Wgq;
  m.mapWu = p->m_Wuq;
  m.mapWd = p->m_Wdq;
  m.mapHr = p->m_ring_hq;
  m.mapHrSt = p->m_ring_hq_st;
  m.mapABSt = m_ab_st;
  m.mapYsSt = p->m_Ys_st;
  m.xq = p->Xtq;
  m.xs = p->Xts;
  m.ring_xq = p->ring_xq;
  m.ring_xs = p->ring_xs;
  m.ring_hs = p->ring_hs;
  m.wgs = p->Wgs;
  m.wus = p->Wus;
  m.wds = p->Wds;
  m.perm_src = rp.perm_src;
  m.mtile_off = rp.mtile_off;
  m.mb_start = p->mb_start;
  m.phase_start = p->phase_start;
  m.n_mb = p->n_mb;
  m.claim = p->counters;
  m.gathered = p->counters + 1;
  m.mb_done = p->counters + 1 + p->nm_max;
  m.g1_done = p->counters + 1 + 2 * p->nm_max;
  m.status = p->status;
  m.timeout_ns = (uint64_t)c.wait_timeout_ns;
  m.E = c.E;
  m.d = c.d;
  m.F = c.F;
  m.k = c.k;
  m.movers = p->mx_movers;
  m.slots = p->slots;
  m.slot_rows = p->cap * BM;
  return m;
}

GemmArgs base_args(moe_plan_s* p, const RoutingPtrs& rp) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.poff = rp.poff;
  a.mtile_off = rp.mtile_off;
  a.status = p->status;
  a.timeout_ns = (uint64_t)p->cfg.wait_timeout_ns;
  a.E = p->cfg.E;
  a.d = p->cfg.d;
  a.F = p->cfg.F;
  return a;
}

// Quantise the plan's whole sorted-row capacity of bf16 rows along d into the
// block-scaled sorted operand (Xq / Xs): MXFP8, or NVFP4 with tensor scale 1.
// Rows past the last expert segment are never read by a GEMM tile.
cudaError_t launch_quant_sorted(moe_plan_s* p, const void* rows, cudaStream_t st) {
  const moe_config_t& c = p->cfg;
  return c.prec == MOE_NVFP4 ? launch_nv_quant_rows(rows, p->Rpm, c.d, nullptr, p->Xq, p->Xs, p->num_sms * 8, st)
                             : launch_quant_rows(rows, p->Rpm, c.d, p->Xq, p->Xs, p->num_sms * 8, st);
}

// Block-scaled (MXFP8 / NVFP4) forward expert GEMMs over the plan's sorted,
// quantised X rows (Xq / Xs): [a|b] GEMM + SwiGLU with h re-quantised along F
// in its epilogue, then the down GEMM into Ys.
cudaError_t launch_block_scaled_fwd_gemms(moe_plan_s* p, const RoutingPtrs& rp, const CUtensorMap& m_ab_st,
                                          const CUtensorMap& m_ab_st16, cudaStream_t st) {
  const moe_config_t& c = p->cfg;
  const bool nv = c.prec == MOE_NVFP4;
  MxArgs a;
  memset(&a, 0, sizeof(a));
  a.poff = rp.poff;
  a.mtile_off = rp.mtile_off;
  a.status = p->status;
  a.timeout_ns = (uint64_t)c.wait_timeout_ns;
  a.E = c.E;
  a.d = c.d;
  a.F = c.F;
  MxArgs b = a;
  a.mapA = p->m_Xq;
  a.mapB0 = p->m_Wgq;
  a.mapB1 = p->m_Wuq;
  a.mapO0 = nv ? m_ab_st16 : m_ab_st;
  a.mapO1 = p->m_Hq_st;
  a.sfA = p->Xs;
  a.sfB0 = p->Wgs;
  a.sfB1 = p->Wus;
  a.sfO = p->Hs;
  a.tsB = nv ? p->nv_scale : nullptr;
  a.dbg = p->dbg_h;
  cudaError_t err = timed_launch(p, nv ? "gemm_nv_up_swiglu" : "gemm_mx_up_swiglu", st,
                     [&] { return launch_gemm_mx(kUp, a, p->num_sms, st, nv); });
  if (err != cudaSuccess) return err;
  b.mapA = p->m_Hq_k;
  b.mapB0 = p->m_Wdq;
  b.mapO0 = nv ? p->m_Ys_st16 : p->m_Ys_st;
  b.sfA = p->Hs;
  b.sfB0 = p->Wds;
  b.tsB = nv ? p->nv_scale + 1 : nullptr;
  err = timed_launch(p, nv ? "gemm_nv_down" : "gemm_mx_down", st,
                     [&] { return launch_gemm_mx(kDown, b, p->num_sms, st, nv); });
  return err;
}

// Block-scaled dgrad GEMMs over the plan's sorted, quantised dY rows (Xq /
// Xs): u GEMM against Wd^T with the SwiGLU-backward epilogue (dA|dB
// re-quantised along F, and the weight gradients' [dA|dB]^T and (w h)^T
// quantised along the rows), then the dx GEMM into Ys.
cudaError_t launch_block_scaled_dgrad_gemms(moe_plan_s* p, const RoutingPtrs& rp, const __nv_bfloat16* ab,
                                            cudaStream_t st) {
  const moe_config_t& c = p->cfg;
  const bool nv = c.prec == MOE_NVFP4;
  MxArgs u;
  memset(&u, 0, sizeof(u));
  u.poff = rp.poff;
  u.mtile_off = rp.mtile_off;
  u.status = p->status;
  u.timeout_ns = (uint64_t)c.wait_timeout_ns;
  u.E = c.E;
  u.d = c.d;
  u.F = c.F;
  MxArgs x = u;
  u.mapA = p->m_Xq;
  u.mapB0 = p->m_WdTq;
  u.mapO0 = p->m_dAB_st;
  u.mapO1 = p->m_dABq_st;
  u.mapO2 = p->m_wH_st;
  u.sfA = p->Xs;
  u.sfB0 = p->WdTs;
  u.sfO = p->dABs;
  u.ab = ab;
  u.perm_src = rp.perm_src;
  u.wts = rp.w;
  u.dgp = p->dgp;
  u.tsB = nv ? p->nv_scale + 1 : nullptr;
  u.dbg = p->dbg_dab;
  // the weight gradients' [dA|dB]^T and (w h)^T, quantised along the sorted
  // rows in the same epilogue
  u.Kcap = (int)p->Rpm;
  u.qT0 = p->dABTq;
  u.sT0 = p->dABTs;
  u.qT1 = p->wHTq;
  u.sT1 = p->wHTs;
  cudaError_t err = timed_launch(p, nv ? "gemm_nv_bwd_u_swiglu" : "gemm_mx_bwd_u_swiglu", st,
                     [&] { return launch_gemm_mx(kBwdU, u, p->num_sms, st, nv); });
  if (err != cudaSuccess) return err;
  x.mapA = p->m_dABq_k;
  x.mapB0 = p->m_WgTq;
  x.mapB1 = p->m_WuTq;
  x.mapO0 = nv ? p->m_Ys_st16 : p->m_Ys_st;
  x.sfA = p->dABs;
  x.sfB0 = p->WgTs;
  x.sfB1 = p->WuTs;
  x.tsB = nv ? p->nv_scale : nullptr;
  err = timed_launch(p, nv ? "gemm_nv_bwd_dx" : "gemm_mx_bwd_dx", st,
                     [&] { return launch_gemm_mx(kBwdX, x, p->num_sms, st, nv); });
  return err;
}

}  // namespace

void moe::set_error_detail(const char* msg) { g_last_error = msg ? msg : ""; }

// ============================================================================ C ABI
extern "C" {

const char* moe_status_string(moe_status_t s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or option";
    case MOE_ERR_OOM: return "device memory allocation failed";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_TIMEOUT: return "device-side wait timed out";
    case MOE_ERR_INTERNAL: return "internal error";
  }
  return "unknown status";
}

const char* moe_last_error(void) { return g_last_error.c_str(); }

moe_status_t moe_minibatch_floor(int32_t num_sms, int32_t tile_m, int32_t tile_n, int32_t n_out, int32_t waves,
                                 int64_t* rows) {
  if (!rows || num_sms <= 0 || tile_m <= 0 || tile_n <= 0 || n_out <= 0 || waves <= 0)
    return fail(MOE_ERR_INVALID_ARG, "moe_minibatch_floor: all arguments must be positive");
  const int64_t num = (int64_t)waves * num_sms * tile_m * tile_n;
  *rows = (num + n_out - 1) / n_out;
  return MOE_OK;
}

moe_status_t moe_plan(const moe_config_t* cfg, moe_plan_t* out) {
  if (!cfg || !out) return fail(MOE_ERR_INVALID_ARG, "moe_plan: null argument");
  *out = nullptr;
  const moe_config_t c = *cfg;
  if (c.T_max < 1 || c.T_max > (1 << 20)) return fail(MOE_ERR_INVALID_ARG, "moe_plan: T_max must be in [1, 2^20]");
  if (c.k < 1 || c.k > 32 || c.E < c.k || c.E > 1024)
    return fail(MOE_ERR_UNSUPPORTED, "moe_plan: need 1 <= k <= 32 and k <= E <= 1024");
  if (c.d <= 0 || c.F <= 0 || c.d % BN || c.F % BN)
    return fail(MOE_ERR_UNSUPPORTED, "moe_plan: d and F must be positive multiples of 256");
  if (c.prec != MOE_BF16 && c.prec != MOE_MXFP8 && c.prec != MOE_NVFP4)
    return fail(MOE_ERR_UNSUPPORTED, "moe_plan: prec must be MOE_BF16, MOE_MXFP8 or MOE_NVFP4");
  if ((int64_t)c.E * c.F * c.d >= (int64_t)1 << 40)
    return fail(MOE_ERR_UNSUPPORTED, "moe_plan: weight tensor too large");
  if (c.ep_ranks < 0 || c.ep_ranks > 64)
    return fail(MOE_ERR_INVALID_ARG, "moe_plan: ep_ranks must be in [0, 64]");
  if (c.ep_ranks >= 2 && (c.E % c.ep_ranks != 0 || (c.debug_flags & MOE_DEBUG_IDENTITY_EXPERTS)))
    return fail(MOE_ERR_UNSUPPORTED, "moe_plan: virtual-rank expert parallelism needs ep_ranks dividing E and real "
                                     "experts");
  if (!encode_fn()) return fail(MOE_ERR_CUDA, "moe_plan: cuTensorMapEncodeTiled unavailable");

  DeviceGuard guard(c.device);
  if (!guard.ok) return fail(MOE_ERR_CUDA, "moe_plan: cudaSetDevice failed");
  cudaDeviceProp prop;
  cudaError_t err = cudaGetDeviceProperties(&prop, c.device);
  if (err != cudaSuccess) return cuda_fail(err, "moe_plan: cudaGetDeviceProperties");
  if (prop.major != 10 || prop.minor != 3)
    return fail(MOE_ERR_UNSUPPORTED, "moe_plan: this library is built for sm_103a (GB300) only; device is sm_" +
                                         std::to_string(prop.major) + std::to_string(prop.minor));

  moe_plan_s* p = new (std::nothrow) moe_plan_s();
  if (!p) return fail(MOE_ERR_OOM, "moe_plan: host allocation failed");
  p->cfg = c;
  if (p->cfg.wait_timeout_ns <= 0) p->cfg.wait_timeout_ns = 2000000000LL;
  p->num_sms = prop.multiProcessorCount;
  const SavedLayout L = saved_layout(c, c.T_max);
  p->Rpm = L.rows;
  const int nch = route_chunks((int)c.T_max);

  size_t o = 0;
  const size_t o_hist = o;  o += align256((size_t)nch * c.E * 4);
  const size_t o_base = o;  o += align256((size_t)nch * c.E * 4);
  const size_t o_stat = o;  o += 256;
  const size_t o_xg = o;    o += align256((size_t)p->Rpm * c.d * 2);
  const size_t o_h = o;     o += align256((size_t)p->Rpm * c.F * 2);
  const size_t o_ys = o;    o += align256((size_t)p->Rpm * c.d * 2);
  const size_t o_dyg = o;   o += align256((size_t)p->Rpm * c.d * 2);
  const size_t o_dab = o;   o += align256((size_t)p->Rpm * 2 * c.F * 2);
  const size_t o_wh = o;    o += align256((size_t)p->Rpm * c.F * 2);
  const size_t o_dgp = o;   o += align256((size_t)p->Rpm * (c.F / 128) * 4);  // <u, h> partials
  err = cudaMalloc(&p->ws, o);
  if (err != cudaSuccess) {
    delete p;
    return fail(MOE_ERR_OOM, std::string("moe_plan: cudaMalloc of workspace failed: ") + cudaGetErrorString(err));
  }
  char* b = static_cast<char*>(p->ws);
  p->chunk_hist = reinterpret_cast<int32_t*>(b + o_hist);
  p->chunk_base = reinterpret_cast<int32_t*>(b + o_base);
  p->status = reinterpret_cast<int32_t*>(b + o_stat);
  p->Xg = b + o_xg;
  p->H = b + o_h;
  p->Ys = b + o_ys;
  p->dYg = b + o_dyg;
  p->dAB = b + o_dab;
  p->wH = b + o_wh;
  p->dgp = reinterpret_cast<float*>(b + o_dgp);
  err = cudaMemset(p->status, 0, 256);
  if (err != cudaSuccess) {
    cudaFree(p->ws);
    delete p;
    return cuda_fail(err, "moe_plan: cudaMemset");
  }
  const uint64_t R = p->Rpm;
  bool ok = map_kmajor(&p->m_Xg_k, p->Xg, c.d, R) && map_mnmajor(&p->m_Xg_mn, p->Xg, c.d, R) &&
            map_kmajor(&p->m_H_k, p->H, c.F, R) && map_store(&p->m_H_st, p->H, c.F, R) &&
            map_store(&p->m_Ys_st, p->Ys, c.d, R) && map_kmajor(&p->m_dYg_k, p->dYg, c.d, R) &&
            map_mnmajor(&p->m_dYg_mn, p->dYg, c.d, R) && map_kmajor(&p->m_dAB_k, p->dAB, 2 * c.F, R) &&
            map_mnmajor(&p->m_dAB_mn, p->dAB, 2 * c.F, R) && map_store(&p->m_dAB_st, p->dAB, 2 * c.F, R) &&
            map_mnmajor(&p->m_wH_mn, p->wH, c.F, R) && map_store(&p->m_wH_st, p->wH, c.F, R);
  if (!ok) {
    cudaFree(p->ws);
    delete p;
    return fail(MOE_ERR_CUDA, "moe_plan: tensor map encoding failed");
  }
  for (int kind = 0; kind < 6; ++kind) {
    err = kind < 2 ? prepare_gemm_fwd(kind) : prepare_gemm_bwd(kind);
    if (err == cudaSuccess && c.prec != MOE_BF16) err = prepare_gemm_mx(kind, c.prec == MOE_NVFP4);
    if (err == cudaSuccess && kind == 0 && c.prec != MOE_BF16) err = prepare_gather_transpose_q(c.prec == MOE_NVFP4);
    if (err != cudaSuccess) {
      cudaFree(p->ws);
      delete p;
      return cuda_fail(err, "moe_plan: cudaFuncSetAttribute");
    }
  }
  {
    // ring token buffer: `slots` slots of `cap` 128-row tiles; minibatches of
    // at least `mbt` tiles (the two-wave floor over the compute SMs)
    // BF16: 0 mover CTAs by default (two mover warps in every compute CTA);
    // the MXFP8 ring keeps dedicated mover CTAs
    p->movers = c.mover_ctas > 0 ? c.mover_ctas : 0;
    p->mx_movers = c.mover_ctas > 0 ? c.mover_ctas : 8;
    p->slots = c.ring_slots > 0 ? c.ring_slots : 4;
    if (p->mx_movers >= p->num_sms - 1 || p->slots < 2) {
      cudaFree(p->ws);
      delete p;
      return fail(MOE_ERR_INVALID_ARG, "moe_plan: need 2 <= ring_slots and mover_ctas < SM count - 1");
    }
    int64_t mb_rows = c.minibatch_rows;
    if (mb_rows <= 0)
      moe_minibatch_floor(p->num_sms - (c.prec == MOE_BF16 ? p->movers : p->mx_movers), BM, 128, c.F, 2, &mb_rows);
    p->mbt = (int)std::max<int64_t>(1, (mb_rows + BM - 1) / BM);
    p->cap = 2 * p->mbt;
    p->nm_max = (int)(p->Rpm / BM);
    const size_t slot_rows = (size_t)p->cap * BM;
    size_t m = 0;
    const size_t o_rh = m; m += align256(p->slots * slot_rows * c.F * 2);
    const size_t o_ct = m; m += align256((1 + 3 * (size_t)p->nm_max) * 4);
    const size_t o_mb = m; m += align256(((size_t)p->nm_max + 1) * 4);
    const size_t o_ph = m; m += align256((2 * (size_t)p->nm_max + 1) * 4);
    const size_t o_nm = m; m += 256;
    const size_t o_gb = m; m += 256;
    const size_t o_tc = m; m += align256((size_t)c.T_max * (c.d / BN) * 4);
    const size_t o_tu = m; m += align256((size_t)c.T_max * 4);
    err = cudaMalloc(&p->ring_ws, m);
    if (err != cudaSuccess) {
      cudaFree(p->ws);
      delete p;
      return fail(MOE_ERR_OOM, std::string("moe_plan: cudaMalloc of ring buffer failed: ") + cudaGetErrorString(err));
    }
    char* rb = static_cast<char*>(p->ring_ws);
    p->ring_h = rb + o_rh;
    p->counters = reinterpret_cast<int*>(rb + o_ct);
    p->mb_start = reinterpret_cast<int32_t*>(rb + o_mb);
    p->phase_start = reinterpret_cast<int32_t*>(rb + o_ph);
    p->n_mb = reinterpret_cast<int32_t*>(rb + o_nm);
    p->gbar = reinterpret_cast<unsigned long long*>(rb + o_gb);
    p->tok_cnt = reinterpret_cast<int*>(rb + o_tc);
    p->tok_u = reinterpret_cast<int*>(rb + o_tu);
    err = cudaMemset(p->gbar, 0, 2 * sizeof(unsigned long long));
    if (err != cudaSuccess) {
      cudaFree(p->ring_ws);
      cudaFree(p->ws);
      delete p;
      return cuda_fail(err, "moe_plan: cudaMemset of the grid-barrier counter");
    }
    const uint64_t ring_rows = p->slots * slot_rows;
    ok = map_kmajor(&p->m_ring_h, p->ring_h, c.F, ring_rows) && map_store(&p->m_ring_h_st, p->ring_h, c.F, ring_rows);
    err = prepare_fwd_megakernel();
    if (err == cudaSuccess) err = prepare_bwd_megakernel();
    if (!ok || err != cudaSuccess) {
      cudaFree(p->ring_ws);
      cudaFree(p->ws);
      delete p;
      return fail(MOE_ERR_CUDA, "moe_plan: ring buffer tensor maps / megakernel attribute");
    }
  }
  if (c.prec == MOE_MXFP8 || c.prec == MOE_NVFP4) {
    // quantised weights (both orientations), activations and their scale
    // atoms: MXFP8 one byte per value and a scale per 32 values, NVFP4 half a
    // byte per value and a scale per 16 (plus the two tensor scales)
    const bool nv = c.prec == MOE_NVFP4;
    const size_t nw = (size_t)c.E * c.F * c.d;  // values of one weight tensor
    auto qb = [nv](size_t v) { return nv ? v / 2 : v; };
    auto sb = [nv](size_t v) { return nv ? v / 16 : v / 32; };
    size_t m = 0;
    const size_t o_wgq = m; m += align256(qb(nw));
    const size_t o_wuq = m; m += align256(qb(nw));
    const size_t o_wdq = m; m += align256(qb(nw));
    const size_t o_wgs = m; m += align256(sb(nw));
    const size_t o_wus = m; m += align256(sb(nw));
    const size_t o_wds = m; m += align256(sb(nw));
    const size_t o_xq = m;  m += align256(qb((size_t)R * c.d));
    const size_t o_xs = m;  m += align256(sb((size_t)R * c.d));
    const size_t o_hq = m;  m += align256(qb((size_t)R * c.F));
    const size_t o_hs = m;  m += align256(sb((size_t)R * c.F));
    const size_t o_wdt = m; m += align256(qb(nw));
    const size_t o_wgt = m; m += align256(qb(nw));
    const size_t o_wut = m; m += align256(qb(nw));
    const size_t o_wdts = m; m += align256(sb(nw));
    const size_t o_wgts = m; m += align256(sb(nw));
    const size_t o_wuts = m; m += align256(sb(nw));
    const size_t o_dabq = m; m += align256(qb((size_t)R * 2 * c.F));
    const size_t o_dabs = m; m += align256(sb((size_t)R * 2 * c.F));
    // MXFP8 ring slots (an NVFP4 plan runs the separate-kernel schedule only)
    const size_t ring_rows = nv ? 0 : (size_t)p->slots * p->cap * BM;
    const size_t o_rxq = m; m += align256(ring_rows * c.d);
    const size_t o_rxs = m; m += align256(ring_rows * c.d / 32);
    const size_t o_rhq = m; m += align256(ring_rows * c.F);
    const size_t o_rhs = m; m += align256(ring_rows * c.F / 32);
    const size_t t_pad = ((size_t)c.T_max + BM - 1) / BM * BM;
    const size_t o_xtq = m; m += align256(qb(t_pad * c.d));
    const size_t o_xts = m; m += align256(sb(t_pad * c.d));
    const size_t o_nvs = m; m += 256;
    // transposed, token-wise quantised weight-gradient operands; 4 KB of slack
    // after each scale buffer covers an NVFP4 half stage's unused atoms
    const size_t o_dytq = m; m += align256(qb((size_t)c.d * R));
    const size_t o_dyts = m; m += align256(sb((size_t)c.d * R)) + 4096;
    const size_t o_xtrq = m; m += align256(qb((size_t)c.d * R));
    const size_t o_xtrs = m; m += align256(sb((size_t)c.d * R)) + 4096;
    const size_t o_dabtq = m; m += align256(qb((size_t)2 * c.F * R));
    const size_t o_dabts = m; m += align256(sb((size_t)2 * c.F * R)) + 4096;
    const size_t o_whtq = m; m += align256(qb((size_t)c.F * R));
    const size_t o_whts = m; m += align256(sb((size_t)c.F * R)) + 4096;
    const bool dump = (c.debug_flags & MOE_DEBUG_DUMP_QUANT) != 0;
    const size_t o_dbh = m; m += dump ? align256((size_t)R * c.F * 4) : 0;
    const size_t o_dbd = m; m += dump ? align256((size_t)R * 2 * c.F * 4) : 0;
    err = cudaMalloc(&p->mx_ws, m);
    if (err != cudaSuccess) {
      if (p->ring_ws) cudaFree(p->ring_ws);
      cudaFree(p->ws);
      delete p;
      return fail(MOE_ERR_OOM, std::string("moe_plan: cudaMalloc of the block-scaled workspace failed: ") +
                                   cudaGetErrorString(err));
    }
    uint8_t* mb = static_cast<uint8_t*>(p->mx_ws);
    p->Wgq = mb + o_wgq; p->Wuq = mb + o_wuq; p->Wdq = mb + o_wdq;
    p->Wgs = mb + o_wgs; p->Wus = mb + o_wus; p->Wds = mb + o_wds;
    p->Xq = mb + o_xq; p->Xs = mb + o_xs; p->Hq = mb + o_hq; p->Hs = mb + o_hs;
    p->WdTq = mb + o_wdt; p->WgTq = mb + o_wgt; p->WuTq = mb + o_wut;
    p->WdTs = mb + o_wdts; p->WgTs = mb + o_wgts; p->WuTs = mb + o_wuts;
    p->dABq = mb + o_dabq; p->dABs = mb + o_dabs;
    p->ring_xq = mb + o_rxq; p->ring_xs = mb + o_rxs; p->ring_hq = mb + o_rhq; p->ring_hs = mb + o_rhs;
    p->Xtq = mb + o_xtq; p->Xts = mb + o_xts;
    p->nv_scale = reinterpret_cast<float*>(mb + o_nvs);
    p->dYTq = mb + o_dytq; p->dYTs = mb + o_dyts; p->XTq = mb + o_xtrq; p->XTs = mb + o_xtrs;
    p->dABTq = mb + o_dabtq; p->dABTs = mb + o_dabts; p->wHTq = mb + o_whtq; p->wHTs = mb + o_whts;
    if (dump) {
      p->dbg_h = reinterpret_cast<float*>(mb + o_dbh);
      p->dbg_dab = reinterpret_cast<float*>(mb + o_dbd);
    }
    const uint64_t EF = (uint64_t)c.E * c.F, Ed = (uint64_t)c.E * c.d;
    const uint32_t qbox = nv ? 16 : 32;  // bytes of 32 quantised values
    ok = map_fp8_kmajor(&p->m_Wgq, p->Wgq, qb(c.d), EF) && map_fp8_kmajor(&p->m_Wuq, p->Wuq, qb(c.d), EF) &&
         map_fp8_kmajor(&p->m_Wdq, p->Wdq, qb(c.F), Ed, BN) && map_fp8_kmajor(&p->m_Xq, p->Xq, qb(c.d), R) &&
         map_fp8_kmajor(&p->m_Hq_k, p->Hq, qb(c.F), R) && map_fp8_store(&p->m_Hq_st, p->Hq, qb(c.F), R, qbox) &&
         map_fp8_kmajor(&p->m_WdTq, p->WdTq, qb(c.d), EF, BN) &&
         map_fp8_kmajor(&p->m_WgTq, p->WgTq, qb(c.F), Ed, BN) &&
         map_fp8_kmajor(&p->m_WuTq, p->WuTq, qb(c.F), Ed, BN) &&
         map_fp8_kmajor(&p->m_dABq_k, p->dABq, qb(2 * c.F), R) &&
         map_fp8_store(&p->m_dABq_st, p->dABq, qb(2 * c.F), R, qbox) &&
         (!nv || map_store16(&p->m_Ys_st16, p->Ys, c.d, R)) &&
         map_fp8_kmajor(&p->m_dYTq, p->dYTq, qb(R), c.d) && map_fp8_kmajor(&p->m_XTq, p->XTq, qb(R), c.d, BN) &&
         map_fp8_kmajor(&p->m_dABTq, p->dABTq, qb(R), 2 * c.F) &&
         map_fp8_kmajor(&p->m_wHTq, p->wHTq, qb(R), c.F, BN);
    if (ok && !nv)
      ok = map_fp8_kmajor(&p->m_ring_xq, p->ring_xq, c.d, ring_rows) &&
           map_fp8_kmajor(&p->m_ring_hq, p->ring_hq, c.F, ring_rows) &&
           map_fp8_store(&p->m_ring_hq_st, p->ring_hq, c.F, ring_rows) && prepare_fwd_megakernel_mx() == cudaSuccess;
    if (!ok) {
      cudaFree(p->mx_ws);
      if (p->ring_ws) cudaFree(p->ring_ws);
      cudaFree(p->ws);
      delete p;
      return fail(MOE_ERR_CUDA, "moe_plan: block-scaled tensor map encoding failed");
    }
  }
  // router GEMM backward: dlogits rounded to bf16 for the tensor cores
  err = cudaMalloc(&p->dlg_bf16, (size_t)std::max<int64_t>(1, c.T_max) * c.E * 2);
  if (err == cudaSuccess) {
    // split-K partials: the logits GEMM splits only while S * ceil(T/128) <=
    // SMs (so S * T <= 128 * SMs) and S <= 8; the dWr GEMM at most its
    // largest split of E x d
    const int64_t fwd = std::min<int64_t>(128 * (int64_t)p->num_sms, kRouterMaxSplit * std::max<int64_t>(1, c.T_max)) *
                        c.E;
    const int64_t tiles_w = ((c.E + BM - 1) / BM) * (c.d / BN);
    const int64_t dw = (int64_t)router_splits(p, tiles_w, kRouterMaxSplit) * c.E * c.d;
    err = cudaMalloc(&p->router_part, (size_t)std::max(fwd, dw) * sizeof(float));
  }
  if (err == cudaSuccess) err = prepare_gemm_router();
  if (err == cudaSuccess && c.ep_ranks >= 2) {
    const size_t pairs = (size_t)c.T_max * c.k;
    // <u, h> partials per pair: F/256 (bf16 u GEMM) or F/128 (block-scaled)
    const size_t ntu = c.prec == MOE_BF16 ? c.F / BN : c.F / 128;
    const size_t o_slot = 0, o_dgs = align256(pairs * c.d * 2), o_ctr = o_dgs + align256(pairs * ntu * 4);
    err = cudaMalloc(&p->ep_ws, o_ctr + 4096);
    if (err == cudaSuccess) {
      char* eb = static_cast<char*>(p->ep_ws);
      p->ep_slot = eb + o_slot;
      p->ep_dgslot = reinterpret_cast<float*>(eb + o_dgs);
      p->ep_ctr = reinterpret_cast<int*>(eb + o_ctr);
      err = cudaMemset(p->ep_ctr, 0, 4096);
    }
    if (err == cudaSuccess) err = prepare_ep();
  }
  if (err != cudaSuccess) {
    if (p->ep_ws) cudaFree(p->ep_ws);
    if (p->dlg_bf16) cudaFree(p->dlg_bf16);
    if (p->router_part) cudaFree(p->router_part);
    if (p->mx_ws) cudaFree(p->mx_ws);
    if (p->ring_ws) cudaFree(p->ring_ws);
    cudaFree(p->ws);
    delete p;
    return cuda_fail(err, "moe_plan: router workspace / GEMM attribute");
  }
  *out = p;
  return MOE_OK;
}

moe_status_t moe_plan_destroy(moe_plan_t p) {
  if (!p) return MOE_OK;
  DeviceGuard guard(p->cfg.device);
  cudaDeviceSynchronize();
  for (auto& t : p->timed) {
    cudaEventDestroy(t.a);
    cudaEventDestroy(t.b);
  }
  for (auto e : p->spare_events) cudaEventDestroy(e);
  if (p->mx_ws) cudaFree(p->mx_ws);
  if (p->ring_ws) cudaFree(p->ring_ws);
  if (p->dlg_bf16) cudaFree(p->dlg_bf16);
  if (p->router_part) cudaFree(p->router_part);
  if (p->ep_ws) cudaFree(p->ep_ws);
  cudaError_t err = cudaFree(p->ws);
  delete p;
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_plan_destroy: cudaFree");
}

moe_status_t moe_plan_info(moe_plan_t p, int32_t* num_sms, int32_t* ring) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "moe_plan_info: null plan");
  if (num_sms) *num_sms = p->num_sms;
  if (ring) {
    ring[0] = p->cfg.prec == MOE_BF16 ? p->movers : p->mx_movers;
    ring[1] = p->slots;
    ring[2] = p->mbt;
    ring[3] = p->cap;
  }
  return MOE_OK;
}

moe_status_t moe_saved_bytes(moe_plan_t p, int64_t T, size_t* bytes) {
  if (!p || !bytes) return fail(MOE_ERR_INVALID_ARG, "moe_saved_bytes: null argument");
  if (T < 0 || T > p->cfg.T_max) return fail(MOE_ERR_INVALID_ARG, "moe_saved_bytes: T outside [0, T_max]");
  *bytes = saved_layout(p->cfg, T).total;
  return MOE_OK;
}

moe_status_t moe_forward(moe_plan_t p, int64_t T, const void* X, const float* logits, const void* Wg,
                         const void* Wu, const void* Wd, void* Y, void* saved, moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "moe_forward: null plan");
  const moe_config_t& c = p->cfg;
  if (T < 0 || T > c.T_max) return fail(MOE_ERR_INVALID_ARG, "moe_forward: T outside [0, T_max]");
  if (T == 0) return MOE_OK;
  const bool ident = (c.debug_flags & MOE_DEBUG_IDENTITY_EXPERTS) != 0;
  if (!X || !logits || !Y || !saved || (!ident && (!Wg || !Wu || !Wd)))
    return fail(MOE_ERR_INVALID_ARG, "moe_forward: null tensor pointer");
  if (!aligned16(X) || !aligned16(Y) || (reinterpret_cast<uintptr_t>(saved) & 255u) ||
      (!ident && (!aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd))) ||
      (reinterpret_cast<uintptr_t>(logits) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "moe_forward: misaligned pointer (16 B tensors, 256 B saved)");
  DeviceGuard guard(c.device);
  if (!guard.ok) return fail(MOE_ERR_CUDA, "moe_forward: cudaSetDevice failed");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const SavedLayout L = saved_layout(c, T);
  const RoutingPtrs rp = routing_ptrs(L, saved);
  const int Ti = (int)T;
  cudaError_t err;
  p->xg_X = nullptr;  // set again below by the schedule that leaves X's sorted rows in Xg

  const bool mx = (c.prec == MOE_MXFP8 || c.prec == MOE_NVFP4) && !ident;  // block-scaled GEMMs
  const bool nv = c.prec == MOE_NVFP4;
  if (mx && !p->weights_quantized)
    return fail(MOE_ERR_INVALID_ARG, "moe_forward: block-scaled plan needs moe_quantize_weights before the forward");
  if (!ident && !ensure_weight_maps(p, Wg, Wu, Wd)) return fail(MOE_ERR_CUDA, "moe_forward: weight tensor maps");
  CUtensorMap m_ab_st, m_ab_st16;
  if (!ident && !map_store(&m_ab_st, static_cast<char*>(saved) + L.ab, 2 * c.F, L.rows))
    return fail(MOE_ERR_CUDA, "moe_forward: saved tensor map");
  if (mx && c.prec == MOE_NVFP4 && !map_store16(&m_ab_st16, static_cast<char*>(saved) + L.ab, 2 * c.F, L.rows))
    return fail(MOE_ERR_CUDA, "moe_forward: saved tensor map");

  // BF16 ring schedule, one launch: routing, layout, ring pipeline and
  // combine in one cooperative persistent kernel
  if (c.ep_ranks >= 2) {
    // expert parallelism over virtual ranks: routing + pull dispatch (one
    // cooperative launch), the grouped GEMMs over the ranks' regions, then
    // push combine with the home-side weighted sum
    EpArgs ea = ep_args(p, rp, T);
    ea.logits = logits;
    ea.X = reinterpret_cast<const uint4*>(X);
    ea.Xg = static_cast<uint4*>(p->Xg);
    err = timed_launch(p, "ep_pull_dispatch", st, [&] { return launch_ep_dispatch(ea, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: EP dispatch launch");
    if (mx) {
      // block-scaled experts: each rank quantises the bf16 rows it pulled
      // along d -- the bytes of quantising each token once and copying them,
      // as the single-GPU schedule does -- then the block-scaled GEMMs
      err = timed_launch(p, "quant_pulled_rows", st, [&] { return launch_quant_sorted(p, p->Xg, st); });
      if (err == cudaSuccess) err = launch_block_scaled_fwd_gemms(p, rp, m_ab_st, m_ab_st16, st);
      if (err != cudaSuccess) return cuda_fail(err, "moe_forward: EP block-scaled GEMM launch");
      ea.Ys = static_cast<const uint4*>(p->Ys);
      ea.out = static_cast<uint4*>(Y);
      ea.w_out = rp.w;
      err = timed_launch(p, "ep_push_combine", st, [&] { return launch_ep_push(ea, st); });
      if (err != cudaSuccess) return cuda_fail(err, "moe_forward: EP combine launch");
      return MOE_OK;
    }
    GemmArgs a = base_args(p, rp);
    a.mapA = p->m_Xg_k;
    a.mapB0 = p->m_Wg_k;
    a.mapB1 = p->m_Wu_k;
    a.mapO0 = m_ab_st;
    a.mapO1 = p->m_H_st;
    err = timed_launch(p, "gemm_up_swiglu", st,
                       [&] { return launch_gemm_fwd(kUp, a, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: up GEMM launch");
    GemmArgs b = base_args(p, rp);
    b.mapA = p->m_H_k;
    b.mapB0 = p->m_Wd_k;
    b.mapO0 = p->m_Ys_st;
    err = timed_launch(p, "gemm_down", st,
                       [&] { return launch_gemm_fwd(kDown, b, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: down GEMM launch");
    ea.Ys = static_cast<const uint4*>(p->Ys);
    ea.out = static_cast<uint4*>(Y);
    ea.w_out = rp.w;
    err = timed_launch(p, "ep_push_combine", st, [&] { return launch_ep_push(ea, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: EP combine launch");
    return MOE_OK;
  }
  const bool ring = (c.debug_flags & MOE_DEBUG_RING_MEGAKERNEL) && !(c.debug_flags & MOE_DEBUG_SEPARATE_KERNELS) &&
                    !(mx && (c.debug_flags & MOE_DEBUG_DUMP_QUANT));
  if (!mx && !ident && ring && !(c.debug_flags & MOE_DEBUG_MULTI_LAUNCH)) {
    MegaArgs m = mega_args(p, rp, X, m_ab_st);
    m.logits = logits;
    m.rp = rp;
    m.chunk_hist = p->chunk_hist;
    m.chunk_base = p->chunk_base;
    m.counters = p->counters;
    m.counters_len = 1 + 3 * p->nm_max;
    m.Ys = reinterpret_cast<const uint4*>(p->Ys);
    m.Y = reinterpret_cast<uint4*>(Y);
    m.tok_cnt = p->tok_cnt;
    m.gbar = p->gbar;
    m.T = Ti;
    m.mbt = p->mbt;
    m.cap = p->cap;
    err = timed_launch(p, "fwd_megakernel", st, [&] { return launch_fwd_megakernel(m, p->num_sms, true, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: one-launch megakernel launch");
    p->xg_X = X;   // the movers left X's sorted rows in Xg
    p->xg_saved = saved;
    p->xg_T = T;
    return MOE_OK;
  }
  if (mx && ring && !nv && !(c.debug_flags & MOE_DEBUG_MULTI_LAUNCH)) {
    // MXFP8 ring schedule, one launch: token quantisation, routing, layout,
    // ring pipeline and combine in one cooperative persistent kernel
    MegaMxArgs m = mx_mega_args(p, rp, m_ab_st);
    m.Xtok = static_cast<const __nv_bfloat16*>(X);
    m.logits = logits;
    m.rp = rp;
    m.chunk_hist = p->chunk_hist;
    m.chunk_base = p->chunk_base;
    m.counters = p->counters;
    m.counters_len = 1 + 3 * p->nm_max;
    m.Ys = reinterpret_cast<const uint4*>(p->Ys);
    m.Y = reinterpret_cast<uint4*>(Y);
    m.tok_cnt = p->tok_cnt;
    m.gbar = p->gbar;
    m.T = Ti;
    m.mbt = p->mbt;
    m.cap = p->cap;
    err = timed_launch(p, "fwd_megakernel_mx", st,
                       [&] { return launch_fwd_megakernel_mx(m, p->num_sms, true, st); });
    if (err != cudaSuccess) {
      const std::string why = g_last_error;
      cuda_fail(err, "moe_forward: MXFP8 one-launch megakernel launch");
      if (err == cudaErrorCooperativeLaunchTooLarge) g_last_error += " (" + why + ")";
      return MOE_ERR_CUDA;
    }
    return MOE_OK;
  }
  err = timed_launch(p, "router_topk_hist", st,
                     [&] { return launch_router(logits, Ti, c.E, c.k, p->chunk_hist, rp, st); });
  if (err == cudaSuccess)
    err = timed_launch(p, "layout_scan", st,
                       [&] { return launch_scan(Ti, c.E, p->chunk_hist, p->chunk_base, rp, st); });
  if (err == cudaSuccess)
    err = timed_launch(p, "layout_permute", st,
                       [&] { return launch_permute(Ti, c.E, c.k, p->chunk_base, rp, st); });
  if (err != cudaSuccess) return cuda_fail(err, "moe_forward: routing launch");
  if (mx && ring && !nv) {
    // MXFP8 ring megakernel: movers gather + quantise into the slots, compute
    // CTAs run the block-scaled [a|b]+SwiGLU (h re-quantised into the slot)
    // and down tiles minibatch by minibatch
    const int counters_len = 1 + 3 * p->nm_max;
    err = timed_launch(p, "plan_minibatches", st, [&] {
      return launch_plan_minibatches(rp.mtile_off, c.E, p->mbt, p->cap, c.F / 128, c.d / BN, counters_len,
                                     p->counters, p->mb_start, p->phase_start, p->n_mb, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: minibatch plan launch");
    err = timed_launch(p, "quant_tokens", st, [&] {
      return launch_quant_rows(X, T, c.d, p->Xtq, p->Xts, p->num_sms * 8, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: token quantisation launch");
    const MegaMxArgs m = mx_mega_args(p, rp, m_ab_st);
    err = timed_launch(p, "fwd_megakernel_mx", st,
                       [&] { return launch_fwd_megakernel_mx(m, p->num_sms, false, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: MXFP8 megakernel launch");
    const int cgrid = (int)std::min<int64_t>(T, (int64_t)p->num_sms * 16);
    err = timed_launch(p, "combine", st,
                       [&] { return launch_combine(p->Ys, rp.dest, rp.w, Ti, c.k, c.d, Y, cgrid, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: combine launch");
    return MOE_OK;
  }
  if (mx) {
    // MXFP8 / NVFP4: gather + quantise X along d, block-scaled [a|b] GEMM with
    // SwiGLU and h re-quantised along F in its epilogue, block-scaled down GEMM.
    // each token quantised once and its codes and scale words stored straight
    // into its k sorted rows (the same bytes as quantising every routed row)
    err = timed_launch(p, "quant_scatter", st, [&] {
      return launch_quant_scatter_rows(nv, X, rp.perm_src, rp.dest, rp.totals, (int)T, c.k, c.d, p->Xq, p->Xs,
                                       p->num_sms * 8, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: gather launch");
    err = launch_block_scaled_fwd_gemms(p, rp, m_ab_st, m_ab_st16, st);
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: block-scaled GEMM launch");
    const int cgrid = (int)std::min<int64_t>(T, (int64_t)p->num_sms * 16);
    err = timed_launch(p, "combine", st,
                       [&] { return launch_combine(p->Ys, rp.dest, rp.w, Ti, c.k, c.d, Y, cgrid, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: combine launch");
    return MOE_OK;
  }
  if (!ident && ring) {
    // one persistent launch: movers fill ring slots, compute CTAs run the
    // [a|b]+SwiGLU and down tiles minibatch by minibatch
    const int counters_len = 1 + 3 * p->nm_max;
    err = timed_launch(p, "plan_minibatches", st, [&] {
      return launch_plan_minibatches(rp.mtile_off, c.E, p->mbt, p->cap, c.F / 128, c.d / BN, counters_len,
                                     p->counters, p->mb_start, p->phase_start, p->n_mb, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: minibatch plan launch");
    const MegaArgs m = mega_args(p, rp, X, m_ab_st);
    err = timed_launch(p, "fwd_megakernel", st, [&] { return launch_fwd_megakernel(m, p->num_sms, false, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: megakernel launch");
    const int cgrid = (int)std::min<int64_t>(T, (int64_t)p->num_sms * 16);
    err = timed_launch(p, "combine", st,
                       [&] { return launch_combine(p->Ys, rp.dest, rp.w, Ti, c.k, c.d, Y, cgrid, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: combine launch");
    p->xg_X = X;
    p->xg_saved = saved;
    p->xg_T = T;
    return MOE_OK;
  }
  err = timed_launch(p, "gather", st, [&] {
    return launch_gather(X, nullptr, rp.perm_src, rp.dest, rp.totals, (int)T, c.k, c.d, p->Xg, nullptr,
                         p->num_sms * 8, st);
  });
  if (err != cudaSuccess) return cuda_fail(err, "moe_forward: gather launch");
  const void* ys = p->Xg;
  if (!ident) {
    GemmArgs a = base_args(p, rp);
    a.mapA = p->m_Xg_k;
    a.mapB0 = p->m_Wg_k;
    a.mapB1 = p->m_Wu_k;
    a.mapO0 = m_ab_st;
    a.mapO1 = p->m_H_st;
    a.stall = (c.debug_flags & MOE_DEBUG_STALL_TEST) ? 1 : 0;
    err = timed_launch(p, "gemm_up_swiglu", st,
                       [&] { return launch_gemm_fwd(kUp, a, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: up GEMM launch");
    GemmArgs b = base_args(p, rp);
    b.mapA = p->m_H_k;
    b.mapB0 = p->m_Wd_k;
    b.mapO0 = p->m_Ys_st;
    err = timed_launch(p, "gemm_down", st,
                       [&] { return launch_gemm_fwd(kDown, b, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_forward: down GEMM launch");
    ys = p->Ys;
  }
  const int cgrid = (int)std::min<int64_t>(T, (int64_t)p->num_sms * 16);
  err = timed_launch(p, "combine", st,
                     [&] { return launch_combine(ys, rp.dest, rp.w, Ti, c.k, c.d, Y, cgrid, st); });
  if (err != cudaSuccess) return cuda_fail(err, "moe_forward: combine launch");
  if (!ident) {
    p->xg_X = X;
    p->xg_saved = saved;
    p->xg_T = T;
  }
  return MOE_OK;
}

moe_status_t moe_backward(moe_plan_t p, int64_t T, const void* dY, const void* X, const void* Wg, const void* Wu,
                          const void* Wd, const void* saved, void* dX, void* dWg, void* dWu, void* dWd, float* dg,
                          float* dlogits, moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "moe_backward: null plan");
  const moe_config_t& c = p->cfg;
  if (c.debug_flags & MOE_DEBUG_IDENTITY_EXPERTS)
    return fail(MOE_ERR_UNSUPPORTED, "moe_backward: identity-expert debug mode has no backward");
  if (c.prec != MOE_BF16 && !p->weights_quantized)
    return fail(MOE_ERR_INVALID_ARG, "moe_backward: block-scaled plan needs moe_quantize_weights first");
  if (T < 0 || T > c.T_max) return fail(MOE_ERR_INVALID_ARG, "moe_backward: T outside [0, T_max]");
  if (!dWg || !dWu || !dWd || !Wg || !Wu || !Wd)
    return fail(MOE_ERR_INVALID_ARG, "moe_backward: null weight or weight-gradient pointer");
  if (T > 0 && (!dY || !X || !saved || !dX || !dg))
    return fail(MOE_ERR_INVALID_ARG, "moe_backward: null tensor pointer");
  if ((T > 0 && (!aligned16(dY) || !aligned16(X) || !aligned16(dX) ||
                 (reinterpret_cast<uintptr_t>(saved) & 255u))) ||
      !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd) || !aligned16(dWg) || !aligned16(dWu) ||
      !aligned16(dWd))
    return fail(MOE_ERR_INVALID_ARG, "moe_backward: misaligned pointer");
  DeviceGuard guard(c.device);
  if (!guard.ok) return fail(MOE_ERR_CUDA, "moe_backward: cudaSetDevice failed");
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err;
  if (T == 0) {  // no tokens: every expert's weight gradient is zero
    const size_t wbytes = (size_t)c.E * c.F * c.d * 2;
    if ((err = cudaMemsetAsync(dWg, 0, wbytes, st)) != cudaSuccess ||
        (err = cudaMemsetAsync(dWu, 0, wbytes, st)) != cudaSuccess ||
        (err = cudaMemsetAsync(dWd, 0, wbytes, st)) != cudaSuccess)
      return cuda_fail(err, "moe_backward: memset");
    return MOE_OK;
  }
  const SavedLayout L = saved_layout(c, T);
  const RoutingPtrs rp = routing_ptrs(L, const_cast<void*>(saved));
  const int Ti = (int)T;
  if (!ensure_weight_maps(p, Wg, Wu, Wd)) return fail(MOE_ERR_CUDA, "moe_backward: weight tensor maps");
  const uint64_t EF = (uint64_t)c.E * c.F, Ed = (uint64_t)c.E * c.d;
  if (dWg != p->p_dwg) {
    if (!map_store(&p->m_dWg_st, dWg, c.d, EF)) return fail(MOE_ERR_CUDA, "moe_backward: dWg map");
    p->p_dwg = dWg;
  }
  if (dWu != p->p_dwu) {
    if (!map_store(&p->m_dWu_st, dWu, c.d, EF)) return fail(MOE_ERR_CUDA, "moe_backward: dWu map");
    p->p_dwu = dWu;
  }
  if (dWd != p->p_dwd) {
    if (!map_store(&p->m_dWd_st, dWd, c.F, Ed)) return fail(MOE_ERR_CUDA, "moe_backward: dWd map");
    p->p_dwd = dWd;
  }
  const __nv_bfloat16* ab = reinterpret_cast<const __nv_bfloat16*>(static_cast<const char*>(saved) + L.ab);

  const bool ep = c.ep_ranks >= 2;
  // BF16 ring schedule: the backward's expert part as one persistent launch
  const bool ring_bwd = !ep && c.prec == MOE_BF16 && (c.debug_flags & MOE_DEBUG_RING_MEGAKERNEL) &&
                        !(c.debug_flags & MOE_DEBUG_SEPARATE_KERNELS);
  err = cudaSuccess;  // block-scaled plans gather no bf16 rows here (their dgrad and wgrad operands are quantised)
  if (ep) {  // pull reverse-combine: each expert rank pulls the dY and X rows of its pairs
    EpArgs ea = ep_args(p, rp, T);
    ea.X = reinterpret_cast<const uint4*>(X);
    ea.dY = reinterpret_cast<const uint4*>(dY);
    ea.Xg = static_cast<uint4*>(p->Xg);
    ea.dYg = static_cast<uint4*>(p->dYg);
    err = timed_launch(p, "ep_pull_reverse_combine", st, [&] { return launch_ep_pull(ea, st); });
  } else if (ring_bwd) {
    // B1-B4 and B6 in one persistent launch: movers pull the dY rows (and the
    // X rows unless the plan's last forward left them in place), u GEMM +
    // SwiGLU backward and dx GEMM tiles minibatch by minibatch, the dX sums
    // and the router gradient as their last inputs land
    const bool xg_current = p->xg_X == X && p->xg_saved == saved && p->xg_T == T;
    BwdMegaArgs m;
    memset(&m, 0, sizeof(m));
    m.mapU_A = p->m_dYg_k;
    m.mapU_B = p->m_Wd_mn;
    m.mapX_A = p->m_dAB_k;
    m.mapX_Bg = p->m_Wg_mn;
    m.mapX_Bu = p->m_Wu_mn;
    m.mapDabSt = p->m_dAB_st;
    m.mapWhSt = p->m_wH_st;
    m.mapYsSt = p->m_Ys_st;
    m.dY = reinterpret_cast<const uint4*>(dY);
    m.X = reinterpret_cast<const uint4*>(X);
    m.dYg = static_cast<uint4*>(p->dYg);
    m.Xg = xg_current ? nullptr : static_cast<uint4*>(p->Xg);
    m.ab = ab;
    m.rp = rp;
    m.dgp = p->dgp;
    m.dg = dg;
    m.dlogits = dlogits;
    m.Ys = static_cast<const uint4*>(p->Ys);
    m.dX = static_cast<uint4*>(dX);
    m.mtile_off = rp.mtile_off;
    m.mb_start = p->mb_start;
    m.phase_start = p->phase_start;
    m.n_mb = p->n_mb;
    m.counters = p->counters;
    m.counters_len = 1 + 2 * p->nm_max;
    m.tok_dx = p->tok_cnt;
    m.tok_u = p->tok_u;
    m.gbar = p->gbar;
    m.status = p->status;
    m.timeout_ns = (uint64_t)c.wait_timeout_ns;
    m.E = c.E;
    m.d = c.d;
    m.F = c.F;
    m.k = c.k;
    m.T = Ti;
    m.mbt = p->mbt;
    m.cap = p->cap;
    m.nm_max = p->nm_max;
    m.slots = 1;
    m.slot_rows = 0;
    err = timed_launch(p, "bwd_megakernel", st, [&] { return launch_bwd_megakernel(m, p->num_sms, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: backward megakernel launch");
    p->xg_X = X;   // the sorted X rows are in place now
    p->xg_saved = saved;
    p->xg_T = T;
  } else if (c.prec == MOE_BF16) {
    // X's sorted rows are still in Xg when this is the backward of the plan's
    // last forward, which ran the separate schedule: gather dY alone then
    const bool xg_current = p->xg_X == X && p->xg_saved == saved && p->xg_T == T;
    err = timed_launch(p, "gather_bwd", st, [&] {
      return launch_gather(dY, xg_current ? nullptr : X, rp.perm_src, rp.dest, rp.totals, Ti, c.k, c.d, p->dYg,
                           xg_current ? nullptr : p->Xg, p->num_sms * 8, st);
    });
  }
  if (err != cudaSuccess) return cuda_fail(err, "moe_backward: gather launch");
  const bool mx = c.prec != MOE_BF16;  // block-scaled dgrad GEMMs
  const bool nv = c.prec == MOE_NVFP4;
  if (mx && ep) {
    // the dY rows each expert rank pulled, quantised along d in place of the
    // per-token quantisation and copy (the same bytes)
    err = timed_launch(p, "quant_pulled_rows_dy", st, [&] { return launch_quant_sorted(p, p->dYg, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: EP dY quantisation launch");
  } else if (mx) {
    // MXFP8 / NVFP4 dgrad: dY quantised along d as it is gathered; u GEMM
    // against Wd^T (quantised along d) with dA|dB re-quantised along F in its
    // epilogue; dx GEMM against [Wg^T; Wu^T] (quantised along F).  The weight
    // gradients below are block-scaled too, on operands quantised along the
    // tokens.
    err = timed_launch(p, "quant_scatter_dy", st, [&] {
      return launch_quant_scatter_rows(nv, dY, rp.perm_src, rp.dest, rp.totals, (int)T, c.k, c.d, p->Xq, p->Xs,
                                       p->num_sms * 8, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: dY gather launch");
  }
  if (mx) {
    err = launch_block_scaled_dgrad_gemms(p, rp, ab, st);
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: block-scaled dgrad GEMM launch");
  }
  if (!mx && !ring_bwd) {
    GemmArgs a = base_args(p, rp);
    a.mapA = p->m_dYg_k;
    a.mapB0 = p->m_Wd_mn;
    a.mapO0 = p->m_dAB_st;
    a.mapO1 = p->m_wH_st;
    a.ab = ab;
    a.perm_src = rp.perm_src;
    a.wts = rp.w;
    a.dgp = p->dgp;
    err = timed_launch(p, "gemm_bwd_u_swiglu", st,
                       [&] { return launch_gemm_bwd(kBwdU, a, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: u GEMM launch");
  }
  if (!mx && !ring_bwd) {
    GemmArgs a = base_args(p, rp);
    a.mapA = p->m_dAB_k;
    a.mapB0 = p->m_Wg_mn;
    a.mapB1 = p->m_Wu_mn;
    a.mapO0 = p->m_Ys_st;
    err = timed_launch(p, "gemm_bwd_dx", st,
                       [&] { return launch_gemm_bwd(kBwdX, a, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: dx GEMM launch");
  }
  if (ep) {
    // push reverse-dispatch: each expert rank pushes the dx rows and <u, h>
    // partials of its pairs to their tokens' homes, which sum dX and form
    // the router gradient
    EpArgs ea = ep_args(p, rp, T);
    ea.Ys = static_cast<const uint4*>(p->Ys);
    ea.out = static_cast<uint4*>(dX);
    ea.dgp = p->dgp;
    ea.dg = dg;
    ea.dlogits = dlogits;
    err = timed_launch(p, "ep_push_reverse_dispatch", st, [&] { return launch_ep_push(ea, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: EP reverse-dispatch launch");
  } else if (!ring_bwd) {
    const int cgrid = (int)std::min<int64_t>(T, (int64_t)p->num_sms * 16);
    err = timed_launch(p, "reduce_dx", st,
                       [&] { return launch_combine(p->Ys, rp.dest, nullptr, Ti, c.k, c.d, dX, cgrid, st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: dx reduce launch");
    const int rgrid = (int)std::min<int64_t>((T + 7) / 8, (int64_t)p->num_sms * 8);
    err = timed_launch(p, "router_grad", st, [&] {
      // <u, h> partials: one per 256 columns (bf16 u GEMM) or per 128 (block-scaled u GEMM)
      return launch_router_grad(p->dgp, rp.dest, rp.idx, rp.w, Ti, c.k, c.E, mx ? c.F / 128 : c.F / BN, dg, dlogits,
                                rgrid, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: router gradient launch");
  }
  if (mx) {
    // block-scaled weight gradients: dY and X transposed and quantised along
    // the tokens here ([dA|dB]^T and (w h)^T came from the u GEMM's
    // epilogue; tensor scale 1 for NVFP4), rows past the ones in use skipped;
    // then dWd = dY^T (w h) and [dWg; dWu] = [dA|dB]^T X with K = each
    // expert's tokens
    const int Rq = (int)p->Rpm;
    err = timed_launch(p, "quant_wgrad_tokens", st, [&] {
      // one wave: two CTAs (three 32 KB stages each) per SM
      return launch_gather_transpose_q(nv, dY, X, rp.perm_src, rp.totals, c.k, Rq, c.d, p->dYTq, p->dYTs, p->XTq,
                                       p->XTs, p->status, (uint64_t)c.wait_timeout_ns,
                                       (c.debug_flags & MOE_DEBUG_STALL_TEST) ? 1 : 0, p->num_sms * 2, st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: weight-gradient token quantisation launch");
    MxArgs w;
    memset(&w, 0, sizeof(w));
    w.poff = rp.poff;
    w.mtile_off = rp.mtile_off;
    w.status = p->status;
    w.timeout_ns = (uint64_t)c.wait_timeout_ns;
    w.E = c.E;
    w.d = c.d;
    w.F = c.F;
    w.Kcap = Rq;
    MxArgs v = w;
    w.mapA = p->m_dYTq;
    w.mapB0 = p->m_wHTq;
    w.sfA = p->dYTs;
    w.sfB0 = p->wHTs;
    w.mapO0 = p->m_dWd_st;
    err = timed_launch(p, nv ? "gemm_nv_wgrad_down" : "gemm_mx_wgrad_down", st,
                       [&] { return launch_gemm_mx(kWgradD, w, p->num_sms, st, nv); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: block-scaled dWd GEMM launch");
    v.mapA = p->m_dABTq;
    v.mapB0 = p->m_XTq;
    v.sfA = p->dABTs;
    v.sfB0 = p->XTs;
    v.mapO0 = p->m_dWg_st;
    v.mapO1 = p->m_dWu_st;
    err = timed_launch(p, nv ? "gemm_nv_wgrad_gate_up" : "gemm_mx_wgrad_gate_up", st,
                       [&] { return launch_gemm_mx(kWgradGU, v, p->num_sms, st, nv); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: block-scaled dWg/dWu GEMM launch");
    return MOE_OK;
  }
  {
    GemmArgs a = base_args(p, rp);
    a.mapA = p->m_dYg_mn;
    a.mapB0 = p->m_wH_mn;
    a.mapO0 = p->m_dWd_st;
    err = timed_launch(p, "gemm_wgrad_down", st,
                       [&] { return launch_gemm_bwd(kWgradD, a, gemm_grid(p), st); });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: dWd GEMM launch");
  }
  {
    GemmArgs a = base_args(p, rp);
    a.mapA = p->m_dAB_mn;
    a.mapB0 = p->m_Xg_mn;
    a.mapO0 = p->m_dWg_st;
    a.mapO1 = p->m_dWu_st;
    err = timed_launch(p, "gemm_wgrad_gate_up", st, [&] {
      return launch_gemm_bwd(kWgradGU, a, gemm_grid(p), st);
    });
    if (err != cudaSuccess) return cuda_fail(err, "moe_backward: dWg/dWu GEMM launch");
  }
  return MOE_OK;
}

moe_status_t moe_get_routing(moe_plan_t p, int64_t T, const void* saved, int32_t* idx, float* w, int32_t* counts,
                             int32_t* offsets, int32_t* perm_src, int32_t* dest, moe_stream_t stream) {
  if (!p || !saved) return fail(MOE_ERR_INVALID_ARG, "moe_get_routing: null argument");
  const moe_config_t& c = p->cfg;
  if (T < 0 || T > c.T_max) return fail(MOE_ERR_INVALID_ARG, "moe_get_routing: T outside [0, T_max]");
  if (T == 0) return MOE_OK;
  DeviceGuard guard(c.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const SavedLayout L = saved_layout(c, T);
  const RoutingPtrs rp = routing_ptrs(L, const_cast<void*>(saved));
  const size_t R = (size_t)T * c.k;
  cudaError_t err = cudaSuccess;
  if (idx && err == cudaSuccess) err = cudaMemcpyAsync(idx, rp.idx, R * 4, cudaMemcpyDeviceToDevice, st);
  if (w && err == cudaSuccess) err = cudaMemcpyAsync(w, rp.w, R * 4, cudaMemcpyDeviceToDevice, st);
  if (counts && err == cudaSuccess) err = cudaMemcpyAsync(counts, rp.counts, c.E * 4, cudaMemcpyDeviceToDevice, st);
  if (offsets && err == cudaSuccess)
    err = cudaMemcpyAsync(offsets, rp.offsets, (c.E + 1) * 4, cudaMemcpyDeviceToDevice, st);
  if (err != cudaSuccess) return cuda_fail(err, "moe_get_routing: copy");
  if (perm_src || dest) {
    err = launch_unpad_routing(rp, (int)R, perm_src, dest, st);
    if (err != cudaSuccess) return cuda_fail(err, "moe_get_routing: unpad launch");
  }
  return MOE_OK;
}

namespace {
// Shape rules first; the pointers are checked only when T > 0 (a T = 0
// call may pass empty tensors), except those listed in `always`.
moe_status_t router_check(moe_plan_t p, int64_t T, const char* who, std::initializer_list<const void*> ptrs,
                          std::initializer_list<const void*> always = {}) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, std::string(who) + ": null plan");
  const moe_config_t& c = p->cfg;
  if (T < 0 || T > c.T_max) return fail(MOE_ERR_INVALID_ARG, std::string(who) + ": T outside [0, T_max]");
  if (c.E % 8 != 0) return fail(MOE_ERR_UNSUPPORTED, std::string(who) + ": the router GEMM needs E % 8 == 0");
  for (const void* q : always)
    if (!q || !aligned16(q)) return fail(MOE_ERR_INVALID_ARG, std::string(who) + ": null or misaligned pointer");
  if (T > 0)
    for (const void* q : ptrs)
      if (!q || !aligned16(q)) return fail(MOE_ERR_INVALID_ARG, std::string(who) + ": null or misaligned pointer");
  return MOE_OK;
}
GemmArgs router_args(moe_plan_s* p, int64_t T) {
  GemmArgs a;
  memset(&a, 0, sizeof(a));
  a.status = p->status;
  a.timeout_ns = (uint64_t)p->cfg.wait_timeout_ns;
  a.E = p->cfg.E;
  a.d = p->cfg.d;
  a.F = p->cfg.F;
  a.T = (int)T;
  return a;
}
int router_grid(const moe_plan_s* p, int64_t tiles) { return (int)std::min<int64_t>(tiles, p->num_sms); }
}  // namespace

moe_status_t moe_router_forward(moe_plan_t p, int64_t T, const void* X, const void* Wr, float* logits,
                                moe_stream_t stream) {
  if (moe_status_t s = router_check(p, T, "moe_router_forward", {X, Wr, logits})) return s;
  if (T == 0) return MOE_OK;
  const moe_config_t& c = p->cfg;
  DeviceGuard guard(c.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  GemmArgs a = router_args(p, T);
  if (!map_kmajor(&a.mapA, X, c.d, T) || !map_kmajor(&a.mapB0, Wr, c.d, c.E, BN))
    return fail(MOE_ERR_CUDA, "moe_router_forward: tensor maps");
  const int64_t tiles = ((T + BM - 1) / BM) * ((c.E + BN - 1) / BN);
  const int S = router_splits(p, tiles, (c.d + BK - 1) / BK);
  a.out_f32 = S > 1 ? p->router_part : logits;
  a.ksplit = S;
  cudaError_t err = timed_launch(p, "gemm_router", st,
                                 [&] { return launch_gemm_router(kRouter, a, router_grid(p, tiles * S), st); });
  if (err == cudaSuccess && S > 1)
    err = timed_launch(p, "router_split_sum", st, [&] {
      return launch_split_sum(p->router_part, S, T * c.E, logits, nullptr, p->num_sms * 4, st);
    });
  if (err != cudaSuccess) return cuda_fail(err, "moe_router_forward: launch");
  return MOE_OK;
}

moe_status_t moe_router_backward(moe_plan_t p, int64_t T, const void* X, const void* Wr, const float* dlogits,
                                 void* dX, void* dWr, moe_stream_t stream) {
  if (moe_status_t s = router_check(p, T, "moe_router_backward", {X, Wr, dlogits, dX}, {dWr})) return s;
  const moe_config_t& c = p->cfg;
  DeviceGuard guard(c.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  if (T == 0) {  // no tokens: dWr = 0, dX untouched
    cudaError_t err = cudaMemsetAsync(dWr, 0, (size_t)c.E * c.d * 2, st);
    return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_router_backward: zero dWr");
  }
  cudaError_t err = timed_launch(p, "router_dlogits_bf16", st, [&] {
    return launch_to_bf16(dlogits, p->dlg_bf16, T * c.E, p->num_sms * 4, st);
  });
  if (err != cudaSuccess) return cuda_fail(err, "moe_router_backward: dlogits conversion launch");
  GemmArgs x = router_args(p, T);
  GemmArgs w = router_args(p, T);
  if (!map_kmajor(&x.mapA, p->dlg_bf16, c.E, T) || !map_mnmajor(&x.mapB0, Wr, c.d, c.E) ||
      !map_mnmajor(&w.mapA, p->dlg_bf16, c.E, T) || !map_mnmajor(&w.mapB0, X, c.d, T) ||
      !map_store(&w.mapO0, dWr, c.d, c.E))
    return fail(MOE_ERR_CUDA, "moe_router_backward: tensor maps");
  x.io_bf16 = static_cast<__nv_bfloat16*>(dX);
  const int64_t tx = ((T + BM - 1) / BM) * (c.d / BN);
  err = timed_launch(p, "gemm_router_dx", st,
                     [&] { return launch_gemm_router(kRouterDX, x, router_grid(p, tx), st); });
  if (err != cudaSuccess) return cuda_fail(err, "moe_router_backward: dX launch");
  const int64_t tw = ((c.E + BM - 1) / BM) * (c.d / BN);
  const int Sw = router_splits(p, tw, (T + BK - 1) / BK);
  w.ksplit = Sw;
  w.part_f32 = p->router_part;
  err = timed_launch(p, "gemm_router_dw", st,
                     [&] { return launch_gemm_router(kRouterDW, w, router_grid(p, tw * Sw), st); });
  if (err == cudaSuccess && Sw > 1)
    err = timed_launch(p, "router_dw_split_sum", st, [&] {
      return launch_split_sum(p->router_part, Sw, (int64_t)c.E * c.d, nullptr, dWr, p->num_sms * 4, st);
    });
  if (err != cudaSuccess) return cuda_fail(err, "moe_router_backward: dWr launch");
  return MOE_OK;
}

moe_status_t moe_mx_quantize(const void* src, int64_t rows, int64_t K, void* q, void* sf, moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 128 != 0 || rows * K >= ((int64_t)1 << 40))
    return fail(MOE_ERR_INVALID_ARG, "moe_mx_quantize: need K a positive multiple of 128 and rows >= 0");
  if (rows == 0) return MOE_OK;
  if (!src || !q || !sf || !aligned16(src) || !aligned16(q) || !aligned16(sf))
    return fail(MOE_ERR_INVALID_ARG, "moe_mx_quantize: null or misaligned pointer");
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t err = launch_quant_rows(src, rows, (int)K, q, sf, std::max(1, sms) * 8,
                                      reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_mx_quantize: launch");
}

moe_status_t moe_mx_quantize_transposed(const void* src, int64_t E, int64_t A, int64_t B, void* q, void* sf,
                                        moe_stream_t stream) {
  if (E < 0 || A <= 0 || B <= 0 || A % 128 != 0 || B % 64 != 0 || E * A * B >= ((int64_t)1 << 40) ||
      A > (1 << 30) || B > (1 << 30))
    return fail(MOE_ERR_INVALID_ARG, "moe_mx_quantize_transposed: need A % 128 == 0, B % 64 == 0, E >= 0");
  if (E == 0) return MOE_OK;
  if (!src || !q || !sf || !aligned16(src) || !aligned16(q) || !aligned16(sf))
    return fail(MOE_ERR_INVALID_ARG, "moe_mx_quantize_transposed: null or misaligned pointer");
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  cudaError_t err = launch_quant_transpose(src, (int)E, (int)A, (int)B, q, sf, std::max(1, sms) * 8,
                                           reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_mx_quantize_transposed: launch");
}

static int current_sms() {
  int dev = 0, sms = 0;
  cudaGetDevice(&dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  return std::max(1, sms);
}

moe_status_t moe_nv_tensor_scale(const void* x0, int64_t n0, const void* x1, int64_t n1, float* g,
                                 moe_stream_t stream) {
  if (n0 < 0 || n1 < 0 || !g || (n0 > 0 && !x0) || (n1 > 0 && !x1) || (x0 && !aligned16(x0)) ||
      (x1 && !aligned16(x1)) || (reinterpret_cast<uintptr_t>(g) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "moe_nv_tensor_scale: null or misaligned pointer, or negative size");
  cudaError_t err = launch_nv_tensor_scale(n0 > 0 ? x0 : nullptr, n0, n1 > 0 ? x1 : nullptr, n1, g,
                                           current_sms() * 8, reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_nv_tensor_scale: launch");
}

moe_status_t moe_nv_quantize(const void* src, int64_t rows, int64_t K, const float* g, void* q, void* sf,
                             moe_stream_t stream) {
  if (rows < 0 || K <= 0 || K % 64 != 0 || K > (1 << 30) || rows * K >= ((int64_t)1 << 40))
    return fail(MOE_ERR_INVALID_ARG, "moe_nv_quantize: need K a positive multiple of 64 and rows >= 0");
  if (rows == 0) return MOE_OK;
  if (!src || !q || !sf || !aligned16(src) || !aligned16(q) || !aligned16(sf) ||
      (reinterpret_cast<uintptr_t>(g) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "moe_nv_quantize: null or misaligned pointer");
  cudaError_t err = launch_nv_quant_rows(src, rows, (int)K, g, q, sf, current_sms() * 8,
                                         reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_nv_quantize: launch");
}

moe_status_t moe_nv_quantize_transposed(const void* src, int64_t E, int64_t A, int64_t B, const float* g,
                                        void* q, void* sf, moe_stream_t stream) {
  if (E < 0 || A <= 0 || B <= 0 || A % 128 != 0 || B % 64 != 0 || E * A * B >= ((int64_t)1 << 40) ||
      A > (1 << 30) || B > (1 << 30))
    return fail(MOE_ERR_INVALID_ARG, "moe_nv_quantize_transposed: need A % 128 == 0, B % 64 == 0, E >= 0");
  if (E == 0) return MOE_OK;
  if (!src || !q || !sf || !aligned16(src) || !aligned16(q) || !aligned16(sf) ||
      (reinterpret_cast<uintptr_t>(g) & 3u))
    return fail(MOE_ERR_INVALID_ARG, "moe_nv_quantize_transposed: null or misaligned pointer");
  cudaError_t err = launch_nv_quant_transpose(src, (int)E, (int)A, (int)B, g, q, sf, current_sms() * 8,
                                              reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_nv_quantize_transposed: launch");
}

moe_status_t moe_quantize_weights(moe_plan_t p, const void* Wg, const void* Wu, const void* Wd, moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "moe_quantize_weights: null plan");
  const moe_config_t& c = p->cfg;
  if (c.prec != MOE_MXFP8 && c.prec != MOE_NVFP4)
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_weights: plan is not MOE_MXFP8 or MOE_NVFP4");
  if (!Wg || !Wu || !Wd || !aligned16(Wg) || !aligned16(Wu) || !aligned16(Wd))
    return fail(MOE_ERR_INVALID_ARG, "moe_quantize_weights: null or misaligned weight pointer");
  DeviceGuard guard(c.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const int64_t EF = (int64_t)c.E * c.F, Ed = (int64_t)c.E * c.d;
  const int grid = p->num_sms * 8;
  cudaError_t err;
  if (c.prec == MOE_NVFP4) {
    // tensor scales first: [0] over Wg and Wu together (the dx GEMM contracts
    // over both), [1] over Wd; every copy of a weight uses its tensor's scale
    const float* g_gu = p->nv_scale;
    const float* g_d = p->nv_scale + 1;
    err = timed_launch(p, "quant_weights", st, [&] {
      cudaError_t e = launch_nv_tensor_scale(Wg, EF * c.d, Wu, EF * c.d, p->nv_scale, grid, st);
      if (e == cudaSuccess) e = launch_nv_tensor_scale(Wd, Ed * c.F, nullptr, 0, p->nv_scale + 1, grid, st);
      if (e == cudaSuccess) e = launch_nv_quant_rows(Wg, EF, c.d, g_gu, p->Wgq, p->Wgs, grid, st);
      if (e == cudaSuccess) e = launch_nv_quant_rows(Wu, EF, c.d, g_gu, p->Wuq, p->Wus, grid, st);
      if (e == cudaSuccess) e = launch_nv_quant_rows(Wd, Ed, c.F, g_d, p->Wdq, p->Wds, grid, st);
      if (e == cudaSuccess) e = launch_nv_quant_transpose(Wd, c.E, c.d, c.F, g_d, p->WdTq, p->WdTs, grid, st);
      if (e == cudaSuccess) e = launch_nv_quant_transpose(Wg, c.E, c.F, c.d, g_gu, p->WgTq, p->WgTs, grid, st);
      if (e == cudaSuccess) e = launch_nv_quant_transpose(Wu, c.E, c.F, c.d, g_gu, p->WuTq, p->WuTs, grid, st);
      return e;
    });
  } else {
    err = timed_launch(p, "quant_weights", st, [&] {
      cudaError_t e = launch_quant_rows(Wg, EF, c.d, p->Wgq, p->Wgs, grid, st);
      if (e == cudaSuccess) e = launch_quant_rows(Wu, EF, c.d, p->Wuq, p->Wus, grid, st);
      if (e == cudaSuccess) e = launch_quant_rows(Wd, Ed, c.F, p->Wdq, p->Wds, grid, st);
      // backward orientation: Wd[e]^T [F, d] along d; Wg[e]^T, Wu[e]^T [d, F] along F
      if (e == cudaSuccess) e = launch_quant_transpose(Wd, c.E, c.d, c.F, p->WdTq, p->WdTs, grid, st);
      if (e == cudaSuccess) e = launch_quant_transpose(Wg, c.E, c.F, c.d, p->WgTq, p->WgTs, grid, st);
      if (e == cudaSuccess) e = launch_quant_transpose(Wu, c.E, c.F, c.d, p->WuTq, p->WuTs, grid, st);
      return e;
    });
  }
  if (err != cudaSuccess) return cuda_fail(err, "moe_quantize_weights: launch");
  p->weights_quantized = true;
  return MOE_OK;
}

moe_status_t moe_plan_padded_rows(moe_plan_t p, int64_t* rows) {
  if (!p || !rows) return fail(MOE_ERR_INVALID_ARG, "moe_plan_padded_rows: null argument");
  *rows = p->Rpm;
  return MOE_OK;
}

moe_status_t moe_debug_quant_dump(moe_plan_t p, int32_t which, float* vals, void* q, void* sf, moe_stream_t stream) {
  if (!p) return fail(MOE_ERR_INVALID_ARG, "moe_debug_quant_dump: null plan");
  const moe_config_t& c = p->cfg;
  if (c.prec == MOE_BF16 || !(c.debug_flags & MOE_DEBUG_DUMP_QUANT) || !p->dbg_h)
    return fail(MOE_ERR_INVALID_ARG, "moe_debug_quant_dump: needs a block-scaled plan made with MOE_DEBUG_DUMP_QUANT");
  if (which < 0 || which > 6)
    return fail(MOE_ERR_INVALID_ARG, "moe_debug_quant_dump: which must be 0 (h), 1 (dA|dB), 2 (dY^T), 3 (X^T), "
                                     "4 ([dA|dB]^T), 5 ((w h)^T) or 6 (dispatched rows)");
  if (vals && (which == 2 || which == 3 || which == 6))
    return fail(MOE_ERR_INVALID_ARG,
                "moe_debug_quant_dump: dY^T, X^T and the dispatched rows keep no source values (vals must be NULL)");
  DeviceGuard guard(c.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  const bool nv = c.prec == MOE_NVFP4;
  const size_t P = (size_t)p->Rpm;
  // which 0, 1, 6: [P, C] quantised along C; 2..5: [C, P] quantised along the P sorted rows
  const size_t C = (size_t)(which == 0 || which == 5 ? c.F : which == 1 || which == 4 ? 2 * c.F : c.d);
  const size_t n = P * C;
  const void* qsrc[7] = {p->Hq, p->dABq, p->dYTq, p->XTq, p->dABTq, p->wHTq, p->Xq};
  const void* ssrc[7] = {p->Hs, p->dABs, p->dYTs, p->XTs, p->dABTs, p->wHTs, p->Xs};
  cudaError_t err = cudaSuccess;
  if (vals) {
    if (which <= 1)
      err = cudaMemcpyAsync(vals, which == 0 ? p->dbg_h : p->dbg_dab, n * 4, cudaMemcpyDeviceToDevice, st);
    else   // the bf16 values the u GEMM's epilogue quantised (stored in this mode), widened
      err = launch_widen_bf16(which == 4 ? p->dAB : p->wH, vals, (int64_t)n, p->num_sms * 4, st);
  }
  if (q && err == cudaSuccess) err = cudaMemcpyAsync(q, qsrc[which], nv ? n / 2 : n, cudaMemcpyDeviceToDevice, st);
  if (sf && err == cudaSuccess)
    err = cudaMemcpyAsync(sf, ssrc[which], nv ? n / 16 : n / 32, cudaMemcpyDeviceToDevice, st);
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_debug_quant_dump: copy");
}

moe_status_t moe_nv_weight_scales(moe_plan_t p, float* out, moe_stream_t stream) {
  if (!p || !out) return fail(MOE_ERR_INVALID_ARG, "moe_nv_weight_scales: null argument");
  if (p->cfg.prec != MOE_NVFP4) return fail(MOE_ERR_INVALID_ARG, "moe_nv_weight_scales: plan is not MOE_NVFP4");
  DeviceGuard guard(p->cfg.device);
  cudaError_t err = cudaMemcpyAsync(out, p->nv_scale, 2 * sizeof(float), cudaMemcpyDeviceToDevice,
                                    reinterpret_cast<cudaStream_t>(stream));
  return err == cudaSuccess ? MOE_OK : cuda_fail(err, "moe_nv_weight_scales: copy");
}

moe_status_t moe_device_status(moe_plan_t p, moe_stream_t stream, int32_t* status) {
  if (!p || !status) return fail(MOE_ERR_INVALID_ARG, "moe_device_status: null argument");
  DeviceGuard guard(p->cfg.device);
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaError_t err = cudaStreamSynchronize(st);
  if (err != cudaSuccess) return cuda_fail(err, "moe_device_status: stream synchronize");
  int32_t v = 0;
  err = cudaMemcpy(&v, p->status, 4, cudaMemcpyDeviceToHost);
  if (err != cudaSuccess) return cuda_fail(err, "moe_device_status: read");
  if (v != 0) cudaMemset(p->status, 0, 4);
  *status = v;
  return MOE_OK;
}

moe_status_t moe_kernel_times(moe_plan_t p, const char** names, double* total_ms, int64_t* launches, int32_t cap,
                              int32_t* n) {
  if (!p || !n) return fail(MOE_ERR_INVALID_ARG, "moe_kernel_times: null argument");
  DeviceGuard guard(p->cfg.device);
  cudaError_t err = cudaDeviceSynchronize();
  if (err != cudaSuccess) return cuda_fail(err, "moe_kernel_times: synchronize");
  std::vector<const char*> nm;
  std::vector<double> ms;
  std::vector<int64_t> cnt;
  for (auto& t : p->timed) {
    float x = 0.f;
    cudaEventElapsedTime(&x, t.a, t.b);
    size_t i = 0;
    while (i < nm.size() && strcmp(nm[i], t.name) != 0) ++i;
    if (i == nm.size()) {
      nm.push_back(t.name);
      ms.push_back(0.0);
      cnt.push_back(0);
    }
    ms[i] += x;
    cnt[i] += 1;
    p->spare_events.push_back(t.a);
    p->spare_events.push_back(t.b);
  }
  p->timed.clear();
  *n = (int32_t)nm.size();
  for (int32_t i = 0; i < *n && i < cap; ++i) {
    if (names) names[i] = nm[i];
    if (total_ms) total_ms[i] = ms[i];
    if (launches) launches[i] = cnt[i];
  }
  return MOE_OK;
}

}  // extern "C"
