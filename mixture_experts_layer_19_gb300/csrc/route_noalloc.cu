// route_noalloc.cu -- routing (top-k experts, gate weights, per-expert
// counts and offsets, stable token permutation) for callers that cannot
// allocate device memory.
//
// Some callers cannot call cudaMalloc: code embedded in a host framework
// whose own allocator has reserved the device memory (a direct allocation
// would fail or escape its accounting), or latency-critical paths that cannot
// pay for an allocation, which may synchronise the device.  moe_plan
// allocates its workspace, so such callers cannot use moe_forward's routing.
// This entry point runs the same routing kernels with their scratch (chunk
// histograms, chunk bases, padded segment table, padded permutation) placed in
// one file-scope device array instead.
//
// The array is kNoAllocScratchInts int32 (4 MiB) and every GPU that loads this
// library keeps it until the process exits.  With CUDA's lazy module loading
// (the default) the array is committed when the module first loads on a
// device, which can be this entry point's first call there; a caller whose
// allocator reserves the device afterwards should make one warm-up call
// first.  All calls share it and it keeps
// the last call's contents; no entry is read before the same call writes it,
// so nothing needs clearing between calls.  Calls that overlap on the GPU
// (e.g. on two streams) race on it and must be serialised by the caller.
#include <cuda_runtime.h>

#include <mutex>
#include <string>

#include "kernels.h"
#include "moe.h"

namespace moe {

constexpr size_t kNoAllocScratchInts = size_t(1) << 20;  // 4 MiB of int32
static __device__ __align__(256) int32_t g_route_scratch[kNoAllocScratchInts];

namespace {

constexpr int kMaxDevices = 64;
int32_t* g_scratch_addr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_route_scratch on `dev` (the current device).  In host
// code the symbol is only a host-side stand-in, so the address is looked up
// with the device current.  It is looked up again on every call made outside
// a stream capture (a device reset reloads the module, which may move the
// array); during a capture the address cached by an earlier call is used, so
// the first call on a device must come before any capture.
cudaError_t scratch_for_device(int dev, bool capturing, int32_t** out) {
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_addr[dev] || !capturing) {
    void* p = nullptr;
    cudaError_t e = cudaGetSymbolAddress(&p, g_route_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_addr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_addr[dev];
  return cudaSuccess;
}

size_t round256(size_t ints) { return (ints + 63) & ~size_t(63); }  // keep 256-byte alignment

}  // namespace
}  // namespace moe

extern "C" moe_status_t moe_route_noalloc(int64_t T, int32_t E, int32_t k, const float* logits, int32_t* idx,
                                          float* w, int32_t* counts, int32_t* offsets, int32_t* perm_src,
                                          int32_t* dest, moe_stream_t stream) {
  using namespace moe;
  if (T < 0 || T > (1 << 20) || k < 1 || k > 32 || E < k || E > 1024) {
    set_error_detail("moe_route_noalloc: need 0 <= T <= 2^20, 1 <= k <= 32, k <= E <= 1024");
    return MOE_ERR_INVALID_ARG;
  }
  if (T == 0) return MOE_OK;
  if (!logits || !idx || !w || !counts || !offsets || !perm_src || !dest) {
    set_error_detail("moe_route_noalloc: null pointer");
    return MOE_ERR_INVALID_ARG;
  }
  const int Ti = (int)T;
  const int nch = route_chunks(Ti);
  const size_t R = (size_t)T * k;
  const size_t rows_pad = R + (size_t)E * (kTileRows - 1);
  // scratch: chunk_hist, chunk_base, poff, mtile_off, totals, padded dest, padded perm
  const size_t need = 2 * round256((size_t)nch * E) + 2 * round256(E + 1) + round256(4) + round256(R) +
                      round256(rows_pad);
  if (need > kNoAllocScratchInts) {
    set_error_detail(("moe_route_noalloc: needs " + std::to_string(need * 4) + " bytes of scratch, the fixed " +
                      "device array holds " + std::to_string(kNoAllocScratchInts * 4) +
                      " (reduce T, or use moe_plan/moe_forward)").c_str());
    return MOE_ERR_UNSUPPORTED;
  }
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
    set_error_detail("moe_route_noalloc: no usable current device");
    return MOE_ERR_CUDA;
  }
  cudaStream_t st = reinterpret_cast<cudaStream_t>(stream);
  cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
  if ((err = cudaStreamIsCapturing(st, &cap)) != cudaSuccess) {
    set_error_detail((std::string("moe_route_noalloc: cudaStreamIsCapturing: ") + cudaGetErrorString(err)).c_str());
    return MOE_ERR_CUDA;
  }
  const bool capturing = cap != cudaStreamCaptureStatusNone;
  if (capturing && !g_scratch_addr[dev]) {
    set_error_detail("moe_route_noalloc: the first call on a device must come before any stream capture");
    return MOE_ERR_INVALID_ARG;
  }
  int32_t* base = nullptr;
  if ((err = scratch_for_device(dev, capturing, &base)) != cudaSuccess) {
    set_error_detail((std::string("moe_route_noalloc: cudaGetSymbolAddress: ") + cudaGetErrorString(err)).c_str());
    return MOE_ERR_CUDA;
  }
  int32_t* p = base;
  int32_t* chunk_hist = p;  p += round256((size_t)nch * E);
  int32_t* chunk_base = p;  p += round256((size_t)nch * E);
  RoutingPtrs rp;
  rp.idx = idx;
  rp.w = w;
  rp.counts = counts;
  rp.offsets = offsets;
  rp.poff = p;       p += round256(E + 1);
  rp.mtile_off = p;  p += round256(E + 1);
  rp.totals = p;     p += round256(4);
  rp.dest = p;       p += round256(R);
  rp.perm_src = p;
  // a launch error read below belongs to these launches, not to earlier work
  // on this thread that left an error pending
  (void)cudaGetLastError();
  if ((err = launch_router(logits, Ti, E, k, chunk_hist, rp, st)) != cudaSuccess ||
      (err = launch_scan(Ti, E, chunk_hist, chunk_base, rp, st)) != cudaSuccess ||
      (err = launch_permute(Ti, E, k, chunk_base, rp, st)) != cudaSuccess ||
      (err = launch_unpad_routing(rp, (int)R, perm_src, dest, st)) != cudaSuccess) {
    set_error_detail((std::string("moe_route_noalloc: launch: ") + cudaGetErrorString(err)).c_str());
    return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

