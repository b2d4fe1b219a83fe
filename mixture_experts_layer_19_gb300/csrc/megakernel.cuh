// megakernel.cuh -- argument block of the ring-buffer forward megakernel
// (megakernel.cu), shared with the host code that fills it (api.cu).
#pragma once
#include <cuda.h>
#include <stdint.h>

namespace moe {

struct MegaArgs {
  CUtensorMap mapXr;    // ring X rows, K-major loads {d, ring rows}, box 64 x 128
  CUtensorMap mapWg;    // Wg K-major {d, E*F}, box 64 x 128
  CUtensorMap mapWu;
  CUtensorMap mapWd;    // Wd K-major {F, E*d}, box 64 x 256
  CUtensorMap mapHr;    // ring h rows, K-major loads {F, ring rows}, box 64 x 128
  CUtensorMap mapHrSt;  // ring h rows, stores, box 32 x 32
  CUtensorMap mapABSt;  // saved a|b {2F, rows}, stores
  CUtensorMap mapYsSt;  // sorted y rows {d, rows}, stores
  const uint4* X;       // [T, d] bf16 tokens
  uint4* ring_x;        // [slots * slot_rows, d] bf16
  const int32_t* perm_src;
  const int32_t* mtile_off;   // [E+1]
  const int32_t* mb_start;    // [n_mb+1] first 128-row tile of each minibatch
  const int32_t* phase_start; // [2 n_mb + 1] first claim index of each phase
  const int32_t* n_mb;
  int* claim;
  int* gathered;
  int* g1_done;
  int* mb_done;
  int32_t* status;
  uint64_t timeout_ns;
  int E, d, F, k, movers, slots, slot_rows;
};

}  // namespace moe
