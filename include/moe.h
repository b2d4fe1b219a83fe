/*
 * moe.h -- C ABI of the fused Mixture-of-Experts layer (router top-k,
 * stable token permutation, gather, grouped SwiGLU expert GEMMs, weighted
 * combine; forward and backward) on one GB300 (sm_103a).
 *
 * The operation is the MoE layer benchmarked by the Mixture-of-Kittens pages:
 * "scheduler, routing, expert FFNs, combine and final weighted fusion"
 * (kucoin page "Cursor's MoK réalise une amélioration des performances de
 * 2,37x sur NVIDIA GB300 NVL72", section 03), with its backward pass
 * ("two more communication steps in the reverse direction", same page,
 * section 01).  The pages give no formulas; this library computes, per token
 * t with router logits l_t:
 *
 *   idx_t = top-k experts of l_t (logit descending, ties to the lower id)
 *   w_tj  = exp(l_t[idx_tj] - max) / sum_i exp(l_t[idx_ti] - max)
 *   a = x_t Wg[e]^T, b = x_t Wu[e]^T, h = silu(a) * b, y_tj = h Wd[e]^T
 *   Y_t   = sum_j w_tj y_tj            (j ascending, fp32, one bf16 rounding)
 *
 * and the gradients of L = <dY, Y>.  The plain fp64 statement of the same
 * arithmetic is the CPU oracle the test suite checks against.
 *
 * Conventions for every entry point below:
 *  - All tensor arguments are DEVICE pointers to row-major, contiguous,
 *    16-byte aligned buffers owned by the caller (e.g. torch tensors).
 *    bf16 buffers are passed as void*.
 *  - Weights use the nn.Linear [out, in] convention:
 *      Wg, Wu: [E, F, d] bf16;  Wd: [E, d, F] bf16.
 *  - The plan owns all device workspace; it is allocated once in moe_plan.
 *    moe_forward / moe_backward never allocate and never synchronise with
 *    the host: they enqueue kernels on `stream` and return.
 *  - Argument / shape errors return synchronously and enqueue nothing.
 *    Errors detected on the device (a bounded wait that ran out) are written
 *    to the plan's device status word and reported by moe_device_status.
 *  - No C++ exception crosses this ABI.  One stream per plan at a time.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* moe_stream_t; /* identical to cudaStream_t */

typedef enum {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = 1,  /* null / misaligned pointer, T > T_max, bad config value */
  MOE_ERR_UNSUPPORTED = 2,  /* shape outside the supported set (see moe_plan) */
  MOE_ERR_OOM = 3,          /* workspace allocation failed in moe_plan */
  MOE_ERR_CUDA = 4,         /* a CUDA runtime / driver call failed */
  MOE_ERR_TIMEOUT = 5,      /* a device-side bounded wait expired */
  MOE_ERR_INTERNAL = 6
} moe_status_t;

/* MOE_NVFP4: E2M1 elements with one E4M3 scale per 16 elements along each
 * GEMM's K and an fp32 scale per weight tensor (Wg and Wu share one);
 * activations quantised with tensor scale 1 (the rules are those of
 * moe_nv_quantize). */
typedef enum { MOE_BF16 = 0, MOE_MXFP8 = 1, MOE_NVFP4 = 2 } moe_precision_t;

/* debug_flags bits */
#define MOE_DEBUG_IDENTITY_EXPERTS 0x1u /* experts return their input (y = x); GEMMs skipped */
#define MOE_DEBUG_TIMING 0x2u           /* bracket each kernel with CUDA events (moe_kernel_times) */
/* Forward schedule.  By default both precisions run separate kernels
 * (routing, gather, grouped GEMMs over the full sorted buffers, combine).
 * MOE_DEBUG_RING_MEGAKERNEL selects the ring-buffer megakernel (movers fill a
 * fixed ring of minibatch slots, compute CTAs run the [a|b] and down tiles
 * minibatch by minibatch); for BF16 it is one launch that also routes and
 * combines, or, with MOE_DEBUG_MULTI_LAUNCH, the megakernel between separate
 * routing and combine launches.  Every schedule gives bitwise identical
 * results. */
#define MOE_DEBUG_SEPARATE_KERNELS 0x4u /* force separate kernels (overrides the ring flag) */
#define MOE_DEBUG_RING_MEGAKERNEL 0x8u  /* use the ring-buffer megakernel */
/* BF16 ring schedule: routing, layout, the minibatch plan and the combine as
 * separate launches around the ring megakernel instead of inside it. */
#define MOE_DEBUG_MULTI_LAUNCH 0x20u
/* Block-scaled plans (MXFP8, NVFP4): the plan keeps the fp32 values its fused
 * epilogues quantise -- h in the forward's up GEMM, dA|dB in the backward's
 * u GEMM -- for moe_debug_quant_dump.  The forward then runs the separate
 * kernels (the ring megakernel keeps no copy). */
#define MOE_DEBUG_DUMP_QUANT 0x40u
/* Fault-injection test hook (tests only): in the separate-kernel BF16
 * forward, the up GEMM's producer issues no loads, and in a block-scaled
 * backward the weight gradients' token pass copies no rows, so the waiting
 * warps' bounded waits expire after wait_timeout_ns.  The kernel then exits
 * cleanly (TMEM freed, nothing in flight), the status word reads
 * MOE_ERR_TIMEOUT at the next moe_device_status, and the CUDA context stays
 * usable.  Y (forward) or the weight gradients (backward) are not valid. */
#define MOE_DEBUG_STALL_TEST 0x80u

typedef struct {
  int64_t T_max;          /* largest token count a call may pass */
  int32_t d;              /* hidden size; multiple of 256 */
  int32_t F;              /* expert FFN width; multiple of 256 */
  int32_t E;              /* experts, k <= E <= 1024 */
  int32_t k;              /* experts per token, 1 <= k <= 32 */
  int32_t prec;           /* moe_precision_t (MOE_MXFP8 / MOE_NVFP4 need moe_quantize_weights) */
  int32_t minibatch_rows; /* rows per ring slot; 0 = two-wave floor (moe_minibatch_floor) */
  int32_t ring_slots;     /* ring buffer slots; 0 = default */
  int32_t mover_ctas;     /* CTAs given over to gathering rows into the ring (data movers);
                             0 = default: the BF16 ring gathers with two extra warps of every
                             compute CTA, the MXFP8 ring with 8 mover CTAs */
  int64_t wait_timeout_ns;/* bound on every device-side wait; 0 = 2e9 (2 s) */
  uint32_t debug_flags;   /* MOE_DEBUG_* */
  int32_t device;         /* CUDA device ordinal the plan binds to */
  int32_t ep_ranks;       /* >= 2: the layer as expert parallelism over this many virtual
                             ranks on the one GPU (pull dispatch, push combine, pull reverse-
                             combine, push reverse-dispatch; block-scaled plans quantise the
                             pulled bf16 rows); must divide E; 0 or 1 = off */
} moe_config_t;

typedef struct moe_plan_s* moe_plan_t;

/* Create a plan: validates `cfg`, binds `cfg->device`, allocates all device
 * workspace for T <= T_max, and returns it in *out (caller frees with
 * moe_plan_destroy).  Supported: d % 256 == 0, F % 256 == 0, 1 <= k <= 32,
 * k <= E <= 1024, 1 <= T_max <= 2^20, prec MOE_BF16, MOE_MXFP8 or MOE_NVFP4
 * (a block-scaled plan also holds quantised copies of the weights in both
 * orientations for its block-scaled forward and dgrad GEMMs; its weight
 * gradients are block-scaled GEMMs on operands quantised along the tokens;
 * NVFP4 plans run the separate-kernel schedule).  Otherwise
 * MOE_ERR_UNSUPPORTED / MOE_ERR_INVALID_ARG; allocation failure MOE_ERR_OOM. */
moe_status_t moe_plan(const moe_config_t* cfg, moe_plan_t* out);

/* Free the plan's workspace (synchronises its device first). NULL is a no-op.
 * Not while any stream of the device is being captured into a CUDA graph: the
 * device synchronisation and the frees would invalidate that capture (the
 * Python binding defers a plan closed or collected during a capture to its
 * next plan creation or close outside one). */
moe_status_t moe_plan_destroy(moe_plan_t plan);

/* Bytes of the caller-owned "saved" context a forward of T tokens writes and
 * the matching backward reads (routing, permutation, tile table and the
 * gate/up pre-activations A|B).  The caller allocates it (256-byte aligned). */
moe_status_t moe_saved_bytes(moe_plan_t plan, int64_t T, size_t* bytes);

/* Forward of T tokens (0 <= T <= T_max; T == 0 is a no-op).
 *   X      [T, d] bf16      tokens
 *   logits [T, E] fp32      router logits (finite)
 *   Wg, Wu [E, F, d] bf16, Wd [E, d, F] bf16
 *   Y      [T, d] bf16      output (written)
 *   saved  moe_saved_bytes(T) bytes, written; pass it unchanged to moe_backward.
 * Enqueued on `stream`; bitwise deterministic for identical inputs.
 * Errors, synchronous with nothing enqueued: MOE_ERR_INVALID_ARG for a null
 * plan or tensor pointer (the weights may be NULL only with
 * MOE_DEBUG_IDENTITY_EXPERTS), a tensor not 16-byte aligned, `saved` not
 * 256-byte aligned, T outside [0, T_max], or a block-scaled plan whose
 * weights were never quantised; MOE_ERR_CUDA when a launch fails.  The
 * sizes of X, Y and `saved` cannot be checked through these pointers: a
 * buffer smaller than stated is overrun. */
moe_status_t moe_forward(moe_plan_t plan, int64_t T, const void* X, const float* logits,
                         const void* Wg, const void* Wu, const void* Wd, void* Y,
                         void* saved, moe_stream_t stream);

/* Backward of the forward that wrote `saved` (same T, X and weights).
 *   dY [T, d] bf16 upstream gradient
 *   dX [T, d] bf16; dWg, dWu [E, F, d] bf16; dWd [E, d, F] bf16 (overwritten,
 *      experts that received no token get zeros)
 *   dg      [T, k] fp32  gradient of the gate weights w (written)
 *   dlogits [T, E] fp32  gradient of the router logits, or NULL to skip
 * Enqueued on `stream`; every reduction runs in a fixed order: bitwise
 * deterministic.  Errors as for moe_forward (dlogits may be NULL). */
moe_status_t moe_backward(moe_plan_t plan, int64_t T, const void* dY, const void* X,
                          const void* Wg, const void* Wu, const void* Wd, const void* saved,
                          void* dX, void* dWg, void* dWu, void* dWd, float* dg, float* dlogits,
                          moe_stream_t stream);

/* MXFP8 and NVFP4 plans: quantise the bf16 expert weights into the plan's
 * E4M3 (MXFP8) or E2M1 (NVFP4: after computing the tensor scales, Wg and Wu
 * sharing one) copies (once per optimiser step, outside the layer's timing).  Forward
 * orientation: Wg, Wu along d, Wd along F; backward orientation (transposed
 * copies for the dgrad GEMMs): Wd[e]^T along d, Wg[e]^T and Wu[e]^T along F;
 * blocks of 32 with one E8M0 scale (the layout of moe_mx_quantize).  Must
 * precede moe_forward / moe_backward on an MXFP8 plan (their weight-streaming
 * GEMMs then read the plan's copies).  Enqueued on `stream`.  MXFP8 activation
 * quantisation
 * is fused into the dispatch / GEMM / SwiGLU datapaths (kucoin page "Cursor's
 * MoK réalise une amélioration des performances de 2,37x sur NVIDIA GB300
 * NVL72", section 02); the format itself is OCP Microscaling v1.0 MXFP8. */
moe_status_t moe_quantize_weights(moe_plan_t plan, const void* Wg, const void* Wu, const void* Wd,
                                  moe_stream_t stream);

/* Quantise a bf16 row-major [rows, K] device matrix to MXFP8 along K
 * (K % 128 == 0): q [rows, K] E4M3 bytes; sf the E8M0 scale bytes
 * (X + 127 with X = floor(log2 amax) - 8 clamped to [-127, 127], all-zero
 * block -> 0) arranged in 512-byte atoms: rows [128 i, 128 i + 128) and
 * blocks [4 j, 4 j + 4) form atom i * (K / 128) + j, and row r / block b sits
 * at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + b % 4 of its atom.  sf must hold
 * ceil(rows / 128) * (K / 128) * 512 bytes.  Elements round to nearest even
 * and saturate at +-448.  The same kernel quantises the weights. */
moe_status_t moe_mx_quantize(const void* src, int64_t rows, int64_t K, void* q, void* sf, moe_stream_t stream);

/* Quantise the transposes of E bf16 row-major [A, B] device matrices
 * (src [E, A, B]) to MXFP8 along A: q [E, B, A] E4M3 bytes, so row e*B + b
 * holds src[e, :, b]; sf the scale atoms of those E*B rows with K = A
 * (the layout of moe_mx_quantize).  A % 128 == 0 and B % 64 == 0
 * (MOE_ERR_INVALID_ARG otherwise).  The same kernel makes the transposed
 * weight copies of moe_quantize_weights.  Enqueued on `stream`. */
moe_status_t moe_mx_quantize_transposed(const void* src, int64_t E, int64_t A, int64_t B, void* q, void* sf,
                                        moe_stream_t stream);

/* NVFP4 tensor scale of one or two bf16 device tensors (x1 may be NULL with
 * n1 = 0): *g = fl32(amax / 2688) over all n0 + n1 elements (2688 = largest
 * E2M1 times largest E4M3), or 1 when every element is zero.  g is a device
 * float, written on `stream`.  Both tensors 16-byte aligned, finite values
 * (MOE_ERR_INVALID_ARG otherwise).  NVIDIA's NVFP4: a second-level fp32
 * scale per tensor; the pages name NVFP4 kernels only (fluidifia page
 * "Cursor ouvre MoK, un mégakernel qui accélère l'entraînement MoE", section
 * "Quand la communication devient le vrai problème"). */
moe_status_t moe_nv_tensor_scale(const void* x0, int64_t n0, const void* x1, int64_t n1, float* g,
                                 moe_stream_t stream);

/* Quantise a bf16 row-major [rows, K] device matrix to NVFP4 along K
 * (K % 64 == 0) with the tensor scale *g (device float; NULL = 1):
 *   rc = fl32(1 / fl32(6 g));  per 16-element block s = E4M3(fl32(amax * rc))
 *   (round to nearest even, saturating at 448);  element code =
 *   E2M1(fl32(v * fl32(1 / fl32(s g)))) (nearest even, saturating at +-6, sign
 *   kept); a block whose scale is 0 gets zero codes.
 *   q  [rows, K / 2] bytes: element 2i in the low nibble of byte i;
 *   sf the E4M3 scale bytes in 512-byte atoms: rows [128 i, 128 i + 128) and
 *      blocks [4 j, 4 j + 4) form atom i * (K / 64) + j; row r / block b sits
 *      at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + b % 4 of its atom;
 *      ceil(rows / 128) * (K / 64) * 512 bytes.
 * All pointers 16-byte aligned (MOE_ERR_INVALID_ARG otherwise).  Enqueued on
 * `stream`.  The same kernel quantises an NVFP4 plan's weights. */
moe_status_t moe_nv_quantize(const void* src, int64_t rows, int64_t K, const float* g, void* q, void* sf,
                             moe_stream_t stream);

/* NVFP4 quantisation of the transposes of E bf16 row-major [A, B] device
 * matrices (src [E, A, B]) along A, tensor scale *g (NULL = 1): q [E, B, A / 2]
 * bytes (row e*B + b holds src[e, :, b]), sf the scale atoms of those E*B rows
 * with K = A (the layout of moe_nv_quantize).  A % 128 == 0, B % 64 == 0
 * (MOE_ERR_INVALID_ARG otherwise).  Enqueued on `stream`. */
moe_status_t moe_nv_quantize_transposed(const void* src, int64_t E, int64_t A, int64_t B, const float* g,
                                        void* q, void* sf, moe_stream_t stream);

/* Block-scaled plans created with MOE_DEBUG_DUMP_QUANT: copy a quantised
 * operand of the last forward / backward and the values it was quantised
 * from, over the plan's full padded row capacity P (the sorted rows of the
 * routing, each expert's segment padded to 128 rows; rows past the last
 * segment are not written).
 * which = 0 (h, forward) or 1 (dA|dB, backward): the fused epilogues'
 * quantisation along C = F (h) or 2F (dA|dB):
 *   vals [P, C] fp32 (the values the epilogue quantised);
 *   q    [P, C] E4M3 bytes (MXFP8) or [P, C / 2] packed E2M1 (NVFP4);
 *   sf   scale atoms of the P rows with K = C (moe_mx_quantize /
 *        moe_nv_quantize layout).
 * which = 2..5: the block-scaled weight gradients' operands, transposed and
 * quantised along the sorted rows (NVFP4 tensor scale 1): 2 dY^T and 3 X^T
 * (C = d), 4 [dA|dB]^T (C = 2F), 5 (w h)^T (C = F):
 *   vals [P, C] fp32: for 4 and 5 the bf16 values the u GEMM's epilogue
 *        quantised (the plan keeps them in this mode only), widened
 *        (must be NULL for 2 and 3, whose rows are the gathered inputs);
 *   q    [C, P] E4M3 bytes or [C, P / 2] packed E2M1;
 *   sf   scale atoms of the C rows with K = P.
 * which = 6: the dispatch's quantised sorted rows of the last call on the
 * separate-kernel schedule (X after moe_forward, dY after moe_backward;
 * quantised along d, NVFP4 tensor scale 1, padding rows zero):
 *   q    [P, d] E4M3 bytes or [P, d / 2] packed E2M1;
 *   sf   scale atoms of the P rows with K = d;  vals must be NULL.
 * P = moe_plan_padded_rows.  Any pointer may be NULL to skip it.  Synchronous
 * argument errors (MOE_ERR_INVALID_ARG) for a plan without the flag, a BF16
 * plan, another `which`, or vals with which 2, 3 or 6.  Enqueued on `stream`. */
moe_status_t moe_debug_quant_dump(moe_plan_t plan, int32_t which, float* vals, void* q, void* sf,
                                  moe_stream_t stream);

/* Padded sorted-row capacity P of a plan (for T = T_max). */
moe_status_t moe_plan_padded_rows(moe_plan_t plan, int64_t* rows);

/* NVFP4 plans: copy the two fp32 tensor scales moe_quantize_weights computed
 * ([0] Wg and Wu together, [1] Wd) into out (2 device floats), on `stream`.
 * MOE_ERR_INVALID_ARG for a null argument or a plan that is not MOE_NVFP4. */
moe_status_t moe_nv_weight_scales(moe_plan_t plan, float* out, moe_stream_t stream);

/* Copy the routing a forward stored in `saved` into caller device buffers
 * (any pointer may be NULL to skip it):
 *   idx [T, k] int32, w [T, k] fp32, counts [E] int32, offsets [E+1] int32
 *   (unpadded exclusive prefix of counts), perm_src [T*k] int32 (flat pair
 *   index t*k+j at each sorted row, padding removed), dest [T, k] int32
 *   (unpadded sorted row of each pair).  Enqueued on `stream`. */
moe_status_t moe_get_routing(moe_plan_t plan, int64_t T, const void* saved, int32_t* idx,
                             float* w, int32_t* counts, int32_t* offsets, int32_t* perm_src,
                             int32_t* dest, moe_stream_t stream);

/* Router GEMM, the step before the layer: logits = X Wr^T (kucoin page,
 * section 01: the router re-decides each token's experts at every step; the
 * pages print no router, and the plain reading is a linear map without bias).
 *   X      [T, d]  bf16 device, row-major (the same tokens moe_forward takes)
 *   Wr     [E, d]  bf16 device, row-major ([out, in] convention)
 *   logits [T, E]  fp32 device, written (the input moe_forward takes)
 * fp32 accumulation on the tensor cores; when T/128 tiles leave SMs idle,
 * the K range (d) is split over up to 8 tiles whose fp32 partials (plan
 * workspace) are summed in split order, so the result is deterministic for
 * a given T.  Needs E % 8 == 0 (MOE_ERR_UNSUPPORTED otherwise); T <= T_max;
 * all pointers 16-byte aligned (MOE_ERR_INVALID_ARG otherwise, nothing
 * enqueued).  T = 0 is a no-op.  Enqueued on `stream`. */
moe_status_t moe_router_forward(moe_plan_t plan, int64_t T, const void* X, const void* Wr, float* logits,
                                moe_stream_t stream);

/* Router GEMM backward.  Given dlogits [T, E] fp32 (moe_backward's dlogits):
 *   dX  [T, d]  bf16 device, read and written: dX += dlogits Wr (fp32 sum,
 *               one bf16 rounding), so passing moe_backward's dX gives the
 *               token gradient through both the experts and the router;
 *   dWr [E, d]  bf16 device, written: dWr = dlogits^T X, reduced over the T
 *               tokens in one fixed order (bitwise deterministic; split over
 *               up to 8 token ranges summed in range order when its
 *               E/128 x d/256 tiles leave SMs idle).
 * dlogits is rounded to bf16 for the tensor cores (into plan workspace).
 * Same shape, alignment and error rules as moe_router_forward; with T = 0,
 * dWr is zeroed and the other pointers are not used. */
moe_status_t moe_router_backward(moe_plan_t plan, int64_t T, const void* X, const void* Wr,
                                 const float* dlogits, void* dX, void* dWr, moe_stream_t stream);

/* Synchronise `stream`, read the plan's device status word into *status
 * (a moe_status_t value; MOE_OK if no device error), and clear it. */
moe_status_t moe_device_status(moe_plan_t plan, moe_stream_t stream, int32_t* status);

/* Per-kernel device times of the calls made since the last read, when the
 * plan was created with MOE_DEBUG_TIMING.  Synchronises the device.  Writes
 * up to `cap` entries: names[i] (static strings), total_ms[i] and launches[i];
 * *n receives the number of distinct kernels.  Resets the accumulators. */
moe_status_t moe_kernel_times(moe_plan_t plan, const char** names, double* total_ms,
                              int64_t* launches, int32_t cap, int32_t* n);

/* Launch geometry the plan chose on this device: num_sms (the persistent
 * kernels' grid: one CTA per SM), and the ring pipeline's shape ring[4] =
 * {mover CTAs (0: mover warps inside the compute CTAs), ring slots, minimum
 * minibatch in 128-row tiles (the two-wave
 * floor or minibatch_rows), largest minibatch in tiles (one slot)}.
 * Host-only; any pointer may be NULL. */
moe_status_t moe_plan_info(moe_plan_t plan, int32_t* num_sms, int32_t* ring);

/* Two-wave minibatch floor: the smallest row count m for which a grouped
 * GEMM of output width n_out cut into tile_m x tile_n tiles gives `waves`
 * full waves on `num_sms` SMs: m = ceil(waves * num_sms * tile_m * tile_n / n_out).
 * Pure host function (fluidifia page "Cursor ouvre
 * MoK, un mégakernel qui accélère l'entraînement MoE", section "Comment MoK
 * tente de gratter des millisecondes partout"; kucoin page, section 02). */
moe_status_t moe_minibatch_floor(int32_t num_sms, int32_t tile_m, int32_t tile_n, int32_t n_out,
                                 int32_t waves, int64_t* rows);

/* Routing without any device allocation.  The Mixture-of-Kittens pages have
 * no counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc -- e.g. code running inside a host framework whose allocator has
 * already reserved the device memory, or latency-critical paths that cannot
 * afford an allocation (which may synchronise the device).  moe_plan
 * allocates, so those callers cannot reach moe_forward's routing.
 *
 * Computes on the current device, enqueued on `stream`, exactly the routing
 * moe_forward stores and moe_get_routing returns (same kernels, same
 * results): idx [T, k] int32, w [T, k] fp32, counts [E] int32, offsets [E+1]
 * int32, perm_src [T*k] int32 and dest [T, k] int32, all caller-owned device
 * buffers.  logits [T, E] fp32.  Requires 1 <= k <= 32, k <= E <= 1024.
 *
 * Scratch lives in one fixed 4 MiB device array inside the library, which
 * every GPU that loads the library keeps until the process exits.  Under
 * CUDA's lazy module loading (the default) the 4 MiB is committed when the
 * library's module first loads on a device, possibly during this entry
 * point's first call there: a caller whose allocator will reserve the device
 * memory should make one warm-up call before it does.  A call needs about
 * 4*(2*ceil(T/64)*E + 2*T*k + 128*E) bytes of the array; larger calls return
 * MOE_ERR_UNSUPPORTED (see moe_last_error) and enqueue nothing.  Each call
 * made outside a stream capture looks up the array's device address on the
 * current device (so a device reset is followed correctly); a call during a
 * capture uses the address an earlier call looked up, so make the first call
 * on each device outside any capture (a first call inside one returns
 * MOE_ERR_INVALID_ARG).  All calls share the array and it
 * keeps the previous call's contents (each call writes every entry it reads,
 * so nothing needs clearing).  Calls that overlap on the GPU -- e.g. on two
 * streams without ordering between them -- race on the array.  Never calls
 * cudaMalloc, cudaFree or any allocating routine. */
moe_status_t moe_route_noalloc(int64_t T, int32_t E, int32_t k, const float* logits, int32_t* idx, float* w,
                               int32_t* counts, int32_t* offsets, int32_t* perm_src, int32_t* dest,
                               moe_stream_t stream);

/* Static description of a status code. */
const char* moe_status_string(moe_status_t s);

/* Human-readable detail of the last error returned on the calling thread. */
const char* moe_last_error(void);

#ifdef __cplusplus
}
#endif
#endif /* MOE_H */
