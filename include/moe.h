/*
 * moe.h -- C ABI of the GB300 fused Mixture-of-Experts expert layer.
 *
 * One layer computes, for T tokens with hidden size H, E experts of
 * intermediate size I and top-k K:
 *   1. routing: per token, the K largest router logits (value descending,
 *      lower expert index first on ties) and a softmax over those K;
 *   2. permutation: a stable histogram / scan / scatter of the T*K
 *      (token, k) slots into expert-contiguous order (per-expert offsets);
 *   3. the gate/up (W13) grouped GEMM, 4. SwiGLU with an optional symmetric
 *      gate/up clamp, fused with re-quantisation of its output,
 *   5. the down (W2) grouped GEMM, 6. the routing-weighted top-k combine
 *      back to token order.
 * The b12x integration report (PR #40082 report, "Integrate flashinfer b12x
 * MoE and FP4 GEMM kernels for SM120/121", sec. 实现拆解 item 1) describes the
 * same sequence run by a single call that takes bf16 hidden states and
 * quantises them itself; the optional gate/up clamp corresponds to
 * resolve_gate_up_clamp in the MegaMoE kernel-drop workflow page
 * ("FlashInfer CuTeDSL MegaMoE kernel-drop update workflow"), sec. 三.
 *
 * Weight formats (canonical inputs of moe_prepare_weights):
 *   MOE_FMT_BF16 : bf16 weights.
 *   MOE_FMT_MXFP8: e4m3 codes with one e8m0 scale per 32 elements along the
 *                  reduction dimension (mxfp8_quantize_per_block_32, same
 *                  workflow page, sec. 三).  Activations are quantised the
 *                  same way inside the layer (OCP MX shared exponent).
 *   MOE_FMT_NVFP4: e2m1 codes (two per byte, element 2j in the low nibble)
 *                  with one e4m3 scale per 16 elements and one fp32 global
 *                  scale per expert (nvfp4_quantize_per_block_16, sec. 三).
 *                  moe_prepare_weights folds the global scale into the block
 *                  scales (block_scale * global_scale re-cast to e4m3) so the
 *                  GEMMs run with alpha = 1, and activations are quantised
 *                  dynamically per 16-block with global scale 1 (PR #40082
 *                  report, sec. 关键源码片段, process_weights_after_loading).
 *
 * Conventions for every entry point:
 *   - Pointers marked "device" point to memory on the handle's CUDA device;
 *     "host" pointers to host memory (pinned memory makes copies faster).
 *     The caller owns every buffer it passes; the library never frees them.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously on it; calls return before
 *     the GPU finishes unless stated otherwise.
 *   - Every function returns a moe_status; MOE_OK is 0.  Argument errors
 *     are detected on the host before anything is enqueued.
 *   - Not thread-safe per handle: one host thread at a time per moe_layer.
 */
#ifndef MOE_GB300_H
#define MOE_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,    /* NULL handle/pointer, T out of range ...   */
    MOE_ERR_UNSUPPORTED = 2,    /* shape/format this build does not run      */
    MOE_ERR_NO_WEIGHTS = 3,     /* moe_forward before moe_prepare_weights    */
    MOE_ERR_CUDA = 4,           /* a CUDA runtime/driver call failed         */
    MOE_ERR_OOM = 5,            /* device allocation failed                  */
    MOE_ERR_DEVICE_TIMEOUT = 6, /* a kernel gave up a bounded wait           */
    MOE_ERR_NO_DEVICE = 7       /* no sm_103-class GPU / kernel image        */
} moe_status;

typedef enum { MOE_FMT_BF16 = 0, MOE_FMT_MXFP8 = 1, MOE_FMT_NVFP4 = 2 } moe_format;

/* Expert activation.  SwiGLU is gated (W13 = gate and up projections);
 * ReLU^2 is the non-gated squared ReLU of one projection, h = max(x, 0)^2,
 * which the b12x backend cannot load (PR #40082 report, sec. 风险与影响
 * item 4: models without a gated act-and-mul MLP, e.g. Nemotron).        */
typedef enum { MOE_ACT_SWIGLU = 0, MOE_ACT_RELU2 = 1 } moe_activation;

/* How the K expert outputs of a token are summed.  GATHER (default): GEMM2
 * stores each routed row's output as bf16 and a separate kernel sums the K
 * rows of every token in k order (deterministic).  REDUCE: GEMM2's epilogue
 * adds w * (fp32 output) into an fp32 accumulator with atomics and the last
 * of a token's K contributions writes the bf16 result, so no combine kernel
 * runs; the summation order, hence the last bits, can differ from run to
 * run (the in-kernel reduce the MegaMoE kernel-drop workflow page, sec. 六,
 * weighs against a deterministic combine).                                 */
/* FUSED: the same deterministic gather as GATHER, done inside GEMM2's
 * epilogue: in each 128-column group, the last of a token's K rows to be
 * stored sums the token's K rows in k order in fp32 and writes the bf16
 * result (bit-identical to GATHER), so no combine kernel runs (the combine
 * folded into the expert GEMM, as the MegaMoE kernel fuses its FC2 with the
 * reduction, sec. 六; here without atomics on the output).  Only
 * prefill-sized launches (T > 1024 and H a multiple of 256: the 256-column
 * GEMM2 items) fuse it;
 * smaller ones run the combine kernel (T <= 16: the single-launch decode
 * kernel's own combine), so their GEMM kernels carry no gather.  Measured
 * slower than GATHER on GB300 (the gathers lengthen GEMM2's epilogue).     */
typedef enum {
    MOE_COMBINE_GATHER = 0,
    MOE_COMBINE_REDUCE = 1,
    MOE_COMBINE_FUSED = 2
} moe_combine;

typedef struct {
    int max_tokens;    /* T_max: largest T any forward will use (>= 1)       */
    int hidden;        /* H: multiple of 128 (NVFP4: of 256)                 */
    int inter;         /* I: multiple of 128 (NVFP4: of 256)                 */
    int num_experts;   /* E: 1..512                                          */
    int top_k;         /* K: 1..min(E, 16)                                   */
    int format;        /* moe_format                                         */
    float clamp_limit; /* L > 0 and finite: clamp gate and up to [-L, L]
                          before silu(gate)*up; otherwise no clamp (a clamp
                          with MOE_ACT_RELU2 is MOE_ERR_UNSUPPORTED)        */
    int activation;    /* moe_activation (0 = SwiGLU)                       */
    int combine;       /* moe_combine (0 = gather)                          */
    int max_ctas;      /* > 0: at most this many CTAs per GEMM launch (to
                          share the GPU with concurrent work); 0: one CTA
                          per SM                                            */
    /* Fault injection for the library's own tests; 0 = off.  Nothing else
     * turns these on (they are not read from the environment).            */
    int test_fail_alloc_at; /* n > 0: the n-th device allocation made by
                               moe_create fails (MOE_ERR_OOM, nothing leaks) */
    int test_stall_gemm;    /* 1: CTA 0 of every GEMM1 launch leaves one
                               shared-memory stage unloaded, so the waits on
                               it run out after 2 s and the forward records
                               MOE_ERR_DEVICE_TIMEOUT (no fault, no hang)   */
} moe_config;

typedef struct moe_layer moe_layer;   /* opaque */

/* Create a layer on the current CUDA device.  Validates `cfg` and allocates
 * every device buffer a forward of up to cfg->max_tokens tokens needs
 * (weights, routing tables, permuted activations, intermediates), so that
 * moe_forward never allocates: the workspace is sized once by the largest
 * token count, as MegaMoE sizes its own by num_max_tokens (MegaMoE
 * kernel-drop workflow page, sec. 六).  E and K are fixed here and every
 * launch uses this E (a global-vs-local expert count mismatch broke the
 * b12x integration: PR #40082 report, sec. 风险与影响 item 3).  *out receives the handle (NULL on error).
 * Errors: MOE_ERR_INVALID_ARG (NULL args), MOE_ERR_UNSUPPORTED (shape),
 * MOE_ERR_NO_DEVICE, MOE_ERR_OOM (nothing leaks), MOE_ERR_CUDA.            */
moe_status moe_create(const moe_config *cfg, moe_layer **out);

/* Copy the canonical weights into the layer's own buffers and transform them
 * into the kernels' layout once, at load time rather than per forward, with
 * the NVFP4 global scale folded into the block scales (the b12x
 * process_weights_after_loading step: PR #40082 report, sec. 关键源码片段;
 * the scale-layout conversion moved to load time: same report, sec.
 * 评论区精华) (untimed set-up, enqueued on `stream`; returns
 * after enqueueing, the caller may free its buffers once `stream` has
 * finished).  All pointers are device pointers, row-major, reduction
 * dimension contiguous; W13 rows 0..I-1 are the gate projection and rows
 * I..2I-1 the up projection (MOE_ACT_RELU2: W13 is the single projection,
 * I rows, so every "2I" below reads "I"):
 *   BF16 : w13 bf16 [E, 2I, H];  w2 bf16 [E, H, I];  *_sf, *_gs unused.
 *   MXFP8: w13 e4m3 [E, 2I, H], w13_sf e8m0 [E, 2I, H/32];
 *          w2  e4m3 [E, H, I],  w2_sf  e8m0 [E, H, I/32];  *_gs unused.
 *   NVFP4: w13 u8 [E, 2I, H/2], w13_sf e4m3 [E, 2I, H/16], w13_gs f32 [E];
 *          w2  u8 [E, H, I/2],  w2_sf  e4m3 [E, H, I/16],  w2_gs  f32 [E].
 * NVFP4 block scales are multiplied by the expert's global scale and re-cast
 * to e4m3 (the global scale becomes 1); scales are re-laid out in 128-row x
 * 4-block tiles for the tensor cores.  Errors: MOE_ERR_INVALID_ARG when a
 * pointer the format needs is NULL; MOE_ERR_CUDA.                          */
moe_status moe_prepare_weights(moe_layer *layer,
                               const void *w13, const void *w13_sf,
                               const float *w13_gs,
                               const void *w2, const void *w2_sf,
                               const float *w2_gs, void *stream);

/* The layer forward: routing, permutation, activation quantisation, GEMM1,
 * SwiGLU, GEMM2 and the combine on bf16 hidden states, as the b12x call runs
 * them (PR #40082 report, sec. 实现拆解 item 1).  hidden: device bf16 [T, H];
 * router_logits: device f32 [T, E]; out: device bf16 [T, H], written in
 * place, never re-bound or reallocated (a backend that re-bound its output
 * left the caller's buffer unwritten: PR 38050 analysis report, sec.
 * 评论区精华).  hidden and out 16-byte aligned, router_logits 4-byte
 * aligned (else MOE_ERR_INVALID_ARG).  0 <= T <= max_tokens; T == 0 is a
 * no-op returning MOE_OK.
 * Asynchronous on `stream`, allocates nothing, never synchronises the host.
 * Results of a later moe_debug_* call describe the latest forward.
 * Errors: MOE_ERR_INVALID_ARG, MOE_ERR_NO_WEIGHTS, MOE_ERR_CUDA (launch).
 * A kernel that gives up a bounded wait records MOE_ERR_DEVICE_TIMEOUT for
 * moe_get_status.                                                          */
moe_status moe_forward(moe_layer *layer, const void *hidden,
                       const float *router_logits, void *out, int T,
                       void *stream);

/* The expert computation on the batched-expert activation format: no
 * routing, permutation or combine (the batched-experts variant of PR 38050
 * analysis report, sec. 实现拆解: activations already grouped per expert,
 * a per-expert token count, outputs in the same layout).  hidden: device
 * bf16 [E, M, H]; counts: device int32 [E], rows 0..counts[e]-1 of block e
 * belong to expert e; out: device bf16 [E, M, H]; hidden and out 16-byte
 * aligned, counts 4-byte aligned.  Each counted row goes
 * through the activation quantisation, GEMM1, the activation with its
 * re-quantisation and GEMM2 of its expert; out receives the bf16 GEMM2
 * output in the same row.  Rows past a count are neither read nor written.
 * 0 <= M and E * roundup(M, 128) <= the capacity moe_create sized for
 * max_tokens * top_k routed rows (else MOE_ERR_UNSUPPORTED); M == 0 is a
 * no-op.  A count outside [0, M] is clamped to that range and recorded as
 * MOE_ERR_INVALID_ARG for moe_get_status.  Asynchronous on `stream`,
 * allocates nothing.  Errors: MOE_ERR_INVALID_ARG, MOE_ERR_UNSUPPORTED,
 * MOE_ERR_NO_WEIGHTS, MOE_ERR_CUDA.                                        */
moe_status moe_forward_batched(moe_layer *layer, const void *hidden,
                               const int32_t *counts, int M, void *out,
                               void *stream);

/* (The build's own call, for the end-to-end measurement.)  Same as
 * moe_forward with HOST buffers: copies hidden [T,H] bf16 and
 * router_logits [T,E] f32 to the device, runs the layer and copies out
 * [T,H] bf16 back, all on `stream`; returns once `stream` has finished
 * (synchronises it).  When all three buffers are page-locked host memory
 * the device can address (cudaHostAlloc / cudaHostRegister on a coherent
 * Grace-Blackwell node) and aligned as moe_forward asks, the kernels read
 * the inputs and write the output in host memory directly instead of
 * copying; host buffers of any alignment go through the copies.  Errors as
 * moe_forward.                                                            */
moe_status moe_forward_host(moe_layer *layer, const void *hidden_host,
                            const float *router_logits_host, void *out_host,
                            int T, void *stream);

/* (The build's own call, no counterpart on the pages.)  moe_forward with
 * HOST buffers, pipelined: enqueues the copy of hidden [T,H] bf16 and
 * router_logits [T,E] f32 to the device, the layer, and the copy of out
 * [T,H] bf16 back, and returns without waiting.  `stream` completes once
 * out_host holds the result; until then the three host buffers must stay
 * as they are (page-locked memory lets the copies overlap).  The copies run
 * on a copy stream and the layer on a compute stream of the layer's own
 * (created on the first call), both ordered after the work `stream` held at
 * the call.  Consecutive calls overlap: step i+1's input copy waits only
 * until step i's front end has read the device input buffers, and step i's
 * output copy runs while step i+1 computes.  Decode-sized steps (T <= 16)
 * whose buffers are page-locked memory the device can address skip the
 * copies: the layer reads and writes the host buffers in place (see
 * moe_forward_host).  One layer's calls must come from one host thread at a
 * time, and they cannot be captured into a CUDA graph (their work runs on
 * the layer's own streams; capture moe_forward with device buffers
 * instead).  Errors as moe_forward; MOE_ERR_CUDA if the streams cannot be
 * created.                                                                */
moe_status moe_forward_host_async(moe_layer *layer, const void *hidden_host,
                                  const float *router_logits_host,
                                  void *out_host, int T, void *stream);

/* Inspection of the latest forward (tests; the build's own call, no
 * counterpart on the pages): device destinations, any may be NULL.  topk_ids int32 [T,K], topk_w f32 [T,K], offsets int32 [E+1]
 * (offsets[e] = first permuted row of expert e, offsets[E] = T*K),
 * perm int32 [T*K] (permuted row -> slot t*K+k).  Enqueued on `stream`.   */
moe_status moe_debug_routing(moe_layer *layer, int32_t *topk_ids,
                             float *topk_w, int32_t *offsets, int32_t *perm,
                             void *stream);

/* GEMM1 input quantisation of the latest forward (tests; the build's own
 * call), per token, canonical layout: codes [T, H/2] (NVFP4) or [T, H] (MXFP8), scales [T, H/16] or
 * [T, H/32].  Device destinations.  MOE_ERR_UNSUPPORTED for BF16.         */
moe_status moe_debug_act_quant(moe_layer *layer, uint8_t *codes,
                               uint8_t *scales, void *stream);

/* (Tests; the build's own call.)  GEMM2 input (SwiGLU output after
 * re-quantisation, dequantised to f32,
 * [T*K, I]) and GEMM2 output (f32 of the stored bf16, [T*K, H]) of the
 * latest forward, in permuted row order.  Device destinations, may be NULL. */
moe_status moe_debug_intermediates(moe_layer *layer, float *h, float *y,
                                   void *stream);

/* The prepared weight tiles of one expert, as moe_prepare_weights left them
 * (inspection for tests of the weight preparation).  which = 13 (W13) or
 * 2 (W2); dst: device or host destination of exactly dst_bytes =
 * (N/128) * (K_bytes/128) * tile_bytes, where N is the matrix's rows (W13:
 * 2I, or I for ReLU^2; W2: H), K_bytes its row length in bytes (H or I
 * times 2, 1 or 1/2 for BF16 / MXFP8 / NVFP4) and tile_bytes 16384 plus
 * 512 per scale tile (NVFP4 4, MXFP8 1, BF16 0).  Layout: tiles ordered by
 * 128-row block, then 128-byte K slice; a tile is 128 rows x 128 bytes of
 * codes, 16-byte chunk c of row r at byte r*128 + (c ^ (r % 8))*16 (the
 * 128-byte swizzle), then the slice's scale tiles, scale j of tile row r at
 * (r % 32)*16 + (r / 32)*4 + j.  W13 rows are interleaved in groups of
 * 64 for SwiGLU: prepared row 128g + r is gate row 64g + r for r < 64 and
 * up row I + 64g + r - 64 otherwise.  NVFP4 scales are the folded ones
 * (e4m3(float(sf) * gs)).  Errors: MOE_ERR_INVALID_ARG (bad which, expert
 * or size), MOE_ERR_NO_WEIGHTS, MOE_ERR_CUDA.  Enqueued on `stream`.
 * The build's own inspection call; the pages have no counterpart.        */
moe_status moe_debug_weight_tiles(moe_layer *layer, int which, int expert,
                                  void *dst, size_t dst_bytes, void *stream);

/* Device-side error word of the handle (the build's own call; the pages
 * have no counterpart): synchronises the device, returns
 * the first error a kernel recorded since the last call (and clears it):
 * MOE_ERR_DEVICE_TIMEOUT if a kernel gave up a bounded wait,
 * MOE_ERR_INVALID_ARG if moe_forward_batched met a count outside [0, M];
 * MOE_ERR_CUDA on a sticky CUDA error; else MOE_OK.                        */
moe_status moe_get_status(moe_layer *layer);

/* Per-kernel timing (profiling; the build's own call).  While on, every moe_forward records a CUDA
 * event before each of its six kernels and one after the last, for at most
 * max_forwards forwards; the events are created here, not in the forward.
 * moe_timing_stop waits for the recorded work, writes the summed duration
 * of each kernel in milliseconds to kernel_ms[6] (routing, scan, scatter +
 * activation quantisation, GEMM1 + SwiGLU, GEMM2, combine; for T <= 16 one
 * kernel does routing .. quantisation and is counted as routing, scan and
 * scatter reading 0) and the number of recorded forwards to *forwards, and
 * turns timing off.  Errors:
 * MOE_ERR_INVALID_ARG, MOE_ERR_CUDA.                                       */
moe_status moe_timing_start(moe_layer *layer, int max_forwards);
moe_status moe_timing_stop(moe_layer *layer, float *kernel_ms, int *forwards);

/* Number of kernel launches the latest moe_forward enqueued (the build's
 * own call).                                                              */
int moe_last_launch_count(const moe_layer *layer);

/* Largest number of CTAs a GEMM launch of this layer uses (the build's own
 * call): wide != 0 for the prefill-sized launches (NVFP4: CTA pairs, two
 * CTAs each), 0 for the others.  0 for a NULL handle.                    */
int moe_gemm_ctas(const moe_layer *layer, int wide);

/* Routing and expert permutation without any device allocation.  The pages
 * have no counterpart of this entry point; it exists for callers that cannot
 * call cudaMalloc -- e.g. a serving framework whose caching allocator
 * already owns the GPU's memory, or a latency-critical caller that cannot
 * accept the device-wide synchronisation an allocation may cause.
 * Computes exactly what moe_forward's routing + permutation step computes
 * (see moe_debug_routing): router_logits device f32 [T,E] in; device
 * outputs topk_ids int32 [T,K], topk_w f32 [T,K], offsets int32 [E+1],
 * perm int32 [T*K].  Needs no handle.  Its scratch is one fixed 256 KiB
 * device array inside the library (held on every GPU that loads it until
 * the process exits), which limits it to T <= 4096, E <= 512, K <= 16:
 * larger sizes return MOE_ERR_UNSUPPORTED.  The first call on a device looks
 * up that array's device address (make that first call before any stream
 * capture).  All calls share the array: calls whose work overlaps on the
 * GPU (other streams, unordered host threads) race and give wrong results.
 * Errors: MOE_ERR_INVALID_ARG (T < 0, K > E, a NULL or not 4-byte aligned
 * pointer; found on the host, nothing is launched), MOE_ERR_UNSUPPORTED,
 * MOE_ERR_CUDA (a launch failed; earlier errors of the context are neither
 * reported nor cleared).  T == 0 is a no-op.                               */
moe_status moe_route_permute_static(const float *router_logits, int T, int E,
                                    int K, int32_t *topk_ids, float *topk_w,
                                    int32_t *offsets, int32_t *perm,
                                    void *stream);

/* Tensor-pipe rate of one MMA kind on this GPU (measurement, not part of the
 * layer): one CTA per SM issues `iters` groups of four back-to-back
 * tcgen05.mma (M = 128, N = n_cols in {128, 256}) on zero operands resident
 * in shared memory -- the layer's instruction shapes: kind::f16 (BF16,
 * K = 16), kind::mxf8f6f4 block-scaled 1X (MXFP8, K = 32) or kind::mxf4nvf4
 * block-scaled 4X (NVFP4, K = 64) -- and reports dense TFLOP/s in *tflops
 * (host pointer), timed with CUDA events on `stream` (blocks until done).
 * copy_scales != 0 (MXFP8/NVFP4, n_cols 128 only) also copies the scale
 * tiles into TMEM before each group, as the layer's GEMM does per stage.
 * The roofline of a block-scaled contraction needs this rate: the pages
 * quote none for GB300.  Errors: MOE_ERR_INVALID_ARG (iters outside
 * 1..2^20, bad format or n_cols), MOE_ERR_UNSUPPORTED, MOE_ERR_NO_DEVICE,
 * MOE_ERR_CUDA, MOE_ERR_DEVICE_TIMEOUT (a wait gave up after 2 s).        */
moe_status moe_measure_mma_rate(int format, int n_cols, int copy_scales,
                                int iters, double *tflops, void *stream);

/* Static description of a status code (never NULL; the build's own call). */
const char *moe_status_string(moe_status s);

/* Free everything the handle owns.  NULL-safe.  Synchronises the device
 * first so no enqueued work still uses the buffers.  (The build's own call:
 * the pages manage the layer's memory through the framework.)            */
void moe_destroy(moe_layer *layer);

#ifdef __cplusplus
}
#endif
#endif
