// internal.h -- declarations shared by the host runtime and the kernel
// translation units of the GB300 MoE expert-layer library.
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

namespace moe {

constexpr int kFmtBF16 = 0, kFmtMXFP8 = 1, kFmtNVFP4 = 2;

constexpr int kMaxExperts = 512;
constexpr int kMaxTopK = 16;
constexpr int kTokensPerRouteBlock = 8;   // tokens per routing/scatter block (warp each)
constexpr int kSmallFrontTokens = 16;     // up to this T one block does routing..quantisation
constexpr int kRowBlock = 128;            // expert segments padded to this

// Device status word codes (read back by moe_get_status).
constexpr int kStatusBadCount = 1;  // MOE_ERR_INVALID_ARG: a batched count outside [0, M]
constexpr int kStatusTimeout = 6;   // MOE_ERR_DEVICE_TIMEOUT: a bounded wait gave up

#ifdef __CUDACC__
// First error wins.
__device__ __forceinline__ void report_status(int* status, int code) {
  if (status) atomicCAS(status, 0, code);
}
#endif

// Per-launch arguments of the grouped GEMMs.  Work items are (expert,
// output tile of 128 columns of the weight rows, 128-row token chunk),
// expert-major, then output tile, then chunk.
struct GemmArgs {
  const int32_t* chunk_off;  // [E+1] exclusive scan of ceil(count/128)
  const int32_t* pad_off;    // [E+1] exclusive scan of round_up(count,128)
  const int32_t* counts;     // [E]
  // [E+1] or null: the three tables above are by table position and this is
  // the expert at each position, then the multi-chunk positions' chunks
  // (the mixed item order, gemm_common.cuh); null: position = expert
  const int32_t* order;
  int E;
  int n_tiles;               // output tiles per expert
  int num_kb;                // 128-byte K stages per item
  const uint8_t* sfa;        // activation scales, 128x4 tiles
  int sfa_tiles_k;
  const uint8_t* b_tiles;    // weight tiles (see weight_tile_bytes), expert-major
  int b_tile_bytes;
  uint8_t* out;              // GEMM1: GEMM2 input codes; GEMM2: y (bf16)
  int64_t out_ld;            // bytes per output row
  uint8_t* out_sf;           // GEMM1 (MX/NV): GEMM2 input scales
  int out_sf_tiles_k;
  float clamp;               // +inf: no clamp
  int pair_scale_copies;     // 1: chunks of <= 32 rows need scales in lanes 0-31 only
  int stage_scales;          // 1: ... which a dedicated warp writes there (tcgen05.st)
  // GEMM2 with the in-kernel reduce (acc != nullptr): out[t] = bf16(sum_k
  // w[t,k] * y), summed in `acc` (fp32 [T, H], zero between forwards) with
  // atomics; acc_cnt [T, H/128] counts contributions per 128-column group.
  float* acc;
  int32_t* acc_cnt;
  const int32_t* prow_slot;  // padded row -> slot t*K + k
  const float* topk_w;       // [T*K]
  uint8_t* comb_out;         // bf16 [T, H]
  // GEMM2 with the fused combine (gather_inv != nullptr): the K-th stored row
  // of a token's 128-column group gathers the token's K rows of y (slot ->
  // padded row) and writes the group of comb_out; acc_cnt counts the rows,
  // prow_slot / topk_w as above, acc unused.
  const int32_t* gather_inv;
  int K, H;
  int32_t* done1;            // fused GEMM1+GEMM2 launch: per expert, GEMM1 epilogue warps done
  int test_stall;            // test hook: CTA 0 never loads one stage, so the waits on it
                             // run out (bounded) and the kernel reports a timeout
  int out_rows_per_expert;   // 0: output row = padded row; M > 0 (batched format):
                             // output row = e * M + row within the expert
  int* status;
};

struct GemmMaps {
  CUtensorMap a[4];  // activation rows, boxes of 16/32/64/128 rows x 128 B
  CUtensorMap b;     // NVFP4 prepared weight tiles as rows of 2 KiB, boxes of 8 rows (a
                     // tile's 16 KiB of codes), no swizzle (stored pre-swizzled);
                     // CTA-pair kernels
};

// Prepared weights are stored as tiles, one per (expert, 128-row block of
// the weight matrix, 128-byte slice of the reduction dimension), in that
// order.  A tile is 16 KiB of codes -- 128 rows of 128 bytes, already in the
// 128-byte-swizzled order the MMA descriptors expect (16-byte chunk c of row
// r stored at chunk c ^ (r % 8)) -- followed by the slice's block-scale
// tiles (NVFP4: 4 x 512 bytes, MXFP8: 1 x 512, BF16: none).  One stage of
// a GEMM fetches one tile with one contiguous bulk copy.
constexpr int weight_sf_tiles(int fmt) { return fmt == kFmtNVFP4 ? 4 : fmt == kFmtMXFP8 ? 1 : 0; }
constexpr int weight_tile_bytes(int fmt) { return 128 * 128 + 512 * weight_sf_tiles(fmt); }

// Programmatic dependent launch: every kernel of a decode-sized forward is
// launched with programmatic stream serialization, lets its dependents
// launch as soon as it starts, runs its input-independent prologue and
// waits for the previous kernel (griddepcontrol.wait) before it touches data
// that kernel produced or still reads.  Prefill-sized (wide) forwards launch
// without it: there the early dependents measured slower (T = 32768: 7.26 ->
// 6.38 ms per layer without; T = 8192: 1.94 -> 1.88 ms).  Set per forward on
// the calling host thread from the layer's settings (moe_create reads
// MOE_DISABLE_PDL=1|gemm|small and MOE_PDL_PREFILL=1).
extern thread_local bool g_pdl_small, g_pdl_gemm;

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(bool pdl, void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cfg.attrs = attr;
  cfg.numAttrs = pdl ? 1 : 0;
  return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

#ifdef __CUDACC__
__device__ __forceinline__ void pdl_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
#endif

cudaError_t gemm_prepare(int fmt);  // raise the dynamic shared-memory limit
// max_rows: upper bound on the rows of any expert in this launch (<= T);
// selects the activation-tile height of the shared-memory stages.
// epi: 1 = GEMM1 + SwiGLU, 3 = GEMM1 + ReLU^2 (both re-quantise into the
// GEMM2 input format), 2 = GEMM2 (bf16 out), 4 = GEMM2 with the fused
// combine (args.gather_inv; wide launches only).  wide: items of two 128-row
// weight tiles (MMA N = 256; args.n_tiles counts those pairs), for launches
// whose chunks are mostly full 128-row blocks.
cudaError_t launch_gemm(int fmt, int epi, const GemmMaps& maps, const GemmArgs& args, int grid,
                        int max_rows, bool wide, cudaStream_t s);
// Decode (chunks of at most 32 rows, narrow items): GEMM1 (epi1 = 1 or 3)
// and GEMM2 in one persistent launch; args1.done1 must be zero per expert.
cudaError_t launch_gemm_fused(int fmt, int epi1, const GemmMaps& maps1, const GemmArgs& args1,
                              const GemmMaps& maps2, const GemmArgs& args2, int grid,
                              int max_rows, cudaStream_t s);

// NVFP4 wide launches on CTA pairs (tcgen05 cta_group::2, 256 x 256 MMA
// tiles): prepare once (sets the shared-memory limit, checks the register
// split, returns the largest number of co-resident CTA pairs); launch with
// `clusters` pairs (args as for wide items: n_tiles counts 256-row pairs).
cudaError_t gemm_pair_prepare(int* max_clusters);
cudaError_t launch_gemm_pair(int epi, const GemmMaps& maps, const GemmArgs& args, int clusters,
                             cudaStream_t s);

// Single-launch decode layer (T <= kSmallFrontTokens): routing, tables,
// GEMM1 input, both GEMMs and the combine in one persistent kernel.  The
// counters below coordinate its CTAs; they are zero between forwards (the
// kernel's last CTA resets them).
struct DecodeCtl {
  int qclaim, qdone;    // GEMM1-input tokens claimed / stored
  int iclaim;           // GEMM items claimed
  int cclaim;           // combine units claimed
  int exits;            // CTAs finished
  int pad[3];
  int done1[kMaxExperts];  // per expert: GEMM1 epilogue warps finished
  int done2[kMaxExperts];  // per expert: GEMM2 epilogue warps finished
};

struct DecodeArgs {
  const float* logits;   // [T, E]
  const void* hidden;    // bf16 [T, H]
  int T, K, H;
  // routing tables (written by CTA 0, for inspection)
  int32_t *ids, *counts, *offsets, *pad_off, *chunk_off, *perm, *inv;
  float* w;
  uint8_t *xq, *xsf;     // GEMM1 input rows and their scale tiles
  uint8_t* out;          // bf16 [T, H]
  DecodeCtl* ctl;
};

cudaError_t decode_prepare(int fmt);
// args1/args2: GEMM1 / GEMM2 arguments as for launch_gemm (narrow items;
// their table pointers are not read: the kernel builds the tables itself).
cudaError_t launch_decode(int fmt, int epi1, const GemmMaps& maps1, const GemmArgs& args1,
                          const GemmMaps& maps2, const GemmArgs& args2, const DecodeArgs& d,
                          int grid, cudaStream_t s);

// Routing, permutation + activation quantisation, combine.
cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* w,
                         int32_t* blockhist, cudaStream_t s);
cudaError_t launch_expert_scan(const int32_t* blockhist, int NB, int E, int32_t* prefix,
                               int32_t* counts, cudaStream_t s);
// prow_slot (may be null): padded row -> slot, for the in-kernel reduce.
// otab (may be null): [4E+2] the GEMMs' item tables in the mixed order
// (GemmArgs::order).
cudaError_t launch_scatter_quant(int fmt, const int32_t* ids, int T, int E, int K,
                                 const void* hidden, int H, const int32_t* prefix,
                                 const int32_t* counts, int32_t* offsets, int32_t* pad_off,
                                 int32_t* chunk_off, int32_t* perm, int32_t* inv,
                                 int32_t* prow_slot, int32_t* otab, uint8_t* xq, uint8_t* xsf,
                                 cudaStream_t s);
cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int T, int K, int H,
                           void* out, cudaStream_t s);
// T <= kSmallFrontTokens: routing, scans, ranks and GEMM1 input in one block.
// done1 (may be null): per-expert counters of a following fused GEMM launch,
// zeroed here.
cudaError_t launch_small_front(int fmt, const float* logits, int T, int E, int K,
                               const void* hidden, int H, int32_t* ids, float* w,
                               int32_t* counts, int32_t* offsets, int32_t* pad_off,
                               int32_t* chunk_off, int32_t* perm, int32_t* inv,
                               int32_t* prow_slot, int32_t* done1, uint8_t* xq, uint8_t* xsf,
                               cudaStream_t s);
// Batched-expert format: per-expert tables from the counts and the GEMM1
// input rows of hidden [E, M, H].
cudaError_t launch_batched_quant(int fmt, const void* hidden, const int32_t* counts_in, int M,
                                 int E, int H, int32_t* counts, int32_t* offsets,
                                 int32_t* pad_off, int32_t* chunk_off, uint8_t* xq, uint8_t* xsf,
                                 int* status, cudaStream_t s);

// Weight preparation.
cudaError_t launch_tile_weights(int fmt, const uint8_t* codes, const uint8_t* sf, const float* gs,
                                uint8_t* tiles, int E, int N, int row_bytes, int nkg,
                                int interleave_half, cudaStream_t s);

// Inspection.
cudaError_t launch_debug_act(int fmt, const int32_t* inv, int T, int K, int H, const uint8_t* xq,
                             const uint8_t* xsf, uint8_t* codes, uint8_t* scales,
                             cudaStream_t s);
cudaError_t launch_debug_rows(int fmt, const int32_t* offsets, const int32_t* pad_off, int E,
                              int R, int I, int H, const uint8_t* hq, const uint8_t* hsf,
                              const void* y, float* h_out, float* y_out, cudaStream_t s);

}  // namespace moe
