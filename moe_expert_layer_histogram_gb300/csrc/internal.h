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
constexpr int kTokensPerRouteBlock = 64;  // tokens per routing/scatter block
constexpr int kRowBlock = 128;            // expert segments padded to this
constexpr int kGemmStages = 6;            // shared-memory pipeline depth
constexpr int kGemmThreads = 192;         // producer, MMA, 4 epilogue warps

// Per-launch arguments of the grouped GEMMs.  Work items are (expert,
// output tile of 128 columns of the weight rows, 128-row token chunk),
// expert-major, then output tile, then chunk.
struct GemmArgs {
  const int32_t* chunk_off;  // [E+1] exclusive scan of ceil(count/128)
  const int32_t* pad_off;    // [E+1] exclusive scan of round_up(count,128)
  const int32_t* counts;     // [E]
  int E;
  int n_tiles;               // output tiles per expert
  int num_kb;                // 128-byte K stages per item
  int b_rows_per_expert;     // weight rows per expert (2I or H)
  const uint8_t* sfa;        // activation scales, 128x4 tiles
  int sfa_tiles_k;
  const uint8_t* sfb;        // weight scales, 128x4 tiles
  int sfb_tiles_k;
  uint8_t* out;              // GEMM1: GEMM2 input codes; GEMM2: y (bf16)
  int64_t out_ld;            // bytes per output row
  uint8_t* out_sf;           // GEMM1 (MX/NV): GEMM2 input scales
  int out_sf_tiles_k;
  float clamp;               // +inf: no clamp
  int* status;
};

struct GemmMaps {
  CUtensorMap a[4];  // activation rows, boxes of 16/32/64/128 rows x 128 B
  CUtensorMap b;     // weight rows, box 128 rows x 128 B
};

size_t gemm_smem_bytes(int fmt);
cudaError_t gemm_prepare(int fmt);  // raise the dynamic shared-memory limit
cudaError_t launch_gemm(int fmt, int epi, const GemmMaps& maps, const GemmArgs& args, int grid,
                        cudaStream_t s);

// Routing, permutation + activation quantisation, combine.
cudaError_t launch_route_hist(const float* logits, int T, int E, int K, int32_t* ids, float* w,
                              int32_t* blockhist, cudaStream_t s);
cudaError_t launch_scan(const int32_t* blockhist, int NB, int E, int32_t* offsets,
                        int32_t* pad_off, int32_t* chunk_off, int32_t* counts, int32_t* base,
                        int32_t* pbase, cudaStream_t s);
cudaError_t launch_scatter_quant(int fmt, const int32_t* ids, int T, int E, int K,
                                 const void* hidden, int H, const int32_t* base,
                                 const int32_t* pbase, int32_t* perm, int32_t* inv, uint8_t* xq,
                                 uint8_t* xsf, cudaStream_t s);
cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int T, int K, int H,
                           void* out, cudaStream_t s);

// Weight preparation.
cudaError_t launch_copy_rows(const uint8_t* src, uint8_t* dst, int64_t rows, int64_t row_bytes,
                             int N, int interleave_half, cudaStream_t s);
cudaError_t launch_sf_tiles(const uint8_t* src, uint8_t* dst, int E, int N, int nkg,
                            const float* gs, int interleave_half, cudaStream_t s);

// Inspection.
cudaError_t launch_debug_act(int fmt, const int32_t* inv, int T, int K, int H, const uint8_t* xq,
                             const uint8_t* xsf, uint8_t* codes, uint8_t* scales,
                             cudaStream_t s);
cudaError_t launch_debug_rows(int fmt, const int32_t* offsets, const int32_t* pad_off, int E,
                              int R, int I, int H, const uint8_t* hq, const uint8_t* hsf,
                              const void* y, float* h_out, float* y_out, cudaStream_t s);

}  // namespace moe
