// prep.cu -- one-time weight preparation (untimed set-up).
//
// The canonical quantised weights are copied into the layer's own buffers
// and re-laid out for the grouped GEMMs:
//  - W13 rows are interleaved in 64-row groups (64 gate rows, then the 64
//    matching up rows, ...), so one 128-row weight tile holds the gate and up
//    halves of the same 64 intermediate features and the GEMM1 epilogue sees
//    both in one accumulator row;
//  - codes are cut into 16 KiB tiles (128 rows x 128 bytes of K), stored
//    contiguously and pre-swizzled, so every GEMM stage reads one contiguous
//    block of HBM instead of 128 short row segments;
//  - block scales are re-laid out into 128-row x 4-scale tiles for the
//    tensor cores; like the b12x integration, which converts its scales to
//    the MMA layout once at weight-load time (PR #40082 report, sec.
//    关键源码片段), this happens once, not per forward;
//  - NVFP4 scales are first multiplied by the expert's fp32 global scale and
//    the product rounded back to e4m3, after which the global scale is 1
//    (same section), so the GEMMs run with alpha = 1.
#include "internal.h"
#include "quant.cuh"

namespace moe {

namespace {

// Source row of destination row n within one expert's [N, .] matrix.
__device__ __forceinline__ int64_t source_row(int64_t n, int interleave_half) {
  if (!interleave_half) return n;
  const int64_t grp = n >> 7, r = n & 127;
  return r < 64 ? grp * 64 + r : interleave_half + grp * 64 + (r - 64);
}

// One thread per 16-byte chunk of destination codes.
__global__ void tile_codes_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ tiles,
                                  int64_t total_chunks, int N, int row_bytes, int tile_bytes,
                                  int interleave_half) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= total_chunks) return;
  const int chunks_per_row = row_bytes / 16;
  const int c16 = static_cast<int>(i % chunks_per_row);
  const int64_t row = i / chunks_per_row;          // destination row, e*N + n
  const int64_t e = row / N, n = row % N;
  const int64_t srow = e * N + source_row(n, interleave_half);
  const int nkb = row_bytes / 128;
  const int64_t tile = (e * (N / 128) + n / 128) * nkb + c16 / 8;
  const int r = static_cast<int>(n & 127), cc = c16 & 7;
  const uint4 v = reinterpret_cast<const uint4*>(src + srow * row_bytes)[c16];
  *reinterpret_cast<uint4*>(tiles + tile * tile_bytes + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
}

// One thread per (destination row, scale index): folds the NVFP4 global
// scale in (gs != nullptr) and stores the scale in its tile's scale block.
__global__ void tile_scales_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ tiles,
                                   int E, int N, int nkg, int sf_tiles, int tile_bytes,
                                   const float* __restrict__ gs, int interleave_half) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(E) * N * nkg;
  if (i >= total) return;
  const int kg = static_cast<int>(i % nkg);
  const int64_t row = i / nkg;
  const int64_t e = row / N, n = row % N;
  uint8_t v = src[(e * N + source_row(n, interleave_half)) * nkg + kg];
  if (gs) v = float_to_e4m3(__fmul_rn(e4m3_to_float(v), gs[e]));
  const int per_stage = 4 * sf_tiles;              // scale groups per 128-byte slice
  const int nkb = nkg / per_stage;
  const int64_t tile = (e * (N / 128) + n / 128) * nkb + kg / per_stage;
  const int j = (kg / 4) % sf_tiles;
  const int r = static_cast<int>(n & 127);
  tiles[tile * tile_bytes + 128 * 128 + j * 512 + (r & 31) * 16 + (r >> 5) * 4 + (kg & 3)] = v;
}

}  // namespace

cudaError_t launch_tile_weights(int fmt, const uint8_t* codes, const uint8_t* sf, const float* gs,
                                uint8_t* tiles, int E, int N, int row_bytes, int nkg,
                                int interleave_half, cudaStream_t s) {
  const int tb = weight_tile_bytes(fmt);
  const int64_t chunks = static_cast<int64_t>(E) * N * (row_bytes / 16);
  tile_codes_kernel<<<static_cast<unsigned>((chunks + 255) / 256), 256, 0, s>>>(
      codes, tiles, chunks, N, row_bytes, tb, interleave_half);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess || fmt == kFmtBF16) return e;
  const int64_t total = static_cast<int64_t>(E) * N * nkg;
  tile_scales_kernel<<<static_cast<unsigned>((total + 255) / 256), 256, 0, s>>>(
      sf, tiles, E, N, nkg, weight_sf_tiles(fmt), tb, fmt == kFmtNVFP4 ? gs : nullptr,
      interleave_half);
  return cudaGetLastError();
}

}  // namespace moe
