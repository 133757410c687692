// prep.cu -- one-time weight preparation (untimed set-up).
//
// The canonical quantised weights are copied into the layer's own buffers
// and re-laid out for the grouped GEMMs:
//  - W13 rows are interleaved in 64-row groups (64 gate rows, then the 64
//    matching up rows, ...), so one 128-row weight tile holds the gate and up
//    halves of the same 64 intermediate features and the GEMM1 epilogue sees
//    both in one accumulator row;
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

// One warp per destination row, 16-byte copies.
__global__ void copy_rows_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst,
                                 int64_t rows, int64_t row_bytes, int N, int interleave_half) {
  const int64_t row = static_cast<int64_t>(blockIdx.x) * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (row >= rows) return;
  const int64_t e = row / N, n = row % N;
  const int64_t srow = e * N + source_row(n, interleave_half);
  const uint4* s = reinterpret_cast<const uint4*>(src + srow * row_bytes);
  uint4* d = reinterpret_cast<uint4*>(dst + row * row_bytes);
  for (int64_t c = threadIdx.x & 31; c < row_bytes / 16; c += 32) d[c] = s[c];
}

// One thread per (destination row, scale index).
__global__ void sf_tiles_kernel(const uint8_t* __restrict__ src, uint8_t* __restrict__ dst, int E,
                                int N, int nkg, const float* __restrict__ gs,
                                int interleave_half) {
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  const int64_t total = static_cast<int64_t>(E) * N * nkg;
  if (i >= total) return;
  const int kg = static_cast<int>(i % nkg);
  const int64_t row = i / nkg;
  const int64_t e = row / N, n = row % N;
  uint8_t v = src[(e * N + source_row(n, interleave_half)) * nkg + kg];
  if (gs) v = float_to_e4m3(__fmul_rn(e4m3_to_float(v), gs[e]));
  dst[sf_tile_offset(row, kg, nkg / 4)] = v;
}

}  // namespace

cudaError_t launch_copy_rows(const uint8_t* src, uint8_t* dst, int64_t rows, int64_t row_bytes,
                             int N, int interleave_half, cudaStream_t s) {
  const int warps = 8;
  const int64_t blocks = (rows + warps - 1) / warps;
  copy_rows_kernel<<<static_cast<unsigned>(blocks), warps * 32, 0, s>>>(src, dst, rows, row_bytes,
                                                                         N, interleave_half);
  return cudaGetLastError();
}

cudaError_t launch_sf_tiles(const uint8_t* src, uint8_t* dst, int E, int N, int nkg,
                            const float* gs, int interleave_half, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(E) * N * nkg;
  const int64_t blocks = (total + 255) / 256;
  sf_tiles_kernel<<<static_cast<unsigned>(blocks), 256, 0, s>>>(src, dst, E, N, nkg, gs,
                                                                 interleave_half);
  return cudaGetLastError();
}

}  // namespace moe
