// rowquant.cuh -- the GEMM1 input of token rows: BF16 copied, MXFP8 / NVFP4
// quantised per block (quant.cuh) into the rows' padded positions, codes
// row-major and scales in the MMA's 128-row scale tiles.  Shared by the
// routing/scatter kernels and the single-launch decode kernel.
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "quant.cuh"

namespace moe {

namespace {

// ---------------------------------------------------------------- row quantisation
// Units of one token row's GEMM1 input: 16-byte chunks (BF16, copied) or
// quantisation blocks of 16 (NVFP4) / 32 (MXFP8) elements.
template <int FMT>
__host__ __device__ constexpr int row_units(int H) {
  return FMT == kFmtBF16 ? H / 8 : FMT == kFmtNVFP4 ? H / 16 : H / 32;
}

// Unit `u` of token row x [H] into the padded rows prows[0..n): BF16 copied,
// MXFP8 / NVFP4 quantised, codes row-major and scales in the MMA's 128-row
// scale tiles.
// A unit's bf16 source: 16 (BF16 copy), 32 (NVFP4) or 64 (MXFP8) bytes.
template <int FMT>
struct RawUnit {
  static constexpr int kVecs = FMT == kFmtBF16 ? 1 : FMT == kFmtNVFP4 ? 2 : 4;
  uint4 v[kVecs];
};

template <int FMT>
__device__ __forceinline__ void load_unit(const __nv_bfloat16* __restrict__ x, int u,
                                          RawUnit<FMT>& r) {
  const uint4* src =
      reinterpret_cast<const uint4*>(x) + static_cast<int64_t>(u) * RawUnit<FMT>::kVecs;
#pragma unroll
  for (int i = 0; i < RawUnit<FMT>::kVecs; ++i) r.v[i] = src[i];
}

template <int N>
__device__ __forceinline__ void unpack_bf16(const uint4* src, float (&f)[N]) {
#pragma unroll
  for (int h = 0; h < N / 8; ++h) {
    const uint32_t wv[4] = {src[h].x, src[h].y, src[h].z, src[h].w};
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const float2 v = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]));
      f[8 * h + 2 * q] = v.x;
      f[8 * h + 2 * q + 1] = v.y;
    }
  }
}

// Where one padded row's GEMM1 input goes: the byte offset of its codes and
// the unit-independent part of its scale bytes' offset in the scale tiles
// (sf_tile_offset(prow, u, tiles_k) is that part plus (u / 4) * 512 + u % 4).
struct RowDst {
  int64_t code;
  int64_t sf;
};

template <int FMT>
__device__ __forceinline__ RowDst row_dst(int prow, int H) {
  const int64_t p = prow;
  if constexpr (FMT == kFmtBF16) return RowDst{p * H * 2, 0};
  else if constexpr (FMT == kFmtNVFP4) return RowDst{p * (H / 2), sf_tile_offset(p, 0, H / 64)};
  else return RowDst{p * H, sf_tile_offset(p, 0, H / 128)};
}

// Destinations given as padded row numbers.
struct PaddedRows {
  const int* prows;
  int H;
  template <int FMT>
  __device__ __forceinline__ RowDst get(int k) const {
    return row_dst<FMT>(prows[k], H);
  }
};

// Destinations precomputed once per row (row_dst).
struct RowDsts {
  const RowDst* d;
  template <int FMT>
  __device__ __forceinline__ RowDst get(int k) const {
    return d[k];
  }
};

// Unit `u` of a token row, already loaded, into the n padded rows `dst`
// names: BF16 copied, MXFP8 / NVFP4 quantised, codes row-major and scales in
// the MMA's 128-row scale tiles.
template <int FMT, class Dst>
__device__ __forceinline__ void store_unit_rows(const RawUnit<FMT>& r, int u, const Dst& dst,
                                                int n, uint8_t* __restrict__ xq,
                                                uint8_t* __restrict__ xsf) {
  if constexpr (FMT == kFmtBF16) {
    for (int k = 0; k < n; ++k)
      reinterpret_cast<uint4*>(xq + dst.template get<FMT>(k).code)[u] = r.v[0];
  } else {
    constexpr int kUnitBytes = FMT == kFmtNVFP4 ? 8 : 32;
    const int64_t cu = static_cast<int64_t>(u) * kUnitBytes;
    const int su = (u >> 2) * 512 + (u & 3);
    if constexpr (FMT == kFmtNVFP4) {
      float f[16];
      unpack_bf16<16>(r.v, f);
      uint32_t codes[2];
      uint8_t sf;
      quant_nvfp4_16(f, codes, sf);
      for (int k = 0; k < n; ++k) {
        const RowDst d = dst.template get<FMT>(k);
        *reinterpret_cast<uint2*>(xq + d.code + cu) = make_uint2(codes[0], codes[1]);
        xsf[d.sf + su] = sf;
      }
    } else {
      float f[32];
      unpack_bf16<32>(r.v, f);
      uint32_t codes[8];
      uint8_t sf;
      quant_mxfp8_32(f, codes, sf);
      for (int k = 0; k < n; ++k) {
        const RowDst d = dst.template get<FMT>(k);
        uint4* out = reinterpret_cast<uint4*>(xq + d.code + cu);
        out[0] = make_uint4(codes[0], codes[1], codes[2], codes[3]);
        out[1] = make_uint4(codes[4], codes[5], codes[6], codes[7]);
        xsf[d.sf + su] = sf;
      }
    }
  }
}

template <int FMT>
__device__ __forceinline__ void quant_unit_to_rows(const __nv_bfloat16* __restrict__ x, int H,
                                                   int u, const int* prows, int n,
                                                   uint8_t* __restrict__ xq,
                                                   uint8_t* __restrict__ xsf) {
  RawUnit<FMT> r;
  load_unit<FMT>(x, u, r);
  store_unit_rows<FMT>(r, u, PaddedRows{prows, H}, n, xq, xsf);
}

// Writes the GEMM1 input of one token row into its padded rows: this thread
// takes units first, first + stride, ... (one warp: first = lane, stride
// 32).  The next unit's load is issued before the current one is quantised
// and stored, so each thread keeps two loads in flight instead of waiting out
// the latency of every one.  loaded: unit `first`, already loaded by the
// caller (or null).
template <int FMT, class Dst>
__device__ __forceinline__ void quant_row_to_rows(const __nv_bfloat16* __restrict__ x, int H,
                                                  const Dst& dst, int n,
                                                  uint8_t* __restrict__ xq,
                                                  uint8_t* __restrict__ xsf, int first,
                                                  int stride = 32,
                                                  const RawUnit<FMT>* loaded = nullptr) {
  const int U = row_units<FMT>(H);
  if (first >= U) return;
  RawUnit<FMT> cur;
  if (loaded) cur = *loaded;
  else load_unit<FMT>(x, first, cur);
  for (int u = first; u < U; u += stride) {
    RawUnit<FMT> nxt;
    const bool more = u + stride < U;
    if (more) load_unit<FMT>(x, u + stride, nxt);
    store_unit_rows<FMT>(cur, u, dst, n, xq, xsf);
    if (more) cur = nxt;
  }
}

}  // namespace

}  // namespace moe
