// gemm_common.cuh -- pieces shared by the grouped-GEMM kernels (the
// single-CTA kernel in gemm.cu and the CTA-pair NVFP4 kernel in
// gemm_pair.cu): tile constants, the per-expert work tables in shared
// memory, register budgets and the epilogues (GEMM1 + SwiGLU with the
// optional clamp or the squared ReLU, re-quantised into GEMM2's input
// format; GEMM2's bf16 store or in-kernel reduce).
#pragma once

#include <cuda_bf16.h>

#include "internal.h"
#include "ptx.cuh"
#include "quant.cuh"

namespace moe {

namespace {

constexpr int kTileBytes = 128 * 128;  // 128 rows x 128 bytes of K
constexpr int kSfColBase = 256;        // TMEM columns for scale tiles
constexpr int kTmemCols = 512;

// NW = weight tiles (of 128 rows) per work item, i.e. the MMA's N / 128.
// NW = 1: two 128-column accumulators (the epilogue of one item overlaps
// the main loop of the next) and 32 scale columns per stage.  NW = 2 (wide
// items, N = 256: half the shared-memory traffic per FLOP for the
// activation operand): one 256-column accumulator and 64 scale columns per
// stage (MXFP8: weight tiles at 0 and 4, activation at 8; NVFP4 copied by
// the MMA thread: activation tile j at 16 j, weight tiles j at 16 j + 8 and
// 16 j + 12; NVFP4 written by the scale-stager warps: weight tiles j at 8 j
// and 8 j + 4, activation rows of lane quarter q at column 32 + 4 j + q).
template <int NW>
struct Wide {
  static constexpr int kAccCols = 128 * NW;       // TMEM columns per accumulator
  static constexpr int kBufs = NW == 1 ? 2 : 1;   // accumulators
  static constexpr int kSfCols = 32 * NW;         // scale columns per stage
  static constexpr int kMaxStages = (kTmemCols - kSfColBase) / kSfCols;
};

template <int FMT>
struct Fmt;
template <>
struct Fmt<kFmtBF16> {
  static constexpr int kSfTiles = 0;  // scale tiles per operand per stage
};
template <>
struct Fmt<kFmtMXFP8> {
  static constexpr int kSfTiles = 1;  // 128 K elements = 4 x 32-blocks
};
template <>
struct Fmt<kFmtNVFP4> {
  static constexpr int kSfTiles = 4;  // 256 K elements = 16 x 16-blocks
};

// Per-expert item tables kept in shared memory: chunk_off[E+1],
// pad_off[E], counts[E] and the expert order order[E+1].
constexpr int kTableInts = 4 * (kMaxExperts + 1);
constexpr int kSmemLimit = 232448;  // opt-in maximum per block

// A stage holds the activation tile (MROWS rows x 128 bytes), the NW weight
// tiles' codes (NW x 128 rows x 128 bytes, consecutive so they form one
// 128*NW-row MMA operand), the weight tiles' scale tiles and the activation
// scale tiles.  MROWS is an upper bound on the real rows of any chunk of
// the launch (rows per expert never exceed T), so decode launches keep a
// short activation region and fit more stages.
// Rounded up to 1 KiB: the operand tiles at the start of every stage must
// sit on 128-byte-swizzle atom boundaries.
template <int FMT, int MROWS, int NW>
__host__ __device__ constexpr int stage_bytes() {
  return (MROWS * 128 + NW * kTileBytes + (NW + 1) * Fmt<FMT>::kSfTiles * 512 + 1023) / 1024 *
         1024;
}

// Stages: as many as shared memory holds, at most as many as TMEM has scale
// columns for.
template <int FMT, int MROWS, int NW>
__host__ __device__ constexpr int num_stages() {
  return (kSmemLimit - 1024 - kTableInts * 4 - 256) / stage_bytes<FMT, MROWS, NW>() >
                 Wide<NW>::kMaxStages
             ? Wide<NW>::kMaxStages
             : (kSmemLimit - 1024 - kTableInts * 4 - 256) / stage_bytes<FMT, MROWS, NW>();
}

template <int FMT, int MROWS, int NW>
__host__ __device__ constexpr int smem_bytes() {
  return 1024 + num_stages<FMT, MROWS, NW>() * stage_bytes<FMT, MROWS, NW>() +
         (3 * num_stages<FMT, MROWS, NW>() + 5) * 8 + 16 + kTableInts * 4;
}

constexpr int kEpiRegs = 176;
constexpr int kLeanRegs = 80;
// registers per thread the 512-thread block must be launched with for the
// split to balance: 2 x 128 threads give up (R - 80), 256 claim (176 - R)
constexpr int kSplitLaunchRegs = (2 * kLeanRegs + 2 * kEpiRegs) / 4;
static_assert(kSplitLaunchRegs * 512 <= 65536, "register split exceeds the register file");

struct Item {
  int e;       // expert (its weight tiles)
  int k;       // its position in the tables
  int n_tile, prow0, rows;
};

// Work item -> (expert, weight tile, chunk).  Items are numbered in table
// order: the expert at table position k owns items [chunk_off[k] * n_tiles,
// chunk_off[k+1] * n_tiles), weight tile major, chunk minor, so that the
// CTAs working at the same time share a weight tile through L2.  Without
// an order table, position k is expert k.  With one (wide launches), the
// experts with several chunks come first (in expert order), then those with
// one chunk at most, and the single-chunk experts' items are spread evenly
// among the others (below).  The tables live in shared memory (loaded once
// per CTA).
struct Tables {
  const int* chunk_off;  // [E+1]
  const int* pad_off;    // [E]
  const int* counts;     // [E]
  const int* order;      // [E+1]: expert at each position, then the chunks of
                         // the multi-chunk positions; nullptr: the identity
};

// A single-chunk expert's weight tiles are read from DRAM once, by one item
// each, while a multi-chunk expert's tiles are read once and then served
// from L2 to its other chunks.  In plain table order the CTAs meet long runs
// of single-chunk items (DRAM-bound, the tensor pipes idle) and long runs of
// multi-chunk items (the reverse).  Mixed in at an even rate (item i is the
// c-th single-chunk item when floor((i+1) nc / n) > c = floor(i nc / n)),
// the weight streams overlap the tensor work.  A bijection on [0, n).
// floor(a b / n) for 0 <= a, b <= n, without an integer divide: a float
// estimate (within one of the result for n below 2^20), then corrected.
__device__ __forceinline__ int floor_mul_div(int a, int b, int n) {
  int q = static_cast<int>(__fdividef(static_cast<float>(a) * static_cast<float>(b),
                                      static_cast<float>(n)));
  const int64_t p = static_cast<int64_t>(a) * b;
  while (q > 0 && static_cast<int64_t>(q) * n > p) --q;
  while (static_cast<int64_t>(q + 1) * n <= p) ++q;
  return q;
}

__device__ __forceinline__ int mix_item(const Tables& t, int E, int n_tiles, int item) {
  if (t.order == nullptr) return item;
  const int n = t.chunk_off[E] * n_tiles;
  const int nh = t.order[E] * n_tiles;
  const int nc = n - nh;
  if (nc <= 0 || nh <= 0) return item;
  const int c0 = floor_mul_div(item, nc, n), c1 = floor_mul_div(item + 1, nc, n);
  return c1 > c0 ? nh + c0 : item - c0;
}

// kOrdered: the kernel may be given an order table (the wide kernels); the
// narrow ones map by expert and carry none of it (a few registers more in
// every narrow GEMM measured 3 % on the stream-launched bf16 T = 512 layer).
template <bool kOrdered>
__device__ __forceinline__ Item map_item(const Tables& t, int E, int n_tiles, int item) {
  const int g = kOrdered ? mix_item(t, E, n_tiles, item) : item;
  int lo = 0, hi = E;  // chunk_off[lo]*nt <= g < chunk_off[hi]*nt
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (t.chunk_off[mid] * n_tiles <= g) lo = mid; else hi = mid;
  }
  const int c0 = t.chunk_off[lo];
  const int nch = t.chunk_off[lo + 1] - c0;
  const int local = g - c0 * n_tiles;
  const int chunk = local % nch;
  Item it;
  it.e = kOrdered && t.order ? t.order[lo] : lo;
  it.k = lo;
  it.n_tile = local / nch;
  it.prow0 = t.pad_off[lo] + chunk * kRowBlock;
  it.rows = min(kRowBlock, t.counts[lo] - chunk * kRowBlock);
  return it;
}

// Accumulator rows past the chunk's real rows come from stale shared memory
// and may hold NaNs or denormals, which would send the division and exp
// below down their slow paths; their results are never stored, so those
// lanes work on zeros instead.
__device__ __forceinline__ float lane_value(uint32_t bits, bool valid) {
  return valid ? __uint_as_float(bits) : 0.0f;
}

// silu(g) * u with the optional clamp.  Uses the hardware exp2 and
// reciprocal approximations (__expf, __fdividef; a few ulp): the accurate
// expf and IEEE division cost several microseconds per 16 features on the
// one warp that holds a decode chunk, longer than a whole GEMM item.  For
// g < -88, exp(-g) overflows to inf and the quotient is 0, as it should be.
__device__ __forceinline__ float silu_mul(float g, float u, float L) {
  g = fminf(fmaxf(g, -L), L);
  u = fminf(fmaxf(u, -L), L);
  return __fdividef(g, 1.0f + __expf(-g)) * u;
}

// ---------------------------------------------------------------- epilogues
// An epilogue covers one 128-column accumulator group in two rounds of 64
// columns.  Narrow items (two accumulators) load each round just before
// computing it; wide items load both rounds first and release their single
// accumulator before computing, so the next item's MMAs can start.
//
// Columns of round p: GEMM1 + SwiGLU reads gate and up of 32 features
// (gate 32p.., up 64+32p..); the other epilogues read columns 64p.. .
template <int EPI>
__device__ __forceinline__ void epilogue_load(uint32_t taddr, int p, uint32_t* v) {
  const int c0 = EPI == 1 ? 32 * p : 64 * p;
  const int c2 = EPI == 1 ? 64 + 32 * p : 64 * p + 32;
  tmem_ld16(taddr + c0, *reinterpret_cast<uint32_t(*)[16]>(v));
  tmem_ld16(taddr + c0 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 16));
  tmem_ld16(taddr + c2, *reinterpret_cast<uint32_t(*)[16]>(v + 32));
  tmem_ld16(taddr + c2 + 16, *reinterpret_cast<uint32_t(*)[16]>(v + 48));
}

__device__ __forceinline__ void epilogue_fence(uint32_t* v) {
#pragma unroll
  for (int i = 0; i < 4; ++i) reg_fence16(*reinterpret_cast<uint32_t(*)[16]>(v + 16 * i));
}

__device__ __forceinline__ uint32_t pack_bf16x2(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t*>(&v);
}

// 16 bf16 values (32 bytes) to dst.
// Each epilogue thread owns one row, so the lanes of a warp store to 32
// different rows: whole 32-byte sectors per store (dst 32-byte aligned; all
// GEMM1 outputs are layer buffers with 32-byte aligned rows) halve the
// requests and L2 sector writes of 16-byte stores.
__device__ __forceinline__ void store32(uint8_t* dst, const uint32_t* w) {
  st_global_v8(dst, w[0], w[1], w[2], w[3], w[4], w[5], w[6], w[7]);
}

__device__ __forceinline__ void store_bf16x16(uint8_t* dst, const float* h) {
  uint32_t o[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) o[i] = pack_bf16x2(h[2 * i], h[2 * i + 1]);
  store32(dst, o);
}

// GEMM1 + SwiGLU, round p: thread = accumulator row (token row `prow`);
// v[0..31] gate and v[32..63] up of intermediate features 64*n_tile + 32p + j.
// NVFP4: round 0 leaves its 16 code bytes and 2 scale bytes in `carry`, and
// round 1 stores both rounds' codes (32 bytes) and scales (4 bytes, adjacent
// in the scale tile) at once.
template <int FMT>
__device__ __forceinline__ void epilogue_gemm1(const uint32_t* v, int p, bool store, int64_t prow,
                                               int n_tile, const GemmArgs& a,
                                               uint32_t (&carry)[5]) {
  float h[32];
#pragma unroll
  for (int i = 0; i < 32; ++i)
    h[i] = silu_mul(lane_value(v[i], store), lane_value(v[32 + i], store), a.clamp);
  if constexpr (FMT == kFmtNVFP4) {
    uint32_t c[4];
    uint8_t sf0, sf1;
    quant_nvfp4_16(h, *reinterpret_cast<uint32_t(*)[2]>(&c[0]), sf0);
    quant_nvfp4_16(h + 16, *reinterpret_cast<uint32_t(*)[2]>(&c[2]), sf1);
    if (p == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) carry[i] = c[i];
      carry[4] = static_cast<uint32_t>(sf0) | (static_cast<uint32_t>(sf1) << 8);
    } else if (store) {
      st_global_v8(a.out + prow * a.out_ld + n_tile * 32, carry[0], carry[1], carry[2], carry[3],
                   c[0], c[1], c[2], c[3]);
      st_global_b32_ef(a.out_sf + sf_tile_offset(prow, n_tile * 4, a.out_sf_tiles_k),
                       carry[4] | (static_cast<uint32_t>(sf0) << 16) |
                           (static_cast<uint32_t>(sf1) << 24));
    }
  } else if constexpr (FMT == kFmtMXFP8) {
    uint32_t c[8];
    uint8_t sf;
    quant_mxfp8_32(h, c, sf);
    if (store) {
      store32(a.out + prow * a.out_ld + n_tile * 64 + p * 32, c);
      st_global_b8_ef(a.out_sf + sf_tile_offset(prow, n_tile * 2 + p, a.out_sf_tiles_k), sf);
    }
  } else {
    if (store) {
      uint8_t* dst = a.out + prow * a.out_ld + (n_tile * 64 + p * 32) * 2;
      store_bf16x16(dst, h);
      store_bf16x16(dst + 32, h + 16);
    }
  }
}

// GEMM1 with the non-gated squared ReLU, round p: v holds intermediate
// features 128*n_tile + 64p + j; h = max(x, 0)^2 (one correctly rounded fp32
// product), then the same re-quantisation per 16- (NVFP4) or 32- (MXFP8)
// block, or a bf16 round.
__device__ __forceinline__ float relu_sq(float x) {
  x = fmaxf(x, 0.0f);
  return __fmul_rn(x, x);
}

template <int FMT>
__device__ __forceinline__ void epilogue_relu2(const uint32_t* v, int p, bool store, int64_t prow,
                                               int n_tile, const GemmArgs& a) {
  float h[64];
#pragma unroll
  for (int i = 0; i < 64; ++i) h[i] = relu_sq(lane_value(v[i], store));
  if constexpr (FMT == kFmtNVFP4) {
    uint32_t c[8];
    uint32_t sf4 = 0;
#pragma unroll
    for (int jb = 0; jb < 4; ++jb) {
      uint8_t sf;
      quant_nvfp4_16(h + 16 * jb, *reinterpret_cast<uint32_t(*)[2]>(&c[2 * jb]), sf);
      sf4 |= static_cast<uint32_t>(sf) << (8 * jb);
    }
    if (store) {
      store32(a.out + prow * a.out_ld + n_tile * 64 + p * 32, c);
      st_global_b32_ef(a.out_sf + sf_tile_offset(prow, n_tile * 8 + p * 4, a.out_sf_tiles_k), sf4);
    }
  } else if constexpr (FMT == kFmtMXFP8) {
#pragma unroll
    for (int jb = 0; jb < 2; ++jb) {
      uint32_t c[8];
      uint8_t sf;
      quant_mxfp8_32(h + 32 * jb, c, sf);
      if (store) {
        store32(a.out + prow * a.out_ld + n_tile * 128 + p * 64 + jb * 32, c);
        st_global_b8_ef(a.out_sf + sf_tile_offset(prow, n_tile * 4 + p * 2 + jb, a.out_sf_tiles_k),
                        sf);
      }
    }
  } else {
    if (store) {
      uint8_t* dst = a.out + prow * a.out_ld + (n_tile * 128 + p * 64) * 2;
#pragma unroll
      for (int q = 0; q < 4; ++q) store_bf16x16(dst + 32 * q, h + 16 * q);
    }
  }
}

// GEMM2, round p: output features 128*n_tile + 64p + j, stored as bf16.
__device__ __forceinline__ void epilogue_gemm2(const uint32_t* v, int p, bool store, int64_t prow,
                                               int n_tile, const GemmArgs& a) {
  if (!store) return;
  uint8_t* row = a.out + prow * a.out_ld + n_tile * 256 + p * 128;
  if (((reinterpret_cast<uintptr_t>(a.out) | static_cast<uintptr_t>(a.out_ld)) & 31) == 0) {
    // each thread owns one row: whole 32-byte sectors halve the store
    // requests and the L2 sector writes of 16-byte stores
#pragma unroll
    for (int q = 0; q < 4; ++q) {
      const uint32_t* w = v + 16 * q;
      st_global_v8(row + 32 * q, pack_bf16x2(__uint_as_float(w[0]), __uint_as_float(w[1])),
                   pack_bf16x2(__uint_as_float(w[2]), __uint_as_float(w[3])),
                   pack_bf16x2(__uint_as_float(w[4]), __uint_as_float(w[5])),
                   pack_bf16x2(__uint_as_float(w[6]), __uint_as_float(w[7])),
                   pack_bf16x2(__uint_as_float(w[8]), __uint_as_float(w[9])),
                   pack_bf16x2(__uint_as_float(w[10]), __uint_as_float(w[11])),
                   pack_bf16x2(__uint_as_float(w[12]), __uint_as_float(w[13])),
                   pack_bf16x2(__uint_as_float(w[14]), __uint_as_float(w[15])));
    }
    return;
  }
  uint4* dst = reinterpret_cast<uint4*>(row);
#pragma unroll
  for (int q = 0; q < 8; ++q)
    dst[q] = make_uint4(pack_bf16x2(__uint_as_float(v[8 * q]), __uint_as_float(v[8 * q + 1])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                        pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
}

// GEMM2 with the in-kernel reduce, round p: adds w * y (fp32) of this row's
// 64 output features into the token's fp32 accumulator (vector atomics).
__device__ __forceinline__ void epilogue_reduce(const uint32_t* v, int p, int64_t t, float wt,
                                                int n_tile, const GemmArgs& a) {
  float4* dst = reinterpret_cast<float4*>(a.acc + t * a.H + n_tile * 128 + p * 64);
#pragma unroll
  for (int q = 0; q < 16; ++q)
    atomicAdd(dst + q, make_float4(__fmul_rn(wt, __uint_as_float(v[4 * q])),
                                   __fmul_rn(wt, __uint_as_float(v[4 * q + 1])),
                                   __fmul_rn(wt, __uint_as_float(v[4 * q + 2])),
                                   __fmul_rn(wt, __uint_as_float(v[4 * q + 3]))));
}

// After both rounds: count this contribution to the token's 128-column
// group; the K-th contributor writes the group as bf16 and leaves the
// accumulator and its counter at zero for the next forward.
__device__ __forceinline__ void reduce_finish(int64_t t, int n_tile, const GemmArgs& a) {
  __threadfence();
  int32_t* cnt = a.acc_cnt + t * (a.H / 128) + n_tile;
  if (atomicAdd(cnt, 1) != a.K - 1) return;
  __threadfence();
  float4* acc = reinterpret_cast<float4*>(a.acc + t * a.H + n_tile * 128);
  uint4* out = reinterpret_cast<uint4*>(a.comb_out + (t * a.H + n_tile * 128) * 2);
#pragma unroll 4
  for (int q = 0; q < 16; ++q) {
    const float4 x = __ldcg(acc + 2 * q), y = __ldcg(acc + 2 * q + 1);
    out[q] = make_uint4(pack_bf16x2(x.x, x.y), pack_bf16x2(x.z, x.w), pack_bf16x2(y.x, y.y),
                        pack_bf16x2(y.z, y.w));
    __stcg(acc + 2 * q, make_float4(0.f, 0.f, 0.f, 0.f));
    __stcg(acc + 2 * q + 1, make_float4(0.f, 0.f, 0.f, 0.f));
  }
  *cnt = 0;
}

// GEMM2 with the fused combine (a.gather_inv != nullptr), after the warp's
// rows of a 128-column group have been stored: each stored row counts itself
// for its token's group; for every token whose K-th row this warp stored,
// the whole warp sums that token's K rows of the group in k order in fp32
// (the combine kernel's operations, so the output is bit-identical), writes
// the bf16 result and resets the counter for the next forward.  Called by
// all 32 lanes of the warp; `stored`: this lane's row was stored.
__device__ __forceinline__ void combine_fused(bool stored, int64_t prow, int n_tile,
                                              const GemmArgs& a) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  const int lane = threadIdx.x & 31;
  __threadfence();  // this lane's row is visible before it is counted
  int t = 0;
  bool last = false;
  if (stored) {
    t = a.prow_slot[prow] / a.K;
    last = atomicAdd(a.acc_cnt + static_cast<int64_t>(t) * (a.H / 128) + n_tile, 1) == a.K - 1;
  }
  unsigned todo = __ballot_sync(kAll, last);
  if (!todo) return;
  __threadfence();  // the token's other rows, counted before, are visible
  while (todo) {
    const int src = __ffs(todo) - 1;
    todo &= todo - 1;
    const int64_t tt = __shfl_sync(kAll, t, src);
    // lane l: columns 4l .. 4l+3 of the group
    uint2 u[kMaxTopK];
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
      if (k < a.K) {
        const int64_t row = a.gather_inv[tt * a.K + k];
        u[k] = __ldcg(reinterpret_cast<const uint2*>(a.out + row * a.out_ld + n_tile * 256) + lane);
      }
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int k = 0; k < kMaxTopK; ++k)
      if (k < a.K) {
        const float wk = a.topk_w[tt * a.K + k];
        const float2 p0 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k].x));
        const float2 p1 = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u[k].y));
        acc[0] = fmaf(wk, p0.x, acc[0]);
        acc[1] = fmaf(wk, p0.y, acc[1]);
        acc[2] = fmaf(wk, p1.x, acc[2]);
        acc[3] = fmaf(wk, p1.y, acc[3]);
      }
    reinterpret_cast<uint2*>(a.comb_out + (tt * a.H + n_tile * 128) * 2)[lane] =
        make_uint2(pack_bf16x2(acc[0], acc[1]), pack_bf16x2(acc[2], acc[3]));
    if (lane == src) a.acc_cnt[tt * (a.H / 128) + n_tile] = 0;
  }
}

template <int FMT, int EPI>
__device__ __forceinline__ void epilogue_round(const uint32_t* v, int p, bool store, int64_t prow,
                                               int64_t orow, int n_tile, const GemmArgs& a,
                                               uint32_t (&carry)[5]) {
  if constexpr (EPI == 1) {
    epilogue_gemm1<FMT>(v, p, store, prow, n_tile, a, carry);
  } else if constexpr (EPI == 3) {
    epilogue_relu2<FMT>(v, p, store, prow, n_tile, a);
  } else if (a.acc) {
    if (store) {
      const int slot = a.prow_slot[prow];
      epilogue_reduce(v, p, slot / a.K, a.topk_w[slot], n_tile, a);
      if (p == 1) reduce_finish(slot / a.K, n_tile, a);
    }
  } else {
    epilogue_gemm2(v, p, store, orow, n_tile, a);
  }
}

}  // namespace

}  // namespace moe
