// route.cu -- routing, histogram / scan / scatter permutation with the GEMM1
// activation quantisation fused into the scatter, the combine, and the
// inspection kernels.
//
// Routing (top-k of the router logits, softmax over the selected k) and the
// routing-weighted reduction back to token order are the first and last
// steps of the fused layer, which the b12x integration runs together with
// both expert GEMMs in one call (PR #40082 report, sec. 实现拆解 item 1).  The
// permutation is the single-GPU form of token dispatch: slots (t, k) are grouped by
// expert with a stable counting sort (histogram per block of 8 tokens, an
// exclusive scan over the blocks per expert, a scatter), and each expert's segment
// is padded to a multiple of 128 rows so every 128-row GEMM tile and its
// scale tiles start on a tile boundary.
#include <cuda_bf16.h>

#include <cfloat>
#include <climits>

#include "internal.h"
#include "quant.cuh"
#include "route_token.cuh"
#include "rowquant.cuh"

namespace moe {

namespace {

constexpr unsigned kFull = 0xFFFFFFFFu;
// Experts with at least this many 128-row chunks form the GEMMs' main item
// stream; the single-chunk ones are mixed into it (store_mixed_tables).
constexpr int kMixMinChunks = 2;

// ---------------------------------------------------------------- routing
// One warp per token (route_token), 8 tokens per block.  Block b also counts
// how many of its slots go to each expert (blockhist[b][e]).
template <int MAXJ>
__global__ void __launch_bounds__(256) route_kernel(const float* __restrict__ logits, int T, int E,
                                                    int K, int32_t* __restrict__ ids,
                                                    float* __restrict__ w,
                                                    int32_t* __restrict__ blockhist) {
  pdl_launch_dependents();
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int t = blockIdx.x * kTokensPerRouteBlock + warp;
  int my_i = 0;
  float my_w = 0.0f;
  if (t < T) route_token<MAXJ>(logits + static_cast<int64_t>(t) * E, E, K, lane, &my_i, &my_w);
  // the previous forward's last kernels may still read ids / w / blockhist
  pdl_wait();
  if (t < T && lane < K) {
    ids[static_cast<int64_t>(t) * K + lane] = my_i;
    w[static_cast<int64_t>(t) * K + lane] = my_w;
    atomicAdd(&hist[my_i], 1);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    blockhist[static_cast<int64_t>(blockIdx.x) * E + e] = hist[e];
}

// ---------------------------------------------------------------- scan
// Exclusive scan of every expert's per-block counts over the routing blocks
// (prefix[b][e] = slots of expert e in blocks < b) and its total count.
// Few routing blocks: one warp per expert.
__global__ void __launch_bounds__(256) expert_scan_warp_kernel(const int32_t* __restrict__ blockhist,
                                                          int NB, int E,
                                                          int32_t* __restrict__ prefix,
                                                          int32_t* __restrict__ counts) {
  pdl_launch_dependents();
  pdl_wait();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 8 + warp;
  if (e >= E) return;
  const int per = (NB + 31) / 32;
  const int b0 = lane * per, b1 = min(NB, b0 + per);
  int sum = 0;
  for (int b = b0; b < b1; ++b) sum += blockhist[static_cast<int64_t>(b) * E + e];
  int inc = sum;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += o;
  }
  int run = inc - sum;
  for (int b = b0; b < b1; ++b) {
    const int64_t i = static_cast<int64_t>(b) * E + e;
    const int c = blockhist[i];
    prefix[i] = run;
    run += c;
  }
  if (lane == 31) counts[e] = inc;
}

// Many routing blocks (prefill):
__global__ void __launch_bounds__(1024) expert_scan_kernel(const int32_t* __restrict__ blockhist,
                                                           int NB, int E,
                                                           int32_t* __restrict__ prefix,
                                                           int32_t* __restrict__ counts) {
  // Block x covers experts 32x .. 32x+31 (lane = expert, so every read of a
  // routing block's histogram row is one coalesced 128-byte segment); its 32
  // warps split the routing blocks into 32 consecutive ranges.  Pass 1: each
  // warp sums its range; warp 0 scans the 32 partial sums of every expert;
  // pass 2: each warp writes the exclusive prefixes of its range.
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int part[32][33];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.x * 32 + lane;
  const int per = (NB + 31) / 32;
  const int b0 = min(NB, warp * per), b1 = min(NB, b0 + per);
  int sum = 0;
  if (e < E)
    for (int b = b0; b < b1; ++b) sum += blockhist[static_cast<int64_t>(b) * E + e];
  part[warp][lane] = sum;
  __syncthreads();
  if (warp == 0) {
    int run = 0;
    for (int w2 = 0; w2 < 32; ++w2) {
      const int v = part[w2][lane];
      part[w2][lane] = run;
      run += v;
    }
    if (e < E) counts[e] = run;
  }
  __syncthreads();
  int run = part[warp][lane];
  if (e < E)
    for (int b = b0; b < b1; ++b) {
      const int64_t i = static_cast<int64_t>(b) * E + e;
      const int c = blockhist[i];
      prefix[i] = run;
      run += c;
    }
}

// Block-wide exclusive scans of the row counts and the 128-row chunk counts
// of the thread's two experts, both in one pass: the pair is packed into one
// 64-bit value (row count high, chunk count low; every partial sum of either
// stays below 2^31, so the low half never carries).  wsum holds one value
// per warp of the block.  The padded-row offsets are kRowBlock times the
// chunk offsets, so they need no scan of their own.
__device__ __forceinline__ void block_scan_counts(int rows, int chunks, uint64_t* wsum,
                                                  int& xrows, int& xchunks) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const uint64_t v = (static_cast<uint64_t>(rows) << 32) | static_cast<uint32_t>(chunks);
  uint64_t inc = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const uint64_t o = __shfl_up_sync(kFull, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  uint64_t add = 0;
  for (int w2 = 0; w2 < warp; ++w2) add += wsum[w2];
  const uint64_t ex = inc - v + add;
  xrows = static_cast<int>(ex >> 32);
  xchunks = static_cast<int>(static_cast<uint32_t>(ex));
}

// The GEMMs' item tables in the mixed order (gemm_common.cuh, mix_item):
// the experts with at least two chunks first, then the others, each group in
// expert order.  otab = chunk_off[E+1], pad_off[E], counts[E] by table
// position, then order[E+1]: the expert at each position and the number of
// chunks of the multi-chunk group.  One block writes them; every thread
// holds experts 2t, 2t+1 (c = rows, p = chunks, xp = first padded row of
// expert 2t).
__device__ __forceinline__ void store_mixed_tables(int E, int c0, int c1, int p0, int p1, int xp,
                                                   uint64_t* wsum, int32_t* __restrict__ otab) {
  __shared__ int s_tot[2];
  const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
  const int h0 = p0 >= kMixMinChunks, h1 = p1 >= kMixMinChunks;
  int xhe, xhc, xle, xlc;  // exclusive: multi-chunk experts / their chunks, the rest
  __syncthreads();         // wsum is reused
  block_scan_counts(h0 + h1, h0 * p0 + h1 * p1, wsum, xhe, xhc);
  __syncthreads();
  block_scan_counts(2 - h0 - h1, (1 - h0) * p0 + (1 - h1) * p1, wsum, xle, xlc);
  if (e0 == E - 1 || e1 == E - 1) {
    // the last thread with experts: totals of the multi-chunk group (an
    // expert 2t+1 >= E has no chunks and does not count)
    const int h1v = e1 < E ? h1 : 0;
    s_tot[0] = xhe + h0 + h1v;
    s_tot[1] = xhc + h0 * p0 + h1v * p1;
  }
  __syncthreads();
  const int nhe = s_tot[0], nhc = s_tot[1];
  int32_t* o_chunk = otab;
  int32_t* o_pad = otab + (E + 1);
  int32_t* o_cnt = otab + (2 * E + 1);
  int32_t* o_ord = otab + (3 * E + 1);
  if (e0 < E) {
    const int k = h0 ? xhe : nhe + xle;
    o_chunk[k] = h0 ? xhc : nhc + xlc;
    o_pad[k] = xp;
    o_cnt[k] = c0;
    o_ord[k] = e0;
  }
  if (e1 < E) {
    const int k = h1 ? xhe + h0 : nhe + xle + (1 - h0);
    o_chunk[k] = h1 ? xhc + h0 * p0 : nhc + xlc + (1 - h0) * p0;
    o_pad[k] = xp + p0 * kRowBlock;
    o_cnt[k] = c1;
    o_ord[k] = e1;
  }
  if (threadIdx.x == 0) o_ord[E] = nhc;
  if (e0 == E - 1 || e1 == E - 1) o_chunk[E] = nhc + xlc + (1 - h0) * p0 + (1 - h1) * p1;
}

// ---------------------------------------------------------------- scatter
// Block b handles the 8 tokens of routing block b.
//  1. Exclusive scans of the per-expert counts, 128-padded counts and 128-row
//     chunk counts (every block computes them; block 0 stores them for the
//     GEMMs).
//  2. Each of the block's slots gets, in slot order, the next row of its
//     expert after the rows of earlier blocks (stable): perm[row] = slot,
//     inv[slot] = padded row.
//  3. W warps per token write token 8b+i's GEMM1 input into its K padded
//     rows (warp Wi + j takes every W-th 32-unit group from group j): BF16
//     copied, MXFP8 / NVFP4 quantised per block (one block per thread).
//     NVFP4 uses W = 2: halving each warp's serial chain of loads and
//     quantisations took the NVFP4 decode scatter (T = 128, 16 blocks) from
//     22.8 to 18.8 us.  For the BF16 copy, two warps per row made the bf16
//     layer 2 us slower, and MXFP8 would lose occupancy (112 registers).
template <int FMT>
__host__ __device__ constexpr int scatter_warps_per_token() {
  return FMT == kFmtNVFP4 ? 2 : 1;
}
template <int FMT>
__host__ __device__ constexpr int scatter_threads() {
  return 32 * kTokensPerRouteBlock * scatter_warps_per_token<FMT>();
}

template <int FMT>
__global__ void __launch_bounds__(scatter_threads<FMT>()) scatter_quant_kernel(
    const int32_t* __restrict__ ids, int T, int E, int K, const __nv_bfloat16* __restrict__ hidden,
    int H, const int32_t* __restrict__ prefix, const int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ pad_off, int32_t* __restrict__ chunk_off,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* __restrict__ prow_slot,
    int32_t* __restrict__ otab, uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int s_off[kMaxExperts], s_poff[kMaxExperts];
  __shared__ int s_e[kTokensPerRouteBlock * kMaxTopK];
  __shared__ RowDst s_dst[kTokensPerRouteBlock * kMaxTopK];
  constexpr int W = scatter_warps_per_token<FMT>();
  __shared__ uint64_t wsum[scatter_threads<FMT>() / 32];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int tok0 = blockIdx.x * kTokensPerRouteBlock;
  const int ntok = min(kTokensPerRouteBlock, T - tok0);
  const int nslot = ntok * K;
  const int tid = static_cast<int>(threadIdx.x);
  const int tok = warp / W, part = warp % W;

  // Loads that do not depend on the scans go out first, so their latency
  // overlaps the scan: each slot's expert and its block prefix, and the
  // first unit of this thread's share of its token row.
  int slot_e = 0, slot_pre = 0;
  if (tid < nslot) {
    slot_e = ids[static_cast<int64_t>(tok0) * K + tid];
    s_e[tid] = slot_e;
    slot_pre = prefix[static_cast<int64_t>(blockIdx.x) * E + slot_e];
  }
  const __nv_bfloat16* xrow = hidden + static_cast<int64_t>(tok0 + tok) * H;
  const int first = part * 32 + lane;
  RawUnit<FMT> unit0;
  if (tok < ntok && first < row_units<FMT>(H)) load_unit<FMT>(xrow, first, unit0);

  // 1. offsets
  const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
  const int c0 = e0 < E ? counts[e0] : 0, c1 = e1 < E ? counts[e1] : 0;
  const int p0 = (c0 + kRowBlock - 1) / kRowBlock, p1 = (c1 + kRowBlock - 1) / kRowBlock;
  int xo, xc;
  block_scan_counts(c0 + c1, p0 + p1, wsum, xo, xc);
  const int xp = xc * kRowBlock;
  if (e0 < E) {
    s_off[e0] = xo;
    s_poff[e0] = xp;
  }
  if (e1 < E) {
    s_off[e1] = xo + c0;
    s_poff[e1] = xp + p0 * kRowBlock;
  }
  if (blockIdx.x == 0) {
    if (e0 < E) {
      offsets[e0] = xo;
      pad_off[e0] = xp;
      chunk_off[e0] = xc;
    }
    if (e1 < E) {
      offsets[e1] = xo + c0;
      pad_off[e1] = xp + p0 * kRowBlock;
      chunk_off[e1] = xc + p0;
    }
    if (e0 == E - 1 || e1 == E - 1) {
      offsets[E] = xo + c0 + c1;
      pad_off[E] = xp + (p0 + p1) * kRowBlock;
      chunk_off[E] = xc + p0 + p1;
    }
  }
  // one block past the routing blocks writes the mixed-order tables (a
  // block without tokens, so no routing block waits for it); it has no
  // slots or rows and ends here
  if (otab && tok0 >= T) {
    store_mixed_tables(E, c0, c1, p0, p1, xp, wsum, otab);
    return;
  }
  __syncthreads();  // s_off, s_poff and s_e are complete

  // 2. stable ranks, all of the block's slots at once: slot j = i*K + k
  //    ranks after the block's earlier slots of its expert, which are those
  //    of earlier tokens (the K experts of one token are distinct), and after
  //    the earlier blocks' slots (prefix)
  if (tid < nslot) {
    const int j = tid;
    const int e = slot_e;
    int r = slot_pre;
    for (int j2 = 0; j2 < j - j % K; ++j2) r += s_e[j2] == e;
    const int64_t s = static_cast<int64_t>(tok0) * K + j;
    perm[s_off[e] + r] = static_cast<int32_t>(s);
    const int prow = s_poff[e] + r;
    inv[s] = prow;
    if (prow_slot) prow_slot[prow] = static_cast<int32_t>(s);
    s_dst[j] = row_dst<FMT>(prow, H);
  }
  __syncthreads();

  // 3. GEMM1 input rows
  if (tok >= ntok) return;
  quant_row_to_rows<FMT>(xrow, H, RowDsts{s_dst + tok * K}, K, xq, xsf, first, 32 * W, &unit0);
}

// ---------------------------------------------------------------- small batches
// Decode batches (T <= kSmallFrontTokens): routing, the expert histogram and
// scans, the stable ranks and the GEMM1 input in one kernel, in place of the
// three kernels above (each of which would otherwise wait for the previous
// one).  One block per token: every block routes all T tokens and derives
// the same tables (a few microseconds of redundant work), block 0 stores
// them, and block b spreads token b's input quantisation over its 256
// threads instead of one warp.
template <int FMT, int MAXJ>
__global__ void __launch_bounds__(256) small_front_kernel(
    const float* __restrict__ logits, int T, int E, int K, const __nv_bfloat16* __restrict__ hidden,
    int H, int32_t* __restrict__ ids, float* __restrict__ w, int32_t* __restrict__ counts,
    int32_t* __restrict__ offsets, int32_t* __restrict__ pad_off, int32_t* __restrict__ chunk_off,
    int32_t* __restrict__ perm, int32_t* __restrict__ inv, int32_t* __restrict__ prow_slot,
    int32_t* __restrict__ done1, uint8_t* __restrict__ xq, uint8_t* __restrict__ xsf) {
  pdl_launch_dependents();
  __shared__ int hist[kMaxExperts], cnt[kMaxExperts], s_off[kMaxExperts], s_poff[kMaxExperts];
  __shared__ int s_ids[kSmallFrontTokens * kMaxTopK], s_prow[kSmallFrontTokens * kMaxTopK];
  __shared__ uint64_t wsum[8];
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = cnt[e] = 0;
  __syncthreads();
  // the previous forward's last kernels may still read what this one writes
  pdl_wait();

  const bool store = blockIdx.x == 0;
  // 1. routing: warp w takes tokens w, w + 8
  for (int t = warp; t < T; t += 8) {
    int my_i;
    float my_w;
    route_token<MAXJ>(logits + static_cast<int64_t>(t) * E, E, K, lane, &my_i, &my_w);
    if (lane < K) {
      if (store) {
        ids[t * K + lane] = my_i;
        w[t * K + lane] = my_w;
      }
      s_ids[t * K + lane] = my_i;
      atomicAdd(&hist[my_i], 1);
    }
  }
  __syncthreads();

  // 2. per-expert offsets (two experts per thread, E <= 512)
  const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
  const int c0 = e0 < E ? hist[e0] : 0, c1 = e1 < E ? hist[e1] : 0;
  const int p0 = (c0 + kRowBlock - 1) / kRowBlock, p1 = (c1 + kRowBlock - 1) / kRowBlock;
  int xo, xc;
  block_scan_counts(c0 + c1, p0 + p1, wsum, xo, xc);
  const int xp = xc * kRowBlock;
  if (e0 < E) {
    s_off[e0] = xo;
    s_poff[e0] = xp;
  }
  if (e1 < E) {
    s_off[e1] = xo + c0;
    s_poff[e1] = xp + p0 * kRowBlock;
  }
  if (store) {
    if (done1) {
      if (e0 < E) done1[e0] = 0;
      if (e1 < E) done1[e1] = 0;
    }
    if (e0 < E) {
      counts[e0] = c0;
      offsets[e0] = xo;
      pad_off[e0] = xp;
      chunk_off[e0] = xc;
    }
    if (e1 < E) {
      counts[e1] = c1;
      offsets[e1] = xo + c0;
      pad_off[e1] = xp + p0 * kRowBlock;
      chunk_off[e1] = xc + p0;
    }
    if (e0 == E - 1 || e1 == E - 1) {
      offsets[E] = xo + c0 + c1;
      pad_off[E] = xp + (p0 + p1) * kRowBlock;
      chunk_off[E] = xc + p0 + p1;
    }
  }
  __syncthreads();

  // 3. stable ranks in slot order s = t*K + k (the K experts of a token
  //    are distinct, so one token's slots never share a counter)
  if (warp == 0) {
    for (int t = 0; t < T; ++t) {
      if (lane < K) {
        const int s = t * K + lane;
        const int e = s_ids[s];
        const int r = cnt[e]++;
        const int prow = s_poff[e] + r;
        if (store) {
          perm[s_off[e] + r] = s;
          inv[s] = prow;
          if (prow_slot) prow_slot[prow] = s;
        }
        s_prow[s] = prow;
      }
      __syncwarp();
    }
  }
  __syncthreads();

  // 4. token b's GEMM1 input rows, its units spread over the block
  const int t = blockIdx.x;
  for (int u = threadIdx.x; u < row_units<FMT>(H); u += blockDim.x)
    quant_unit_to_rows<FMT>(hidden + static_cast<int64_t>(t) * H, H, u, s_prow + t * K, K, xq,
                            xsf);
}

// ---------------------------------------------------------------- batched format
// Batched-expert input [E, M, H] with per-expert counts: block (x, e)
// writes the GEMM1 input of rows 8x..8x+7 of expert e (one warp each) into
// that expert's 128-row-padded segment.  Every block scans the counts over
// the experts itself (a block scan, E <= 512) for its segment base; block
// (0, 0) also stores the tables the GEMMs read.  A count outside [0, M] is
// clamped and reported through the status word.
template <int FMT>
__global__ void __launch_bounds__(256) batched_quant_kernel(
    const __nv_bfloat16* __restrict__ hidden, const int32_t* __restrict__ counts_in, int M, int E,
    int H, int32_t* __restrict__ counts, int32_t* __restrict__ offsets,
    int32_t* __restrict__ pad_off, int32_t* __restrict__ chunk_off, uint8_t* __restrict__ xq,
    uint8_t* __restrict__ xsf, int* status) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ uint64_t wsum[8];
  __shared__ int s_base, s_cnt;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e = blockIdx.y;
  const bool first = blockIdx.x == 0 && blockIdx.y == 0;
  const int e0 = 2 * threadIdx.x, e1 = e0 + 1;
  int c0 = e0 < E ? counts_in[e0] : 0, c1 = e1 < E ? counts_in[e1] : 0;
  if (first && (c0 < 0 || c0 > M || c1 < 0 || c1 > M)) report_status(status, kStatusBadCount);
  c0 = min(max(c0, 0), M);
  c1 = min(max(c1, 0), M);
  const int p0 = (c0 + kRowBlock - 1) / kRowBlock, p1 = (c1 + kRowBlock - 1) / kRowBlock;
  int xo, xc;
  block_scan_counts(c0 + c1, p0 + p1, wsum, xo, xc);
  const int xp = xc * kRowBlock;
  if (e0 == e) {
    s_base = xp;
    s_cnt = c0;
  }
  if (e1 == e) {
    s_base = xp + p0 * kRowBlock;
    s_cnt = c1;
  }
  if (first) {
    if (e0 < E) {
      counts[e0] = c0;
      offsets[e0] = xo;
      pad_off[e0] = xp;
      chunk_off[e0] = xc;
    }
    if (e1 < E) {
      counts[e1] = c1;
      offsets[e1] = xo + c0;
      pad_off[e1] = xp + p0 * kRowBlock;
      chunk_off[e1] = xc + p0;
    }
    if (e0 == E - 1 || e1 == E - 1) {
      offsets[E] = xo + c0 + c1;
      pad_off[E] = xp + (p0 + p1) * kRowBlock;
      chunk_off[E] = xc + p0 + p1;
    }
  }
  __syncthreads();
  const int r = blockIdx.x * kTokensPerRouteBlock + warp;
  if (r >= s_cnt) return;
  const int prow = s_base + r;
  quant_row_to_rows<FMT>(hidden + (static_cast<int64_t>(e) * M + r) * H, H, PaddedRows{&prow, H}, 1,
                         xq, xsf, lane);
}

// ---------------------------------------------------------------- combine
// out[t] = bf16( sum_k w[t,k] * y[row(t,k)] ), fp32 accumulation in k order.
// Grid (T, H/1024): each thread owns 8 consecutive columns (16-byte loads and
// stores, coalesced along H).
// kGroup rows' loads are in flight before their sums (which still run in k
// order): 8 for prefill-sized launches (171 -> 165 us at T = 8192, 95 % of
// the copy bandwidth), 1 for smaller ones, where the kernel launches early
// behind GEMM2 (programmatic dependent launch) and its 64 registers per
// thread instead of 32 cost the bf16 T = 512 layer 3 %.
template <int kGroup>
__global__ void __launch_bounds__(128) combine_kernel(const __nv_bfloat16* __restrict__ y,
                                                      const int32_t* __restrict__ inv,
                                                      const float* __restrict__ w, int K, int H,
                                                      __nv_bfloat16* __restrict__ out) {
  pdl_launch_dependents();
  pdl_wait();
  __shared__ int64_t s_row[kMaxTopK];
  __shared__ float s_w[kMaxTopK];
  const int t = blockIdx.x;
  if (threadIdx.x < K) {
    s_row[threadIdx.x] = inv[static_cast<int64_t>(t) * K + threadIdx.x];
    s_w[threadIdx.x] = w[static_cast<int64_t>(t) * K + threadIdx.x];
  }
  __syncthreads();
  const int c = blockIdx.y * blockDim.x + threadIdx.x;
  if (c >= H / 8) return;
  float acc[8];
#pragma unroll
  for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
  for (int k0 = 0; k0 < K; k0 += kGroup) {
    uint4 u[kGroup];
#pragma unroll
    for (int i = 0; i < kGroup; ++i)
      if (k0 + i < K) u[i] = __ldg(reinterpret_cast<const uint4*>(y + s_row[k0 + i] * H) + c);
#pragma unroll
    for (int i = 0; i < kGroup; ++i) {
      if (k0 + i >= K) break;
      const uint32_t wv[4] = {u[i].x, u[i].y, u[i].z, u[i].w};
      const float wk = s_w[k0 + i];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[q]));
        acc[2 * q] = fmaf(wk, p.x, acc[2 * q]);
        acc[2 * q + 1] = fmaf(wk, p.y, acc[2 * q + 1]);
      }
    }
  }
  uint32_t o[4];
#pragma unroll
  for (int q = 0; q < 4; ++q) {
    const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * q], acc[2 * q + 1]);
    o[q] = *reinterpret_cast<const uint32_t*>(&b);
  }
  reinterpret_cast<uint4*>(out + static_cast<int64_t>(t) * H)[c] = make_uint4(o[0], o[1], o[2], o[3]);
}

// ---------------------------------------------------------------- inspection
// GEMM1 input of each token back in token order, canonical layout.
__global__ void debug_act_kernel(int fmt, const int32_t* __restrict__ inv, int K, int H,
                                 const uint8_t* __restrict__ xq, const uint8_t* __restrict__ xsf,
                                 uint8_t* __restrict__ codes, uint8_t* __restrict__ scales) {
  const int t = blockIdx.x;
  const int64_t prow = inv[static_cast<int64_t>(t) * K];
  const int cb = fmt == kFmtNVFP4 ? H / 2 : H;
  const int nsf = fmt == kFmtNVFP4 ? H / 16 : H / 32;
  const int tiles_k = nsf / 4;
  for (int i = threadIdx.x; i < cb; i += blockDim.x)
    codes[static_cast<int64_t>(t) * cb + i] = xq[prow * cb + i];
  for (int j = threadIdx.x; j < nsf; j += blockDim.x)
    scales[static_cast<int64_t>(t) * nsf + j] = xsf[sf_tile_offset(prow, j, tiles_k)];
}

// GEMM2 input (dequantised) and GEMM2 output rows in unpadded row order.
__global__ void debug_rows_kernel(int fmt, const int32_t* __restrict__ offsets,
                                  const int32_t* __restrict__ pad_off, int E, int I, int H,
                                  const uint8_t* __restrict__ hq, const uint8_t* __restrict__ hsf,
                                  const __nv_bfloat16* __restrict__ y, float* __restrict__ h_out,
                                  float* __restrict__ y_out) {
  const int r = blockIdx.x;
  int lo = 0, hi = E;  // offsets[lo] <= r < offsets[hi]
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (offsets[mid] <= r) lo = mid; else hi = mid;
  }
  const int64_t prow = pad_off[lo] + (r - offsets[lo]);
  if (h_out) {
    for (int i = threadIdx.x; i < I; i += blockDim.x) {
      float v;
      if (fmt == kFmtBF16) {
        v = __bfloat162float(reinterpret_cast<const __nv_bfloat16*>(hq)[prow * I + i]);
      } else if (fmt == kFmtNVFP4) {
        const uint8_t byte = hq[prow * (I / 2) + i / 2];
        const uint8_t q = (i & 1) ? (byte >> 4) : (byte & 0xF);
        const float mag[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
        const float e2 = (q & 8) ? -mag[q & 7] : mag[q & 7];
        v = e2 * e4m3_to_float(hsf[sf_tile_offset(prow, i / 16, I / 64)]);
      } else {
        const float sc = exact_pow2(static_cast<int>(hsf[sf_tile_offset(prow, i / 32, I / 128)]) - 127);
        v = e4m3_to_float(hq[prow * I + i]) * sc;
      }
      h_out[static_cast<int64_t>(r) * I + i] = v;
    }
  }
  if (y_out)
    for (int j = threadIdx.x; j < H; j += blockDim.x)
      y_out[static_cast<int64_t>(r) * H + j] = __bfloat162float(y[prow * H + j]);
}

}  // namespace

cudaError_t launch_route(const float* logits, int T, int E, int K, int32_t* ids, float* w,
                         int32_t* blockhist, cudaStream_t s) {
  const int nb = (T + kTokensPerRouteBlock - 1) / kTokensPerRouteBlock;
  auto k = E <= 128   ? route_kernel<4>
           : E <= 256 ? route_kernel<8>
           : E <= 384 ? route_kernel<12>
                      : route_kernel<16>;
  return launch_pdl(g_pdl_small, k, dim3(nb), dim3(256), 0, s, logits, T, E, K, ids, w,
                    blockhist);
}

cudaError_t launch_expert_scan(const int32_t* blockhist, int NB, int E, int32_t* prefix,
                               int32_t* counts, cudaStream_t s) {
  // the two-pass kernel only pays off for long histograms: for a few routing
  // blocks (bf16 T = 512: 64) it measured 8 us slower per layer
  if (NB < 256)
    return launch_pdl(g_pdl_small, expert_scan_warp_kernel, dim3((E + 7) / 8), dim3(256), 0, s,
                      blockhist, NB, E, prefix, counts);
  return launch_pdl(g_pdl_small, expert_scan_kernel, dim3((E + 31) / 32), dim3(1024), 0, s,
                    blockhist, NB, E, prefix, counts);
}

cudaError_t launch_scatter_quant(int fmt, const int32_t* ids, int T, int E, int K,
                                 const void* hidden, int H, const int32_t* prefix,
                                 const int32_t* counts, int32_t* offsets, int32_t* pad_off,
                                 int32_t* chunk_off, int32_t* perm, int32_t* inv,
                                 int32_t* prow_slot, int32_t* otab, uint8_t* xq, uint8_t* xsf,
                                 cudaStream_t s) {
  const int nb = (T + kTokensPerRouteBlock - 1) / kTokensPerRouteBlock;
  const auto* hb = static_cast<const __nv_bfloat16*>(hidden);
  auto k = fmt == kFmtBF16 ? scatter_quant_kernel<kFmtBF16>
           : fmt == kFmtMXFP8 ? scatter_quant_kernel<kFmtMXFP8>
                              : scatter_quant_kernel<kFmtNVFP4>;
  const int threads = fmt == kFmtBF16    ? scatter_threads<kFmtBF16>()
                      : fmt == kFmtMXFP8 ? scatter_threads<kFmtMXFP8>()
                                         : scatter_threads<kFmtNVFP4>();
  return launch_pdl(g_pdl_small, k, dim3(nb + (otab ? 1 : 0)), dim3(threads), 0, s, ids, T, E, K,
                    hb, H, prefix, counts, offsets, pad_off, chunk_off, perm, inv, prow_slot, otab,
                    xq, xsf);
}

cudaError_t launch_small_front(int fmt, const float* logits, int T, int E, int K,
                               const void* hidden, int H, int32_t* ids, float* w,
                               int32_t* counts, int32_t* offsets, int32_t* pad_off,
                               int32_t* chunk_off, int32_t* perm, int32_t* inv,
                               int32_t* prow_slot, int32_t* done1, uint8_t* xq, uint8_t* xsf,
                               cudaStream_t s) {
  if (T > kSmallFrontTokens) return cudaErrorInvalidValue;
  const auto* hb = static_cast<const __nv_bfloat16*>(hidden);
  auto pick = [&](auto k4, auto k8, auto k16) { return E <= 128 ? k4 : E <= 256 ? k8 : k16; };
  auto k = fmt == kFmtBF16
               ? pick(small_front_kernel<kFmtBF16, 4>, small_front_kernel<kFmtBF16, 8>,
                      small_front_kernel<kFmtBF16, 16>)
           : fmt == kFmtMXFP8
               ? pick(small_front_kernel<kFmtMXFP8, 4>, small_front_kernel<kFmtMXFP8, 8>,
                      small_front_kernel<kFmtMXFP8, 16>)
               : pick(small_front_kernel<kFmtNVFP4, 4>, small_front_kernel<kFmtNVFP4, 8>,
                      small_front_kernel<kFmtNVFP4, 16>);
  return launch_pdl(g_pdl_small, k, dim3(T), dim3(256), 0, s, logits, T, E, K, hb, H, ids, w,
                    counts, offsets, pad_off, chunk_off, perm, inv, prow_slot, done1, xq, xsf);
}

cudaError_t launch_batched_quant(int fmt, const void* hidden, const int32_t* counts_in, int M,
                                 int E, int H, int32_t* counts, int32_t* offsets,
                                 int32_t* pad_off, int32_t* chunk_off, uint8_t* xq, uint8_t* xsf,
                                 int* status, cudaStream_t s) {
  const dim3 grid((M + kTokensPerRouteBlock - 1) / kTokensPerRouteBlock, E);
  const auto* hb = static_cast<const __nv_bfloat16*>(hidden);
  auto k = fmt == kFmtBF16 ? batched_quant_kernel<kFmtBF16>
           : fmt == kFmtMXFP8 ? batched_quant_kernel<kFmtMXFP8>
                              : batched_quant_kernel<kFmtNVFP4>;
  return launch_pdl(g_pdl_small, k, grid, dim3(256), 0, s, hb, counts_in, M, E, H, counts,
                    offsets, pad_off, chunk_off, xq, xsf, status);
}

cudaError_t launch_combine(const void* y, const int32_t* inv, const float* w, int T, int K, int H,
                           void* out, cudaStream_t s) {
  const dim3 grid(T, (H / 8 + 127) / 128);
  auto k = T > 1024 ? combine_kernel<8> : combine_kernel<1>;
  return launch_pdl(g_pdl_small, k, grid, dim3(128), 0, s,
                    static_cast<const __nv_bfloat16*>(y), inv, w, K, H,
                    static_cast<__nv_bfloat16*>(out));
}

cudaError_t launch_debug_act(int fmt, const int32_t* inv, int T, int K, int H, const uint8_t* xq,
                             const uint8_t* xsf, uint8_t* codes, uint8_t* scales,
                             cudaStream_t s) {
  debug_act_kernel<<<T, 256, 0, s>>>(fmt, inv, K, H, xq, xsf, codes, scales);
  return cudaGetLastError();
}

cudaError_t launch_debug_rows(int fmt, const int32_t* offsets, const int32_t* pad_off, int E,
                              int R, int I, int H, const uint8_t* hq, const uint8_t* hsf,
                              const void* y, float* h_out, float* y_out, cudaStream_t s) {
  debug_rows_kernel<<<R, 256, 0, s>>>(fmt, offsets, pad_off, E, I, H, hq, hsf,
                                      static_cast<const __nv_bfloat16*>(y), h_out, y_out);
  return cudaGetLastError();
}

}  // namespace moe
