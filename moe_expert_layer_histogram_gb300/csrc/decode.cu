// decode.cu -- the whole layer in one launch for decode batches (T <= 16).
//
// The b12x backend runs routing, both expert GEMMs with SwiGLU between them
// and the reduction in a single call (PR #40082 report, sec. 实现拆解 item 1),
// and MegaMoE fuses its layer into one kernel too (MegaMoE kernel-drop
// workflow page, sec. 一).  Here one persistent launch does, per forward:
//   1. routing of all T tokens and the expert tables (counts, offsets,
//      128-row-padded offsets, chunk offsets, stable ranks) -- every CTA
//      computes them itself in shared memory (T <= 16 tokens, a few hundred
//      experts), CTA 0 also stores them for inspection;
//   2. the GEMM1 input of each token, quantised into its K padded rows in
//      row segments, each by whichever CTA claims it (an atomic counter);
//   3. the GEMM1 (+ SwiGLU or squared ReLU, re-quantised) and GEMM2 work
//      items, claimed one at a time from an atomic counter in order (all
//      GEMM1 items before any GEMM2 item); a GEMM2 item of expert e waits
//      until every GEMM1 epilogue warp of expert e has stored its rows;
//   4. the combine: units (token, block of columns) claimed from a counter
//      once a CTA has no GEMM item left, each waiting until every GEMM2
//      epilogue warp of the token's K experts has stored its rows; the sum
//      runs in k order in fp32, as the combine kernel's does.
// Every wait is bounded (2 s), and a CTA only ever waits for work that a
// running CTA has already claimed, so the launch needs no co-residency of
// its CTAs.  The last CTA to leave resets the counters for the next forward.
//
// Before waiting -- for the activations of its first GEMM1 item, or for
// GEMM1 results of a GEMM2 item -- the producer prefetches the item's weight
// tiles into L2, so the weight stream starts while the routing, the
// quantisation or GEMM1 is still in progress.
//
// Warp roles during the GEMMs (224 threads): warp 0 writes the stage scales
// into TMEM lane quarter 0 (tcgen05.st; all decode chunks hold <= 16 rows),
// warp 1 issues the MMAs, warp 2 claims items and streams the ring, warps
// 3-6 run the epilogues.  The other phases use all 224 threads.
#include "gemm_common.cuh"
#include "route_token.cuh"
#include "rowquant.cuh"

namespace moe {

namespace {

constexpr int kDecThreads = 224;
constexpr int kDecWarps = kDecThreads / 32;
constexpr int kDecMRows = 32;
constexpr int kItemRing = 4;

template <int FMT>
__host__ __device__ constexpr int dec_stages() {
  return num_stages<FMT, kDecMRows, 1>();
}
template <int FMT>
__host__ __device__ constexpr int dec_stage_bytes() {
  return stage_bytes<FMT, kDecMRows, 1>();
}

// Shared memory after the ring: barriers, then the tables.
struct DecSmem {
  int tab[3 * (kMaxExperts + 1)];   // chunk_off[E+1], pad_off[E], counts[E] (GEMM item tables)
  int off[kMaxExperts + 1];         // unpadded offsets
  int rank[kMaxExperts];            // stable-rank counters
  int ids[kSmallFrontTokens * kMaxTopK];
  float w[kSmallFrontTokens * kMaxTopK];
  int prow[kSmallFrontTokens * kMaxTopK];
  int rank2[kSmallFrontTokens * kMaxTopK];
  int wsum[3 * kDecWarps];
  int items[kItemRing];
  int bcast;
};

template <int FMT>
__host__ __device__ constexpr int dec_smem_bytes() {
  return 1024 + dec_stages<FMT>() * dec_stage_bytes<FMT>() +
         (3 * dec_stages<FMT>() + 5 + 2 * kItemRing) * 8 + 16 + static_cast<int>(sizeof(DecSmem));
}

// Three exclusive scans over E <= 512 experts at once (each thread takes
// three consecutive experts): counts -> off, 128-padded counts -> pad_off,
// 128-row chunks -> chunk_off; totals at [E].
__device__ __forceinline__ void scan_tables(const int* counts, int E, DecSmem& S) {
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int e0 = 3 * threadIdx.x;
  int c[3], a = 0, b = 0, d = 0;
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    c[i] = e0 + i < E ? counts[e0 + i] : 0;
    a += c[i];
    b += (c[i] + kRowBlock - 1) / kRowBlock * kRowBlock;
    d += (c[i] + kRowBlock - 1) / kRowBlock;
  }
  int ia = a, ib = b, id = d;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int xa = __shfl_up_sync(0xFFFFFFFFu, ia, o);
    const int xb = __shfl_up_sync(0xFFFFFFFFu, ib, o);
    const int xd = __shfl_up_sync(0xFFFFFFFFu, id, o);
    if (lane >= o) {
      ia += xa;
      ib += xb;
      id += xd;
    }
  }
  if (lane == 31) {
    S.wsum[warp] = ia;
    S.wsum[kDecWarps + warp] = ib;
    S.wsum[2 * kDecWarps + warp] = id;
  }
  __syncthreads();
  int pa = ia - a, pb = ib - b, pd = id - d;
  for (int w = 0; w < warp; ++w) {
    pa += S.wsum[w];
    pb += S.wsum[kDecWarps + w];
    pd += S.wsum[2 * kDecWarps + w];
  }
  int* chunk_off = S.tab;
  int* pad_off = S.tab + (E + 1);
#pragma unroll
  for (int i = 0; i < 3; ++i) {
    const int e = e0 + i;
    if (e < E) {
      S.off[e] = pa;
      pad_off[e] = pb;
      chunk_off[e] = pd;
    }
    pa += c[i];
    pb += (c[i] + kRowBlock - 1) / kRowBlock * kRowBlock;
    pd += (c[i] + kRowBlock - 1) / kRowBlock;
    if (e == E - 1) {
      S.off[E] = pa;
      chunk_off[E] = pd;
    }
  }
}

// Bounded wait until *counter >= need; warp-uniform result.
__device__ __forceinline__ bool wait_counter(const int* counter, int need, volatile int* abort) {
  return wait_count_at_least(counter, need, abort);
}

__device__ __forceinline__ int ld_acquire(const int* p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

__device__ __forceinline__ void prefetch_l2(const void* p, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(p), "r"(bytes) : "memory");
}

template <int FMT, int EPI1>
__global__ void __launch_bounds__(kDecThreads, 1)
    moe_decode_kernel(const __grid_constant__ GemmMaps maps1, const __grid_constant__ GemmArgs a1,
                      const __grid_constant__ GemmMaps maps2, const __grid_constant__ GemmArgs a2,
                      const __grid_constant__ DecodeArgs d) {
  constexpr int SFT = Fmt<FMT>::kSfTiles;
  constexpr int SB = dec_stage_bytes<FMT>();
  constexpr int kStages = dec_stages<FMT>();
  constexpr int A_BYTES = kDecMRows * 128;
  constexpr int kOffBsf = A_BYTES + kTileBytes;
  constexpr int kOffAsf = kOffBsf + SFT * 512;
  constexpr int kAccCols = 128;
  constexpr int kSfColsPerStage = 32;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * SB);
  uint64_t* empty = full + kStages;
  uint64_t* sf_ready = empty + kStages;
  uint64_t* tfull = sf_ready + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drained = tempty + 2;
  uint64_t* ifull = drained + 1;
  uint64_t* iempty = ifull + kItemRing;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(iempty + kItemRing);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  DecSmem& S = *reinterpret_cast<DecSmem*>(tmem_holder + 4);
  DecodeCtl* ctl = d.ctl;
  const int T = d.T, E = a1.E, K = d.K, H = d.H;
  const bool staged = SFT > 0;
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4);
    }
    mbar_init(drained, 1);
    for (int i = 0; i < kItemRing; ++i) {
      mbar_init(&ifull[i], 1);
      mbar_init(&iempty[i], 1 + 4 + (staged ? 1 : 0));  // MMA, epilogue warps, stager
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32 * 2 + 1)
    for (int i = 0; i < 4; ++i) {
      prefetch_tmap(&maps1.a[i]);
      prefetch_tmap(&maps2.a[i]);
    }
  int* counts = S.tab + 2 * E + 1;
  for (int e = threadIdx.x; e < E; e += blockDim.x) counts[e] = S.rank[e] = 0;
  __syncthreads();

  // ---------------------------------------------------------------- 1. routing, tables
  // Routing reads only the router logits, which the layer's own kernels never
  // write (the router GEMM producing them is not launched with programmatic
  // dependencies), so it runs before the wait on the previous kernel, like
  // the multi-kernel path's routing kernel; everything it writes to global
  // memory waits.
  for (int t = warp; t < T; t += kDecWarps) {
    int my_i;
    float my_w;
    route_token<kMaxExperts / 32>(d.logits + static_cast<int64_t>(t) * E, E, K, lane, &my_i,
                                  &my_w);
    if (lane < K) {
      S.ids[t * K + lane] = my_i;
      S.w[t * K + lane] = my_w;
      atomicAdd(&counts[my_i], 1);
    }
  }
  __syncthreads();
  scan_tables(counts, E, S);
  __syncthreads();
  const int* pad_off = S.tab + (E + 1);
  const bool store_tables = blockIdx.x == 0;
  if (warp == 0) {
    // stable ranks in slot order s = t*K + k (a token's K experts are distinct)
    for (int t = 0; t < T; ++t) {
      if (lane < K) {
        const int s = t * K + lane;
        const int e = S.ids[s];
        const int r = S.rank[e]++;
        S.prow[s] = pad_off[e] + r;
        S.rank2[s] = S.off[e] + r;  // unpadded row, for the permutation table
      }
      __syncwarp();
    }
  }
  __syncthreads();
  // the previous forward's kernels may still read what this one writes, and
  // a layer's hidden states may be the previous layer's output
  pdl_wait();
  if (store_tables) {
    for (int i = threadIdx.x; i < T * K; i += blockDim.x) {
      d.perm[S.rank2[i]] = i;
      d.inv[i] = S.prow[i];
    }
    for (int i = threadIdx.x; i < T * K; i += blockDim.x) {
      d.ids[i] = S.ids[i];
      d.w[i] = S.w[i];
    }
    for (int e = threadIdx.x; e <= E; e += blockDim.x) {
      d.offsets[e] = S.off[e];
      d.chunk_off[e] = S.tab[e];
      if (e < E) {
        d.pad_off[e] = pad_off[e];
        d.counts[e] = counts[e];
      }
    }
    if (threadIdx.x == 0) d.pad_off[E] = S.tab[E] * kRowBlock;  // every decode chunk is one block
  }
  __syncthreads();

  // ---------------------------------------------------------------- 2. GEMM1 input
  // Work units are row segments of kDecThreads quantisation blocks (one per
  // thread), claimed in order, so a token's row is spread over several CTAs.
  const int segs = (row_units<FMT>(H) + kDecThreads - 1) / kDecThreads;  // segments per token
  for (;;) {
    if (threadIdx.x == 0) S.bcast = atomicAdd(&ctl->qclaim, 1);
    __syncthreads();
    const int u = S.bcast;
    __syncthreads();
    if (u >= T * segs) break;
    const int t = u / segs;
    const int unit = (u - t * segs) * kDecThreads + threadIdx.x;
    if (unit < row_units<FMT>(H))
      quant_unit_to_rows<FMT>(static_cast<const __nv_bfloat16*>(d.hidden) + static_cast<int64_t>(t) * H,
                              H, unit, S.prow + t * K, K, d.xq, d.xsf);
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) atomicAdd(&ctl->qdone, 1);
  }

  // ---------------------------------------------------------------- 3. GEMM items
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const Tables tab{S.tab, S.tab + (E + 1), S.tab + (2 * E + 1), nullptr};
  const int n1 = S.tab[E] * a1.n_tiles;
  const int total = n1 + S.tab[E] * a2.n_tiles;
  auto second = [&](int item) { return item >= n1; };
  auto local_item = [&](int item) { return second(item) ? item - n1 : item; };
  auto gargs = [&](int item) -> const GemmArgs& { return second(item) ? a2 : a1; };
  // The next item of this CTA's sequence, published by the producer: -1 ends
  // the sequence, -2 means the wait gave up.  next_item_warp: all 32 lanes
  // call it (lane 0 releases the slot); next_item_thread: one thread.
  auto next_item_warp = [&](int& slot, uint32_t& ph) -> int {
    const bool ok = mbar_wait(&ifull[slot], ph, abort_flag);
    const int item = ok ? S.items[slot] : -2;
    __syncwarp();
    if (ok && lane == 0) mbar_arrive(&iempty[slot]);
    if (++slot == kItemRing) {
      slot = 0;
      ph ^= 1u;
    }
    return __all_sync(0xFFFFFFFFu, item != -2) ? item : -2;
  };
  auto next_item_thread = [&](int& slot, uint32_t& ph) -> int {
    if (!mbar_wait(&ifull[slot], ph, abort_flag)) return -2;
    const int item = S.items[slot];
    mbar_arrive(&iempty[slot]);
    if (++slot == kItemRing) {
      slot = 0;
      ph ^= 1u;
    }
    return item;
  };

  if (warp == 0) {
    // ------------------------------------------------ scale stager
    if (staged) {
      int stage = 0, slot = 0;
      uint32_t phase = 0, iph = 0;
      bool ok = true;
      for (;;) {
        const int item = next_item_warp(slot, iph);
        if (item == -2) {
          ok = false;
          break;
        }
        if (item < 0) break;
        const GemmArgs& A = gargs(item);
        for (int kb = 0; kb < A.num_kb; ++kb) {
          const bool landed = mbar_wait(&full[stage], phase, abort_flag);
          if (!__all_sync(0xFFFFFFFFu, landed)) {
            ok = false;
            break;
          }
          const uint8_t* sp = smem + stage * SB;
          const uint32_t col = tmem + kSfColBase + stage * kSfColsPerStage;  // lanes 0-31
          if constexpr (FMT == kFmtNVFP4) {
            // per 64-element substep j: activation row (lane) scales in
            // column 8j, the 128 weight rows' scales in columns 8j+4..8j+7
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 b = *reinterpret_cast<const uint4*>(sp + kOffBsf + j * 512 + lane * 16);
              v[8 * j] = *reinterpret_cast<const uint32_t*>(sp + kOffAsf + j * 512 + lane * 16);
              v[8 * j + 1] = v[8 * j + 2] = v[8 * j + 3] = 0u;
              v[8 * j + 4] = b.x;
              v[8 * j + 5] = b.y;
              v[8 * j + 6] = b.z;
              v[8 * j + 7] = b.w;
            }
            tmem_st32(col, v);
          } else {
            // weight rows' scales in columns 0-3, activation row in 4
            uint32_t v[8];
            const uint4 b = *reinterpret_cast<const uint4*>(sp + kOffBsf + lane * 16);
            v[0] = b.x;
            v[1] = b.y;
            v[2] = b.z;
            v[3] = b.w;
            v[4] = *reinterpret_cast<const uint32_t*>(sp + kOffAsf + lane * 16);
            v[5] = v[6] = v[7] = 0u;
            tmem_st8(col, v);
          }
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(&sf_ready[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      if (!ok && lane == 0) report_status(a1.status, kStatusTimeout);
    }
  } else if (warp == 2) {
    // ------------------------------------------------ producer: claims items, fills the ring
    if (lane == 0) {
      const uint64_t once = l2_policy_evict_first();
      int stage = 0, slot = 0;
      uint32_t phase = 0, iph = 0;
      int slots = 0;
      int skipped = -1;  // ring position the fault injection left unloaded
      bool ok = true, a_ready = false;
      for (;;) {
        if (!mbar_wait(&iempty[slot], iph ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        int item = atomicAdd(&ctl->iclaim, 1);
        if (item >= total) item = -1;
        S.items[slot] = item;
        mbar_arrive(&ifull[slot]);
        if (++slot == kItemRing) {
          slot = 0;
          iph ^= 1u;
        }
        if (item < 0) break;
        const GemmArgs& A = gargs(item);
        const CUtensorMap* amaps = second(item) ? maps2.a : maps1.a;
        const Item it = map_item<false>(tab, E, A.n_tiles, local_item(item));
        const int amap = it.rows <= 16 ? 0 : 1;
        const uint32_t bytes = (16u << amap) * 128u + A.b_tile_bytes + SFT * 512u;
        const uint8_t* sfa = A.sfa + static_cast<int64_t>(it.prow0 >> 7) * A.sfa_tiles_k * 512;
        const uint8_t* btile =
            A.b_tiles + (static_cast<int64_t>(it.e) * A.n_tiles + it.n_tile) * A.num_kb *
                            A.b_tile_bytes;
        if (second(item) || !a_ready) {
          // GEMM2's activations are GEMM1's output for this expert; GEMM1's
          // are the quantised tokens
          const int* counter = second(item) ? ctl->done1 + it.e : &ctl->qdone;
          const int need =
              second(item) ? 4 * a1.n_tiles * (tab.chunk_off[it.k + 1] - tab.chunk_off[it.k])
                         : T * segs;
          if (ld_acquire(counter) < need) {
            // start the weight stream before waiting for the activations
            for (int kb = 0; kb < A.num_kb; ++kb)
              prefetch_l2(btile + static_cast<int64_t>(kb) * A.b_tile_bytes, A.b_tile_bytes);
            if (!wait_counter(counter, need, abort_flag)) {
              ok = false;
              break;
            }
          }
          if (!second(item)) a_ready = true;
          fence_proxy_async_global();  // generic-proxy stores -> the TMA reads below
        }
        for (int kb = 0; kb < A.num_kb; ++kb) {
          if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (a1.test_stall && blockIdx.x == 0 && skipped < 0) {
            // fault injection: nothing ever completes this stage
            skipped = slots++;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
            continue;
          }
          uint8_t* sp = smem + stage * SB;
          mbar_arrive_expect_tx(&full[stage], bytes);
          tma_load_2d(sp, &amaps[amap], &full[stage], kb * 128, it.prow0);
          bulk_load_hint(sp + A_BYTES, btile + static_cast<int64_t>(kb) * A.b_tile_bytes,
                         A.b_tile_bytes, &full[stage], once);
          if constexpr (SFT > 0) bulk_load(sp + kOffAsf, sfa + kb * SFT * 512, SFT * 512, &full[stage]);
          ++slots;
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
      }
      for (int back = 1; back <= kStages && back <= slots; ++back) {
        const int idx = slots - back;
        if (idx == skipped) continue;
        mbar_wait(&full[idx % kStages], static_cast<uint32_t>((idx / kStages) & 1), nullptr);
      }
      if (!ok) report_status(a1.status, kStatusTimeout);
    }
  } else if (warp == 1) {
    // ------------------------------------------------ MMA issuer
    if (lane == 0) {
      uint32_t idesc;
      if constexpr (FMT == kFmtBF16) idesc = idesc_bf16(128, 128);
      else if constexpr (FMT == kFmtNVFP4) idesc = idesc_nvf4(128, 128);
      else idesc = 0;
      int stage = 0, slot = 0, local = 0;
      uint32_t phase = 0, iph = 0;
      bool ok = true;
      for (;; ++local) {
        const int item = next_item_thread(slot, iph);
        if (item == -2) {
          ok = false;
          break;
        }
        if (item < 0) break;
        const GemmArgs& A = gargs(item);
        const int buf = local & 1;
        const uint32_t use = static_cast<uint32_t>(local >> 1);
        if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem + buf * kAccCols;
        for (int kb = 0; kb < A.num_kb; ++kb) {
          if (!mbar_wait(staged ? &sf_ready[stage] : &full[stage], phase, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          uint8_t* sp = smem + stage * SB;
          const uint32_t a_addr = smem_u32(sp), b_addr = smem_u32(sp + A_BYTES);
          const uint32_t sf_col = tmem + kSfColBase + stage * kSfColsPerStage;
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            if constexpr (FMT == kFmtNVFP4)
              mma_nvf4(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                       sf_col + j * 8, sf_col + j * 8 + 4, (kb | j) != 0);
            else if constexpr (FMT == kFmtMXFP8)
              mma_mxf8(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32),
                       idesc_mxf8(128, 128, j), sf_col + 4, sf_col, (kb | j) != 0);
            else
              mma_bf16(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                       (kb | j) != 0);
          }
          tc_commit(&empty[stage]);
          if (++stage == kStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
        if (!ok) break;
        tc_commit(&tfull[buf]);
      }
      tc_commit(drained);
      mbar_wait(drained, 0, nullptr);
      if (!ok) report_status(a1.status, kStatusTimeout);
    }
  } else if (warp >= 3) {
    // ------------------------------------------------ epilogue warps
    // Warp w reads TMEM lane quarter w % 4; a decode chunk's <= 16 real rows
    // are all in quarter 0, so only warp 4's rows are ever stored, but every
    // warp releases the accumulator and counts the item.
    const int q = warp & 3;
    int slot = 0, local = 0;
    uint32_t iph = 0;
    for (;; ++local) {
      const int item = next_item_warp(slot, iph);
      if (item == -2) {
        if (lane == 0) report_status(a1.status, kStatusTimeout);
        break;
      }
      if (item < 0) break;
      const GemmArgs& A = gargs(item);
      const bool g2 = second(item);
      const Item it = map_item<false>(tab, E, A.n_tiles, local_item(item));
      const int buf = local & 1;
      const uint32_t use = static_cast<uint32_t>(local >> 1);
      if (!mbar_wait(&tfull[buf], use & 1u, abort_flag)) {
        if (lane == 0) report_status(a1.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const int r = q * 32 + lane;
      const bool active = q * 32 < it.rows;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kAccCols;
      const int64_t prow = it.prow0 + r;
      if (active) {
        uint32_t carry[5];
#pragma unroll
        for (int p = 0; p < 2; ++p) {
          uint32_t v[64];
          if (g2) epilogue_load<2>(taddr, p, v);
          else epilogue_load<EPI1>(taddr, p, v);
          tmem_ld_wait();
          epilogue_fence(v);
          if (g2) epilogue_round<FMT, 2>(v, p, r < it.rows, prow, prow, it.n_tile, A, carry);
          else epilogue_round<FMT, EPI1>(v, p, r < it.rows, prow, prow, it.n_tile, A, carry);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[buf]);
      // this warp's rows of the item are stored: count them for the
      // dependent GEMM2 items (GEMM1) or the combine (GEMM2)
      __threadfence();
      __syncwarp();
      if (lane == 0) atomicAdd((g2 ? ctl->done2 : ctl->done1) + it.e, 1);
    }
  }

  // ---------------------------------------------------------------- 4. combine
  // out[t, c] = bf16( sum_k w[t,k] * y[row(t,k), c] ), fp32 in k order; a unit
  // is one token and 8 * 224 columns.
  tc_fence_before();
  __syncthreads();
  const int cols_per_unit = 8 * kDecThreads;
  const int nblk = (H + cols_per_unit - 1) / cols_per_unit;
  const __nv_bfloat16* y = reinterpret_cast<const __nv_bfloat16*>(a2.out);
  bool cok = true;
  for (;;) {
    if (threadIdx.x == 0) S.bcast = atomicAdd(&ctl->cclaim, 1);
    __syncthreads();
    const int c = S.bcast;
    __syncthreads();
    if (c >= T * nblk) break;
    const int t = c / nblk, blk = c % nblk;
    if (warp == 0 && lane < K) {
      // every GEMM2 epilogue warp of each of the token's experts has stored
      const int e = S.ids[t * K + lane];
      const int need = 4 * a2.n_tiles * (tab.chunk_off[e + 1] - tab.chunk_off[e]);
      if (!wait_counter(ctl->done2 + e, need, abort_flag)) cok = false;
    }
    __syncthreads();
    const int col = blk * cols_per_unit + threadIdx.x * 8;
    if (col < H) {
      float acc[8];
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[j] = 0.0f;
      for (int k = 0; k < K; ++k) {
        const int64_t row = S.prow[t * K + k];
        const uint4 u = __ldcg(reinterpret_cast<const uint4*>(y + row * H + col));
        const uint32_t wv[4] = {u.x, u.y, u.z, u.w};
        const float wk = S.w[t * K + k];
#pragma unroll
        for (int qq = 0; qq < 4; ++qq) {
          const float2 p = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&wv[qq]));
          acc[2 * qq] = fmaf(wk, p.x, acc[2 * qq]);
          acc[2 * qq + 1] = fmaf(wk, p.y, acc[2 * qq + 1]);
        }
      }
      uint32_t o[4];
#pragma unroll
      for (int qq = 0; qq < 4; ++qq) {
        const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * qq], acc[2 * qq + 1]);
        o[qq] = *reinterpret_cast<const uint32_t*>(&b);
      }
      *reinterpret_cast<uint4*>(d.out + (static_cast<int64_t>(t) * H + col) * 2) =
          make_uint4(o[0], o[1], o[2], o[3]);
    }
  }
  if (!cok) report_status(a1.status, kStatusTimeout);

  // ---------------------------------------------------------------- teardown
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
  // the last CTA to leave resets the counters for the next forward (which
  // reads them only after this grid has completed)
  __threadfence();
  if (threadIdx.x == 0) S.bcast = atomicAdd(&ctl->exits, 1) == static_cast<int>(gridDim.x) - 1;
  __syncthreads();
  if (S.bcast) {
    __threadfence();
    for (int e = threadIdx.x; e < E; e += blockDim.x) ctl->done1[e] = ctl->done2[e] = 0;
    if (threadIdx.x == 0) {
      ctl->qclaim = ctl->qdone = ctl->iclaim = ctl->cclaim = 0;
      ctl->exits = 0;
    }
  }
}

template <int FMT, int EPI1>
cudaError_t dec_prepare_one() {
  return cudaFuncSetAttribute(moe_decode_kernel<FMT, EPI1>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, dec_smem_bytes<FMT>());
}

template <int FMT>
cudaError_t dec_launch(int epi1, const GemmMaps& m1, const GemmArgs& a1, const GemmMaps& m2,
                       const GemmArgs& a2, const DecodeArgs& d, int grid, cudaStream_t s) {
  auto k = epi1 == 3 ? moe_decode_kernel<FMT, 3> : moe_decode_kernel<FMT, 1>;
  return launch_pdl(g_pdl_gemm, k, dim3(grid), dim3(kDecThreads), dec_smem_bytes<FMT>(), s, m1, a1,
                    m2, a2, d);
}

}  // namespace

cudaError_t decode_prepare(int fmt) {
  cudaError_t e;
  if (fmt == kFmtBF16) {
    e = dec_prepare_one<kFmtBF16, 1>();
    if (e == cudaSuccess) e = dec_prepare_one<kFmtBF16, 3>();
  } else if (fmt == kFmtMXFP8) {
    e = dec_prepare_one<kFmtMXFP8, 1>();
    if (e == cudaSuccess) e = dec_prepare_one<kFmtMXFP8, 3>();
  } else {
    e = dec_prepare_one<kFmtNVFP4, 1>();
    if (e == cudaSuccess) e = dec_prepare_one<kFmtNVFP4, 3>();
  }
  return e;
}

cudaError_t launch_decode(int fmt, int epi1, const GemmMaps& maps1, const GemmArgs& args1,
                          const GemmMaps& maps2, const GemmArgs& args2, const DecodeArgs& d,
                          int grid, cudaStream_t s) {
  if (d.T < 1 || d.T > kSmallFrontTokens || grid < 1) return cudaErrorInvalidValue;
  if (fmt == kFmtBF16) return dec_launch<kFmtBF16>(epi1, maps1, args1, maps2, args2, d, grid, s);
  if (fmt == kFmtMXFP8) return dec_launch<kFmtMXFP8>(epi1, maps1, args1, maps2, args2, d, grid, s);
  return dec_launch<kFmtNVFP4>(epi1, maps1, args1, maps2, args2, d, grid, s);
}

}  // namespace moe
