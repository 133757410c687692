// gemm_pair.cu -- NVFP4 grouped expert GEMMs on CTA pairs (prefill launches).
//
// The same GEMM1 (W13 + SwiGLU / squared ReLU + re-quantisation) and GEMM2
// (W2, bf16 out or in-kernel reduce) as gemm.cu's wide items, computed by
// clusters of two CTAs that share one tcgen05 MMA (cta_group::2, M = 256,
// N = 256): a work item is (expert, pair of 128-row weight tiles, pair of
// 128-row token chunks).  CTA r of the pair loads token chunk 2c + r and
// weight tile 2n + r, so each weight tile reaches shared memory once for two
// token chunks, and each SM's tensor core reads 16 KiB of operands per
// 128-byte K slice instead of 24 KiB.  In the single-CTA wide kernel the
// shared-memory traffic of the TMA writes and MMA reads (about 108 KB per K
// slice and SM) paced the prefill GEMMs; here it is about 72 KB.  (The tile
// and cluster shape are the knobs the MegaMoE kernel-drop workflow page
// exposes as mma_tiler_mnk / cluster_shape_mnk, sec. 四 and 六.)
//
// Measured on GB300 (probe, one 256 x 256 x 64 MMA with coordinates encoded
// in the operands and scales): rank 0 supplies A rows 0-127 and B rows
// 0-127 (the first weight tile), rank 1 A rows 128-255 and B rows 128-255;
// D rows 0-127 land in rank 0's TMEM, 128-255 in rank 1's; each CTA's half
// reads its own rows' activation scales and the scales of all 256 weight
// rows from its own TMEM, laid out as for the single-CTA MMA.
//
// Roles per CTA (512 threads, same warpgroup budgets as the wide kernel):
//   warp 2      operand producer: this CTA's activation slice and its weight
//               tile's codes (TMA), completing on rank 0's stage barrier;
//   warp 3      scale producer: the stage's activation scales and both weight
//               tiles' scales (bulk copies) into this CTA's scale ring;
//   warp 1      rank 0: issues the pair MMAs; both ranks: TMEM alloc/free;
//   warps 4-11  epilogue of this CTA's 128 rows x 256 columns;
//   warps 12-15 scale stagers: write a stage's scales into a free TMEM scale
//               slot of this CTA (tcgen05.st), then arrive on rank 0's slot
//               barrier.
// Rank 0's MMA thread waits for the stage's operands (one barrier, both
// CTAs' copies) and for both CTAs' stagers (8 arrivals, 4 of them from the
// peer), issues four MMAs and commits to the operand stage's empty barrier
// and the scale slot's free barrier in both CTAs; accumulator-full is
// committed to both CTAs, accumulator-empty counts the 16 epilogue warps of
// both.  The trace of an earlier version, which forwarded each stage through
// the stagers and loaded the scales with the operands, showed one stage per
// 512 ns against 264 ns of MMA work: a ring refill took about 2 us.
#include "gemm_common.cuh"

namespace moe {

namespace {

// Operand ring (warp 2): activation codes (128 rows x 128 bytes) + this
// CTA's weight tile codes per stage; both CTAs' copies complete on rank 0's
// barrier, so rank 0's MMA thread waits on one barrier for both halves.
// Scale ring (warp 3): the stage's activation scale tiles (4 x 512 bytes)
// and the scale tiles of both weight tiles (2 x 4 x 512 bytes), loaded ahead
// into this CTA and written into TMEM by its stager warps before the
// operands are needed.  TMEM holds the 256-column accumulator and four scale
// slots of 64 columns (weight scales of substep j at 8j..8j+7, activation
// scales of lane quarter q at 32 + 4j + q).
constexpr int kOpStages = 6;
constexpr int kSfStages = 4;
constexpr int kTSlots = 4;
constexpr int kPairThreads = 512;
constexpr int kOpBytes = 2 * kTileBytes;
constexpr int kSfBytes = 3 * 4 * 512;
constexpr int kSfOffB = 4 * 512;       // weight scales after the activation scales
constexpr int kPSfCols = 64;
static_assert(kSfColBase + kTSlots * kPSfCols <= kTmemCols, "TMEM scale columns");
// Tables in shared memory: chunk_off[E+1], pair_off[E+1], 16 scan sums (the
// per-item pad_off / counts are read from global memory).
constexpr int kPairTableInts = 2 * (kMaxExperts + 1) + 16;
constexpr int kPairBarriers = 2 * kOpStages + 2 * kSfStages + 2 * kTSlots + 3;
constexpr int kPairSmem = 1024 + kOpStages * kOpBytes + kSfStages * kSfBytes + kPairBarriers * 8 +
                          16 + kPairTableInts * 4;
static_assert(kPairSmem <= kSmemLimit, "shared memory");

// A work item as seen by CTA `rank`: its token chunk (2c + rank of the
// expert's chunks; rows <= 0 when the expert has no such chunk) and the
// pair of weight tiles n_pair.
struct PairItem {
  int e, n_pair, prow0, rows, npairs;
};

// Items are numbered expert-major, expert e owning items
// [pair_off[e] * n_pairs, pair_off[e + 1] * n_pairs), chunk pairs fastest
// (clusters running at the same time share an expert's weight tiles in L2).
__device__ __forceinline__ PairItem map_pair_item(const int* pair_off, const int* pad_off,
                                                  const int* counts, int E, int n_pairs, int item,
                                                  uint32_t rank) {
  int lo = 0, hi = E;  // pair_off[lo]*n_pairs <= item < pair_off[hi]*n_pairs
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (pair_off[mid] * n_pairs <= item) lo = mid; else hi = mid;
  }
  const int np = pair_off[lo + 1] - pair_off[lo];
  const int local = item - pair_off[lo] * n_pairs;
  const int chunk = 2 * (local % np) + static_cast<int>(rank);
  PairItem it;
  it.e = lo;
  it.n_pair = local / np;
  it.prow0 = pad_off[lo] + chunk * kRowBlock;
  it.rows = min(kRowBlock, counts[lo] - chunk * kRowBlock);
  it.npairs = np;
  return it;
}

__device__ __forceinline__ uint32_t a_box(int rows) {
  return rows <= 16 ? 0u : rows <= 32 ? 1u : rows <= 64 ? 2u : 3u;
}

// Walks this CTA's (item, K slice) sequence; `it` (and, in rank 0's
// producer, the peer's view `pe`) is mapped once per item.
struct Cursor {
  int item, kb;
  PairItem it, pe;
};

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ GemmMaps maps,
                         const __grid_constant__ GemmArgs args) {
  constexpr int FMT = kFmtNVFP4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sf_ring = smem + kOpStages * kOpBytes;
  uint64_t* full = reinterpret_cast<uint64_t*>(sf_ring + kSfStages * kSfBytes);  // rank 0's used
  uint64_t* empty = full + kOpStages;
  uint64_t* sfull = empty + kOpStages;
  uint64_t* sempty = sfull + kSfStages;
  uint64_t* tfree = sempty + kSfStages;
  uint64_t* sf_ready = tfree + kTSlots;       // rank 0's used: both CTAs' stagers
  uint64_t* tfull = sf_ready + kTSlots;
  uint64_t* tempty = tfull + 1;               // rank 0's used: both CTAs' epilogues
  uint64_t* drained = tempty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* t_chunk = reinterpret_cast<int*>(tmem_holder + 4);
  const int E = args.E;
  const int* t_pad = args.pad_off;
  const int* t_cnt = args.counts;
  int* t_pair = t_chunk + (E + 1);
  int* t_wsum = t_pair + (E + 1);
  pdl_launch_dependents();

  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kOpStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kSfStages; ++s) {
      mbar_init(&sfull[s], 1);
      mbar_init(&sempty[s], 4);
    }
    for (int s = 0; s < kTSlots; ++s) {
      mbar_init(&tfree[s], 1);
      mbar_init(&sf_ready[s], 8);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 16);
    mbar_init(drained, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(tmem_holder, kTmemCols);
    tmem_relinquish_pair();
  }
  if (threadIdx.x == 32 * 2 + 1) {
    for (int i = 0; i < 4; ++i) prefetch_tmap(&maps.a[i]);
    prefetch_tmap(&maps.b);
  }
  // Everything below reads what the previous kernels wrote.
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) t_chunk[i] = args.chunk_off[i];
  __syncthreads();
  {
    // pair_off: exclusive scan of the chunk pairs per expert (E <= 512 =
    // one value per thread)
    const int v =
        threadIdx.x < E ? (t_chunk[threadIdx.x + 1] - t_chunk[threadIdx.x] + 1) >> 1 : 0;
    int inc = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(0xFFFFFFFFu, inc, off);
      if (lane >= off) inc += o;
    }
    if (lane == 31) t_wsum[warp] = inc;
    __syncthreads();
    int add = 0;
    for (int w = 0; w < warp; ++w) add += t_wsum[w];
    if (threadIdx.x < E) t_pair[threadIdx.x] = inc - v + add;
    if (threadIdx.x == E - 1) t_pair[E] = inc + add;
  }
  tc_fence_before();
  __syncthreads();
  // both CTAs' barriers are initialised before either arrives on the other's
  cluster_sync();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int n_pairs = args.n_tiles;
  const int total = t_pair[E] * n_pairs;
  const int cluster = static_cast<int>(blockIdx.x >> 1), nclusters = static_cast<int>(gridDim.x >> 1);
  const int num_kb = args.num_kb;
  const int tile_rows = args.b_tile_bytes / 2048;  // rows of 2 KiB per weight tile (9)
  auto map_cursor = [&](Cursor& c, bool peer) {
    if (c.item >= total) return;
    c.it = map_pair_item(t_pair, t_pad, t_cnt, E, n_pairs, c.item, rank);
    if (peer) c.pe = map_pair_item(t_pair, t_pad, t_cnt, E, n_pairs, c.item, 1);
  };
  auto advance = [&](Cursor& c, bool peer) {
    if (++c.kb == num_kb) {
      c.kb = 0;
      c.item += nclusters;
      map_cursor(c, peer);
    }
  };
  // first 128-row weight tile of an item's pair; the second follows num_kb tiles later
  auto tile_index = [&](const PairItem& it) {
    return (static_cast<int64_t>(it.e) * n_pairs + it.n_pair) * 2 * num_kb;
  };

  const bool epi_warp = warp >= 4 && warp < 12;
  if (!epi_warp) {
    regs_release<kLeanRegs>();
    if (warp == 3) {
      // ------------------------------------------------ scale producer
      // the scale ring runs ahead of the operands by up to kSfStages stages
      // (its stages are released by the stagers, which wait for TMEM slots)
      if (lane == 0) {
        Cursor sc{cluster, 0, {}, {}};
        map_cursor(sc, false);
        int g_sf = 0;
        bool ok = true;
        while (sc.item < total) {
          const int s = g_sf % kSfStages;
          if (!mbar_wait(&sempty[s], ((g_sf / kSfStages) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          const PairItem& it = sc.it;
          const bool has_a = it.rows > 0;
          const int64_t t0 = tile_index(it);
          const uint8_t* w0 =
              args.b_tiles + (t0 + sc.kb) * static_cast<int64_t>(args.b_tile_bytes) + kTileBytes;
          const uint8_t* w1 = w0 + static_cast<int64_t>(num_kb) * args.b_tile_bytes;
          uint8_t* sp = sf_ring + s * kSfBytes;
          mbar_arrive_expect_tx(&sfull[s], (has_a ? 4u * 512u : 0u) + 2u * 4u * 512u);
          if (has_a)
            bulk_load(sp, args.sfa + (static_cast<int64_t>(it.prow0 >> 7) * args.sfa_tiles_k +
                                      sc.kb * 4) * 512,
                      4 * 512, &sfull[s]);
          bulk_load(sp + kSfOffB, w0, 4 * 512, &sfull[s]);
          bulk_load(sp + kSfOffB + 4 * 512, w1, 4 * 512, &sfull[s]);
          ++g_sf;
          advance(sc, false);
        }
        // no copy this thread issued may still be in flight when it leaves
        for (int back = 1; back <= kSfStages && back <= g_sf; ++back) {
          const int idx = g_sf - back;
          mbar_wait(&sfull[idx % kSfStages], static_cast<uint32_t>((idx / kSfStages) & 1), nullptr);
        }
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (warp == 2) {
      // ------------------------------------------------ operand producer
      if (lane == 0) {
        const uint64_t once = l2_policy_evict_first();
        const uint64_t reused = l2_policy_evict_normal();
        // activation tiles are read again by the expert's other weight tiles
        const uint64_t act_policy = reused;
        const uint32_t full_lead = mapa_shared(smem_u32(full), 0);  // rank 0's full[0]
        Cursor op{cluster, 0, {}, {}};
        map_cursor(op, lead);
        int g_op = 0, skipped = -1;
        bool ok = true;
        while (op.item < total) {
          const int s = g_op % kOpStages;
          if (!mbar_wait(&empty[s], ((g_op / kOpStages) & 1) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          if (args.test_stall && blockIdx.x == 0 && skipped < 0) {
            // fault injection: this stage's operands never arrive
            skipped = g_op++;
            advance(op, lead);
            continue;
          }
          const PairItem& it = op.it;
          // weights read by several chunk pairs stay in L2 for the later ones
          const uint64_t policy = it.npairs > 1 ? reused : once;
          if (lead) {
            // rank 0's barrier counts both CTAs' operand bytes
            const PairItem& pe = op.pe;
            const uint32_t bytes = 2u * kTileBytes +
                                   (it.rows > 0 ? (16u << a_box(it.rows)) * 128u : 0u) +
                                   (pe.rows > 0 ? (16u << a_box(pe.rows)) * 128u : 0u);
            mbar_arrive_expect_tx(&full[s], bytes);
          }
          uint8_t* sp = smem + s * kOpBytes;
          const uint32_t bar = full_lead + s * 8;
          if (it.rows > 0)
            tma_load_2d_pair(sp, &maps.a[a_box(it.rows)], bar, op.kb * 128, it.prow0, act_policy);
          const int64_t tile = tile_index(it) + static_cast<int64_t>(rank) * num_kb + op.kb;
          tma_load_2d_pair(sp + kTileBytes, &maps.b, bar, 0, static_cast<int32_t>(tile * tile_rows),
                           policy);
          ++g_op;
          advance(op, lead);
        }
        // rank 0's barriers count the operand copies of both CTAs: once they
        // have all completed, no copy of either CTA is still in flight
        if (lead)
          for (int back = 1; back <= kOpStages && back <= g_op; ++back) {
            const int idx = g_op - back;
            if (idx == skipped) continue;
            mbar_wait(&full[idx % kOpStages], static_cast<uint32_t>((idx / kOpStages) & 1),
                      nullptr);
          }
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer (rank 0)
      if (lane == 0 && lead) {
        const uint32_t idesc = idesc_nvf4(256, 256);
        const uint64_t desc0 = desc_sw128(smem_u32(smem));  // stage 0's activation tile
        const uint32_t sf0 = tmem + kSfColBase;
        int s = 0, slot = 0, local = 0;
        uint32_t oph = 0, sph = 0;
        bool ok = true;
        for (int item = cluster; item < total && ok; item += nclusters, ++local) {
          if (!mbar_wait(tempty, (static_cast<uint32_t>(local) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&sf_ready[slot], sph, abort_flag) ||
                !mbar_wait(&full[s], oph, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            // descriptors of stage s: start address (16-byte units) in the low bits
            const uint64_t da = desc0 + static_cast<uint64_t>(s * (kOpBytes >> 4));
            const uint64_t db = da + (kTileBytes >> 4);
            const uint32_t sf_col = sf0 + slot * kPSfCols;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_nvf4_pair(tmem, da + 2 * j, db + 2 * j, idesc, sf_col + 32 + j * 4,
                            sf_col + j * 8, (kb | j) != 0);
            tc_commit_pair(&empty[s], 3);
            tc_commit_pair(&tfree[slot], 3);
            if (++s == kOpStages) {
              s = 0;
              oph ^= 1u;
            }
            if (++slot == kTSlots) {
              slot = 0;
              sph ^= 1u;
            }
          }
          if (ok) tc_commit_pair(tfull, 3);
        }
        // both CTAs free TMEM (and the peer leaves its shared memory) only
        // once every MMA has completed
        tc_commit_pair(drained, 3);
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (warp >= 12) {
      // ------------------------------------------------ scale stagers
      // Warp w writes TMEM lane quarter q = w % 4 of a scale slot: both weight
      // tiles' scales (every quarter holds all 256 rows') and its own 32
      // activation rows' scales, once the slot's previous MMAs have finished,
      // then releases the smem scale stage and reports the slot to rank 0.
      const int q = warp & 3;
      Cursor sc{cluster, 0, {}, {}};
      map_cursor(sc, false);
      int g = 0;
      bool ok = true;
      while (sc.item < total) {
        const int s = g % kSfStages, slot = g % kTSlots;
        const bool ready = mbar_wait(&sfull[s], (g / kSfStages) & 1, abort_flag) &&
                           mbar_wait(&tfree[slot], ((g / kTSlots) & 1) ^ 1u, abort_flag);
        if (!__all_sync(0xFFFFFFFFu, ready)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const PairItem& it = sc.it;
        const uint8_t* sp = sf_ring + s * kSfBytes;
        uint32_t v[32];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint4 b0 = *reinterpret_cast<const uint4*>(sp + kSfOffB + j * 512 + lane * 16);
          const uint4 b1 =
              *reinterpret_cast<const uint4*>(sp + kSfOffB + (4 + j) * 512 + lane * 16);
          v[8 * j + 0] = b0.x;
          v[8 * j + 1] = b0.y;
          v[8 * j + 2] = b0.z;
          v[8 * j + 3] = b0.w;
          v[8 * j + 4] = b1.x;
          v[8 * j + 5] = b1.y;
          v[8 * j + 6] = b1.z;
          v[8 * j + 7] = b1.w;
        }
        uint32_t a4[4];
#pragma unroll
        for (int j = 0; j < 4; ++j)
          a4[j] = it.rows > 0
                      ? *reinterpret_cast<const uint32_t*>(sp + j * 512 + lane * 16 + q * 4)
                      : 0u;
        const uint32_t col =
            tmem + (static_cast<uint32_t>(q * 32) << 16) + kSfColBase + slot * kPSfCols;
        tmem_st32(col, v);
#pragma unroll
        for (int j = 0; j < 4; ++j) tmem_st1(col + 32 + 4 * j + q, a4[j]);
        tmem_st_wait();
        // the smem scale stage has been read (its values are in TMEM now);
        // the next bulk copy into it is an async-proxy write after these
        // generic-proxy reads
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(&sempty[s]);
          mbar_arrive_cluster(&sf_ready[slot], 0);
        }
        ++g;
        advance(sc, false);
      }
      if (!ok && lane == 0) report_status(args.status, kStatusTimeout);
    }
  } else {
    regs_claim<kEpiRegs>();
    // ------------------------------------------------ epilogue warps
    // Warp w reads TMEM lane quarter w % 4 (this CTA's rows 32q..) of
    // accumulator column group (w - 4) / 4 (one 128-column group per weight
    // tile of the pair).
    const int q = warp & 3;
    const int grp = (warp - 4) >> 2;
    int local = 0;
    for (int item = cluster; item < total; item += nclusters, ++local) {
      const PairItem it = map_pair_item(t_pair, t_pad, t_cnt, E, n_pairs, item, rank);
      if (!mbar_wait(tfull, static_cast<uint32_t>(local) & 1u, abort_flag)) {
        if (lane == 0) report_status(args.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const int r = q * 32 + lane;
      const bool active = q * 32 < it.rows;
      const uint32_t taddr = tmem + (static_cast<uint32_t>(q * 32) << 16) + grp * 128;
      const int64_t prow = it.prow0 + r;
      const int64_t orow = args.out_rows_per_expert
                               ? static_cast<int64_t>(it.e) * args.out_rows_per_expert +
                                     (it.prow0 - t_pad[it.e]) + r
                               : prow;
      const int n128 = it.n_pair * 2 + grp;
      uint32_t v[128];
      if (active) {
        epilogue_load<EPI>(taddr, 0, v);
        epilogue_load<EPI>(taddr, 1, v + 64);
        tmem_ld_wait();
        epilogue_fence(v);
        epilogue_fence(v + 64);
      }
      // the accumulator is free for the pair's next MMAs from here on
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive_cluster(tempty, 0);
      if (active) {
        uint32_t carry[5];
        epilogue_round<FMT, EPI>(v, 0, r < it.rows, prow, orow, n128, args, carry);
        epilogue_round<FMT, EPI>(v + 64, 1, r < it.rows, prow, orow, n128, args, carry);
        if (EPI == 2 && args.gather_inv) combine_fused(r < it.rows, prow, n128, args);
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && lane == 0) mbar_wait(drained, 0, nullptr);
  __syncthreads();
  // neither CTA leaves while the other may still arrive on its barriers or
  // read its shared memory
  cluster_sync();
  tc_fence_after();
  if (warp == 1) tmem_dealloc_pair(tmem, kTmemCols);
}

template <int EPI>
bool& pair_split_checked() {
  static bool ok = false;
  return ok;
}

template <int EPI>
cudaError_t pair_prepare_one(int* max_clusters) {
  auto k = moe_gemm_pair_kernel<EPI>;
  cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, kPairSmem);
  if (e != cudaSuccess) return e;
  // the register split balances only at kSplitLaunchRegs registers per
  // thread; with fewer, the claiming warpgroups would wait forever
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, k);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kSplitLaunchRegs) return cudaErrorInvalidConfiguration;
  cudaLaunchConfig_t cfg{};
  cfg.gridDim = dim3(2);
  cfg.blockDim = dim3(kPairThreads);
  cfg.dynamicSmemBytes = kPairSmem;
  int n = 0;
  e = cudaOccupancyMaxActiveClusters(&n, k, &cfg);
  if (e != cudaSuccess) return e;
  if (n < 1) return cudaErrorInvalidConfiguration;
  *max_clusters = *max_clusters ? min(*max_clusters, n) : n;
  pair_split_checked<EPI>() = true;
  return cudaSuccess;
}

}  // namespace

cudaError_t gemm_pair_prepare(int* max_clusters) {
  int n = 0;
  cudaError_t e = pair_prepare_one<1>(&n);
  if (e == cudaSuccess) e = pair_prepare_one<2>(&n);
  if (e == cudaSuccess) e = pair_prepare_one<3>(&n);
  if (e == cudaSuccess) *max_clusters = n;
  return e;
}

cudaError_t launch_gemm_pair(int epi, const GemmMaps& maps, const GemmArgs& args, int clusters,
                             cudaStream_t s) {
  auto k = epi == 1 ? moe_gemm_pair_kernel<1> : epi == 3 ? moe_gemm_pair_kernel<3>
                                                         : moe_gemm_pair_kernel<2>;
  const bool checked = epi == 1 ? pair_split_checked<1>() : epi == 3 ? pair_split_checked<3>()
                                                                     : pair_split_checked<2>();
  if (!checked || clusters < 1) return cudaErrorInvalidConfiguration;
  return launch_pdl(g_pdl_gemm, k, dim3(2 * clusters), dim3(kPairThreads), kPairSmem, s, maps,
                    args);
}

}  // namespace moe
