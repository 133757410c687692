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
//   warp 2      producer: this CTA's activation slice (TMA) + scales, its
//               weight tile's codes, both weight tiles' scales (bulk copies);
//   warp 1      rank 0: issues the pair MMAs; both ranks: TMEM alloc/free;
//   warps 4-11  epilogue of this CTA's 128 rows x 256 columns;
//   warps 12-15 scale stagers: write the stage's scales into this CTA's
//               TMEM (tcgen05.st), then arrive on rank 0's stage barrier.
// Rank 0's MMA thread waits until both CTAs' stagers have released a stage
// (8 arrivals, 4 of them from the peer), issues four MMAs and commits to the
// stage's empty barrier in both CTAs; accumulator-full is committed to both
// CTAs, accumulator-empty counts the 16 epilogue warps of both.
#include "gemm_common.cuh"

namespace moe {

namespace {

constexpr int kPairStages = 4;
constexpr int kPairThreads = 512;
// Stage layout (per CTA): activation codes (128 rows x 128 bytes), this
// CTA's weight tile codes, the scale tiles of both weight tiles (4 x 512
// bytes each), the activation scale tiles (4 x 512 bytes).
constexpr int kPOffB = 128 * 128;
constexpr int kPOffBsf = kPOffB + kTileBytes;
constexpr int kPOffAsf = kPOffBsf + 2 * 4 * 512;
constexpr int kPStageBytes = (kPOffAsf + 4 * 512 + 1023) / 1024 * 1024;
// TMEM columns per stage: weight scales of substep j at 8j..8j+7 (tile 0 at
// 8j..8j+3, tile 1 at 8j+4..8j+7), activation scales of lane quarter q at
// 32 + 4j + q.
constexpr int kPSfCols = 64;
static_assert(kSfColBase + kPairStages * kPSfCols <= kTmemCols, "TMEM scale columns");
// Tables: chunk_off[E+1], pad_off[E], counts[E], pair_off[E+1], 16 scan sums.
constexpr int kPairTableInts = 4 * (kMaxExperts + 1) + 16;
constexpr int kPairBarriers = 3 * kPairStages + 3;
constexpr int kPairSmem =
    1024 + kPairStages * kPStageBytes + kPairBarriers * 8 + 16 + kPairTableInts * 4;
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

template <int EPI>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(kPairThreads, 1)
    moe_gemm_pair_kernel(const __grid_constant__ GemmMaps maps,
                         const __grid_constant__ GemmArgs args) {
  constexpr int FMT = kFmtNVFP4;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kPairStages * kPStageBytes);
  uint64_t* empty = full + kPairStages;
  uint64_t* sf_ready = empty + kPairStages;  // used in rank 0: both CTAs' stagers
  uint64_t* tfull = sf_ready + kPairStages;
  uint64_t* tempty = tfull + 1;              // used in rank 0: both CTAs' epilogues
  uint64_t* drained = tempty + 1;
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(drained + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* t_chunk = reinterpret_cast<int*>(tmem_holder + 4);
  const int E = args.E;
  int* t_pad = t_chunk + (E + 1);
  int* t_cnt = t_pad + E;
  int* t_pair = t_cnt + E;
  int* t_wsum = t_pair + (E + 1);
  pdl_launch_dependents();

  const uint32_t rank = cluster_ctarank();
  const bool lead = rank == 0;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kPairStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
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
  if (threadIdx.x == 32 * 2 + 1)
    for (int i = 0; i < 4; ++i) prefetch_tmap(&maps.a[i]);
  // Everything below reads what the previous kernels wrote.
  pdl_wait();
  for (int i = threadIdx.x; i <= E; i += blockDim.x) t_chunk[i] = args.chunk_off[i];
  for (int i = threadIdx.x; i < E; i += blockDim.x) {
    t_pad[i] = args.pad_off[i];
    t_cnt[i] = args.counts[i];
  }
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

  const bool epi_warp = warp >= 4 && warp < 12;
  if (!epi_warp) {
    regs_release<kLeanRegs>();
    if (warp == 2) {
      // ------------------------------------------------ producer
      if (lane == 0) {
        const uint64_t once = l2_policy_evict_first();
        const uint64_t reused = l2_policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0;
        int slots = 0;
        int skipped = -1;
        bool ok = true;
        for (int item = cluster; item < total && ok; item += nclusters) {
          const PairItem it = map_pair_item(t_pair, t_pad, t_cnt, E, n_pairs, item, rank);
          const bool has_a = it.rows > 0;
          const int amap = it.rows <= 16 ? 0 : it.rows <= 32 ? 1 : it.rows <= 64 ? 2 : 3;
          // weights read by several chunk pairs stay in L2 for the later ones
          const uint64_t policy = it.npairs > 1 ? reused : once;
          const uint32_t bytes =
              (has_a ? (16u << amap) * 128u + 4u * 512u : 0u) + kTileBytes + 2u * 4u * 512u;
          const uint8_t* sfa =
              args.sfa + static_cast<int64_t>(it.prow0 >> 7) * args.sfa_tiles_k * 512;
          const uint8_t* tile0 =
              args.b_tiles + (static_cast<int64_t>(it.e) * n_pairs + it.n_pair) * 2 * num_kb *
                                 args.b_tile_bytes;
          const uint8_t* tile1 = tile0 + static_cast<int64_t>(num_kb) * args.b_tile_bytes;
          const uint8_t* own = rank ? tile1 : tile0;
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            if (args.test_stall && blockIdx.x == 0 && skipped < 0) {
              // fault injection: nothing ever completes this stage
              skipped = slots++;
              if (++stage == kPairStages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            uint8_t* sp = smem + stage * kPStageBytes;
            const int64_t woff = static_cast<int64_t>(kb) * args.b_tile_bytes;
            mbar_arrive_expect_tx(&full[stage], bytes);
            if (has_a) {
              tma_load_2d(sp, &maps.a[amap], &full[stage], kb * 128, it.prow0);
              bulk_load(sp + kPOffAsf, sfa + kb * 4 * 512, 4 * 512, &full[stage]);
            }
            bulk_load_hint(sp + kPOffB, own + woff, kTileBytes, &full[stage], policy);
            bulk_load_hint(sp + kPOffBsf, tile0 + woff + kTileBytes, 4 * 512, &full[stage], policy);
            bulk_load_hint(sp + kPOffBsf + 4 * 512, tile1 + woff + kTileBytes, 4 * 512,
                           &full[stage], policy);
            ++slots;
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // no copy this thread issued may still be in flight when it leaves
        for (int back = 1; back <= kPairStages && back <= slots; ++back) {
          const int idx = slots - back;
          if (idx == skipped) continue;
          mbar_wait(&full[idx % kPairStages], static_cast<uint32_t>((idx / kPairStages) & 1),
                    nullptr);
        }
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer (rank 0)
      if (lane == 0 && lead) {
        const uint32_t idesc = idesc_nvf4(256, 256);
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int item = cluster; item < total && ok; item += nclusters, ++local) {
          if (!mbar_wait(tempty, (static_cast<uint32_t>(local) & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          for (int kb = 0; kb < num_kb; ++kb) {
            if (!mbar_wait(&sf_ready[stage], phase, abort_flag)) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint8_t* sp = smem + stage * kPStageBytes;
            const uint32_t a_addr = smem_u32(sp), b_addr = smem_u32(sp + kPOffB);
            const uint32_t sf_col = tmem + kSfColBase + stage * kPSfCols;
#pragma unroll
            for (int j = 0; j < 4; ++j)
              mma_nvf4_pair(tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                            sf_col + 32 + j * 4, sf_col + j * 8, (kb | j) != 0);
            tc_commit_pair(&empty[stage], 3);
            if (++stage == kPairStages) {
              stage = 0;
              phase ^= 1u;
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
      // Warp w writes TMEM lane quarter q = w % 4 of each stage's scale
      // columns: both weight tiles' scales (every quarter holds all 256
      // rows') and its own 32 activation rows' scales, then releases the
      // stage to rank 0's MMA thread.
      const int q = warp & 3;
      int stage = 0;
      uint32_t phase = 0;
      bool ok = true;
      for (int item = cluster; item < total && ok; item += nclusters) {
        const PairItem it = map_pair_item(t_pair, t_pad, t_cnt, E, n_pairs, item, rank);
        const bool has_a = it.rows > 0;
        for (int kb = 0; kb < num_kb; ++kb) {
          const bool landed = mbar_wait(&full[stage], phase, abort_flag);
          if (!__all_sync(0xFFFFFFFFu, landed)) {
            ok = false;
            break;
          }
          const uint8_t* sp = smem + stage * kPStageBytes;
          uint32_t v[32];
#pragma unroll
          for (int j = 0; j < 4; ++j) {
            const uint4 b0 = *reinterpret_cast<const uint4*>(sp + kPOffBsf + j * 512 + lane * 16);
            const uint4 b1 =
                *reinterpret_cast<const uint4*>(sp + kPOffBsf + (4 + j) * 512 + lane * 16);
            v[8 * j + 0] = b0.x;
            v[8 * j + 1] = b0.y;
            v[8 * j + 2] = b0.z;
            v[8 * j + 3] = b0.w;
            v[8 * j + 4] = b1.x;
            v[8 * j + 5] = b1.y;
            v[8 * j + 6] = b1.z;
            v[8 * j + 7] = b1.w;
          }
          const uint32_t col =
              tmem + (static_cast<uint32_t>(q * 32) << 16) + kSfColBase + stage * kPSfCols;
          tmem_st32(col, v);
#pragma unroll
          for (int j = 0; j < 4; ++j)
            tmem_st1(col + 32 + 4 * j + q,
                     has_a ? *reinterpret_cast<const uint32_t*>(sp + kPOffAsf + j * 512 +
                                                                lane * 16 + q * 4)
                           : 0u);
          tmem_st_wait();
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive_cluster(&sf_ready[stage], 0);
          if (++stage == kPairStages) {
            stage = 0;
            phase ^= 1u;
          }
        }
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
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  if (warp == 1 && lane == 0) mbar_wait(drained, 0, nullptr);
  __syncthreads();
  // neither CTA leaves while the other may still arrive on its barriers
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
