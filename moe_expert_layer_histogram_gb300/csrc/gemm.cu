// gemm.cu -- grouped expert GEMMs on the sm_103a tensor cores (tcgen05).
//
// GEMM1 (W13) and GEMM2 (W2) of the layer: for every expert e with rows
// [pad_off[e], pad_off[e] + count[e]) of the permuted activations,
//   C = A_rows x W_e^T   (fp32 accumulation),
// with A and W in BF16, MXFP8 (e4m3, e8m0 per 32) or NVFP4 (e2m1, e4m3 per
// 16, global scale folded in); the block-scaled MMA applies both operands'
// scales.  GEMM1's epilogue applies SwiGLU with the optional gate/up clamp
// (or the non-gated squared ReLU) and re-quantises the result into GEMM2's
// input format; GEMM2's epilogue stores bf16 (or, with the in-kernel
// reduce, adds the weighted rows into an fp32 accumulator).  (The two expert
// GEMMs with SwiGLU between them: PR #40082 report, sec. 实现拆解 item 1.)
//
// Structure: one persistent CTA per SM walks the device-built work list
// (expert, weight tile(s), 128-row token chunk), expert-major.  Warp 2 (one
// thread) streams 128-byte K slices into a shared-memory ring (4-8 stages):
// the activation tile by TMA (box height = the chunk's real rows, rounded
// up to 16/32/64/128) plus its scale tiles, and each pre-swizzled weight
// tile with its scales by bulk copy.  Stage layout: A codes (MROWS x 128
// bytes), B codes (NW x 16 KiB), B scales, A scales.  The MMA always reads
// 128 A rows; rows past the region only feed accumulator rows that are
// never stored.  Warp 1 (one thread) owns TMEM: it copies the scale tiles
// into TMEM (tcgen05.cp) and issues 128 x (128 NW) tcgen05.mma into an fp32
// accumulator (two of 128 columns, or one of 256 for wide items).  For decode
// chunks warp 0 writes the scales with tcgen05.st instead.  Wide NVFP4 items
// keep their scale tiles in a ring of their own that warp 3 fills ahead of
// the operands; four stager warps (12-15, one per TMEM lane quarter) write a
// stage's scales into TMEM as soon as the stage's previous MMAs are done and
// report on the stage's full barrier, so the MMA thread waits once per stage
// and the staging overlaps the operand copies.  At N = 256 a K slice takes
// the MMA thread about as long as its wait, four MMA issues, commit and
// loop (measured ~700 cycles; the tensor pipe alone needs 524), and moves
// about 127 KB through the SM's shared memory (54 KB of copies, 48 KB of MMA
// operand reads, the stagers' scale reads), about 490 ns at 128 bytes per
// clock: both limits sit near the measured ~480 ns per slice.
// The epilogue warps (3.., or 4-11 in the 16-warp wide NVFP4 kernel) drain
// the accumulator (tcgen05.ld), run the epilogue and store, each thread one
// row, in whole 32-byte sectors and marked L2 evict-first.  The token tile is the
// MMA's M (only the chunk's real rows are loaded and stored) and the weight
// tile its N, so decode-sized chunks cost no extra weight traffic.  Decode
// launches (T <= 16) run GEMM1 and GEMM2 in one persistent launch (FUSED).
#include <cuda_bf16.h>

#include "gemm_common.cuh"

namespace moe {

namespace {

// Warp 0 stages decode scales into TMEM lane quarter 0, warp 1 issues the
// MMAs, warp 2 the copies, then four epilogue warps per 128-column group.
// Wide NVFP4 items add four scale-stager warps (warps 12-15, one per TMEM
// lane quarter) and start the epilogue warps at warp 4, so that every
// warpgroup has one role and one register budget: warps 0-3 and 12-15 keep
// kLeanRegs registers, the epilogue warpgroups (which hold a 128-column
// accumulator slice in registers) kEpiRegs.
__host__ __device__ constexpr bool wide_stager(int fmt, int nw) {
  return fmt == kFmtNVFP4 && nw == 2;
}
__host__ __device__ constexpr int gemm_threads(int fmt, int nw) {
  return wide_stager(fmt, nw) ? 512 : 96 + 128 * nw;
}

// Dynamic shared memory of a kernel instance: the wide NVFP4 kernel adds the
// scale ring's barriers (its slots take the bytes the stages no longer hold).
template <int FMT, int MROWS, int NW>
__host__ __device__ constexpr int gemm_smem() {
  return smem_bytes<FMT, MROWS, NW>() +
         (wide_stager(FMT, NW) ? 2 * num_stages<FMT, MROWS, NW>() * 8 : 0);
}
static_assert(gemm_smem<kFmtNVFP4, 128, 2>() <= kSmemLimit, "wide NVFP4 shared memory");

// ---------------------------------------------------------------- kernel
// FUSED (decode): one launch runs GEMM1's items (args/maps) and then
// GEMM2's (args2/maps2).  Each CTA finishes issuing its GEMM1 items before
// its GEMM2 items; a GEMM2 item of expert e waits (bounded) until every
// GEMM1 item of expert e has stored its output, counted in args.done1[e] by
// each epilogue warp.  CTAs whose GEMM1 share ends early move on to GEMM2
// work instead of idling until the slowest CTA finishes.
template <int FMT, int EPI, int MROWS, int NW, bool FUSED>
__global__ void __launch_bounds__(gemm_threads(FMT, NW), 1)
    moe_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ GemmArgs args,
                    const __grid_constant__ GemmMaps maps2,
                    const __grid_constant__ GemmArgs args2) {
  constexpr int SFT = Fmt<FMT>::kSfTiles;
  constexpr int SB = stage_bytes<FMT, MROWS, NW>();
  constexpr int kStages = num_stages<FMT, MROWS, NW>();
  constexpr int A_BYTES = MROWS * 128;
  constexpr int kAccCols = Wide<NW>::kAccCols;
  constexpr int kBufs = Wide<NW>::kBufs;
  constexpr int kSfColsPerStage = Wide<NW>::kSfCols;
  constexpr bool WS = wide_stager(FMT, NW);
  constexpr int kEpiWarp0 = WS ? 4 : 3;  // first epilogue warp
  // Shared-memory offsets inside a stage (A codes, B codes, B scale tiles,
  // A scale tiles).  Wide NVFP4 kernels keep the scale tiles in a ring of
  // their own (SBO: operand stage bytes; the scale ring follows the operand
  // stages, one slot per stage, the same bytes in total), filled ahead of
  // the operands by warp 3, so that writing a stage's scales into TMEM is
  // done by the time its operands land.
  constexpr int SBO = WS ? A_BYTES + NW * kTileBytes : SB;
  constexpr int kOffBsf = WS ? 0 : A_BYTES + NW * kTileBytes;  // weight scale tiles
  constexpr int kOffAsf = kOffBsf + NW * SFT * 512;              // activation scale tiles
  constexpr int kSfSlot = (NW + 1) * SFT * 512;                  // scale ring slot (WS)
  static_assert(!WS || SBO + kSfSlot == SB, "wide stage layout");
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  uint8_t* sring = smem + kStages * SBO;  // WS: scale ring
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + kStages * SB);
  uint64_t* empty = full + kStages;
  uint64_t* tfull = empty + kStages;
  uint64_t* tempty = tfull + 2;
  uint64_t* drained = tempty + 2;
  uint64_t* sf_ready = drained + 1;  // [kStages] scales of the stage are in TMEM
  uint64_t* sfull = sf_ready + kStages;   // WS: [kStages] scale ring slot landed
  uint64_t* sempty = sfull + kStages;     // WS: [kStages] scale ring slot read
  uint32_t* tmem_holder = reinterpret_cast<uint32_t*>(sf_ready + kStages + (WS ? 2 * kStages : 0));
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_holder + 1);
  int* s_tab = reinterpret_cast<int*>(tmem_holder + 4);
  const Tables tab{s_tab, s_tab + (args.E + 1), s_tab + (2 * args.E + 1),
                   NW == 2 && args.order ? s_tab + (3 * args.E + 1) : nullptr};
  pdl_launch_dependents();

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      // WS with stagers: the stage's operand bytes and the four stager
      // warps' reports that its scales are in TMEM
      mbar_init(&full[s], WS && args.stage_scales ? 5 : 1);
      mbar_init(&empty[s], 1);
      mbar_init(&sf_ready[s], 1);
      if constexpr (WS) {
        mbar_init(&sfull[s], 1);
        mbar_init(&sempty[s], args.stage_scales ? 4 : 1);
      }
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], 4 * NW);  // every epilogue warp releases the accumulator
    }
    mbar_init(drained, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 1) {
    tmem_alloc(tmem_holder, kTmemCols);
    tmem_relinquish();
  }
  if (threadIdx.x == 32 * 2 + 1)
    for (int i = 0; i < 4; ++i) prefetch_tmap(&maps.a[i]);
  // Everything below reads what the previous kernels wrote.
  pdl_wait();
  for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_tab[i] = args.chunk_off[i];
  for (int i = threadIdx.x; i < args.E; i += blockDim.x) {
    s_tab[args.E + 1 + i] = args.pad_off[i];
    s_tab[2 * args.E + 1 + i] = args.counts[i];
  }
  if (NW == 2 && args.order)
    for (int i = threadIdx.x; i <= args.E; i += blockDim.x) s_tab[3 * args.E + 1 + i] = args.order[i];
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_holder;
  const int n1 = tab.chunk_off[args.E] * args.n_tiles;  // GEMM1 (or the only GEMM) items
  const int total = FUSED ? n1 + tab.chunk_off[args.E] * args2.n_tiles : n1;
  // item -> (GEMM, item within it)
  auto second = [&](int item) { return FUSED && item >= n1; };
  auto local_item = [&](int item) { return second(item) ? item - n1 : item; };
  auto gargs = [&](int item) -> const GemmArgs& { return second(item) ? args2 : args; };
  // Decode launches: a chunk of at most 32 rows keeps all its real
  // accumulator rows in TMEM lane quarter 0, and the MMA of each lane quarter
  // reads both operands' scales from that quarter's own lanes, so such a
  // chunk needs its stage's scales in lanes 0-31 only.  Warp 0 (the quarter-0
  // warp) writes just those lanes from shared memory with tcgen05.st (4 KiB
  // per stage instead of the 16 KiB a broadcast tcgen05.cp writes), off the
  // tensor pipe; every stage of such a launch then reaches the MMA through
  // warp 0's sf_ready barrier.
  const bool staged = NW == 1 && SFT > 0 && args.pair_scale_copies && args.stage_scales;
  // Wide NVFP4 items: warps 12-15 write every stage's scales into their lane
  // quarters with tcgen05.st (the activation scales of quarter q in one
  // column per 64-element substep, the weight scales replicated in every
  // quarter) instead of the MMA thread broadcasting twelve tiles with
  // tcgen05.cp, which queue in order with the MMAs on the tensor pipe
  // (measured: twelve copies per K slice take a 128 x 256 x 256 slice from
  // 262 to 483 ns of tensor-pipe time; staged scales leave it at the MMAs').
  const bool wstaged = WS && args.stage_scales;

  // Roles by warpgroup: a warpgroup's register budget changes at the top of
  // its branch, before any of its roles' code.
  const bool epi_warp = warp >= kEpiWarp0 && warp < kEpiWarp0 + 4 * NW;
  if (!epi_warp) {
    if constexpr (WS) regs_release<kLeanRegs>();
    if (warp == 0) {
      // ------------------------------------------------ scale stager
      if (staged) {
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
          const GemmArgs& A = gargs(item);
          const bool q0 = map_item<NW == 2>(tab, args.E, A.n_tiles, local_item(item)).rows <= 32;
          for (int kb = 0; kb < A.num_kb; ++kb) {
            const bool landed = mbar_wait(&full[stage], phase, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, landed)) {
              ok = false;
              break;
            }
            if (q0) {
              const uint8_t* sp = smem + stage * SB;
              const uint32_t col = tmem + kSfColBase + stage * kSfColsPerStage;  // lanes 0-31
              if constexpr (FMT == kFmtNVFP4) {
                // per 64-element substep j: activation row (lane) scales in
                // column 8j, the 128 weight rows' scales in columns 8j+4..8j+7
                uint32_t v[32];
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint4 b =
                      *reinterpret_cast<const uint4*>(sp + kOffBsf + j * 512 + lane * 16);
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
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&sf_ready[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok && lane == 0) report_status(args.status, kStatusTimeout);
      }
    } else if (warp == 2) {
      // ------------------------------------------------ TMA producer
      if (lane == 0) {
        // A weight tile is read once per chunk of its expert: experts with a
        // single chunk (every decode expert) read it once, so it is evicted
        // first; wide (prefill) launches keep multi-chunk experts' tiles
        // evict-normal for the later chunks.
        const uint64_t once = l2_policy_evict_first();
        const uint64_t reused = NW == 2 ? l2_policy_evict_normal() : once;
        int stage = 0;
        uint32_t phase = 0;
        int slots = 0;          // ring positions used so far
        int skipped = -1;       // position the test hook left unloaded
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
          const GemmArgs& A = gargs(item);
          const CUtensorMap* amaps = second(item) ? maps2.a : maps.a;
          const Item it = map_item<NW == 2>(tab, args.E, A.n_tiles, local_item(item));
          const int amap = it.rows <= 16 ? 0 : it.rows <= 32 ? 1 : it.rows <= 64 ? 2 : 3;
          if ((16 << amap) > MROWS) {   // the host bounded the rows per chunk by MROWS
            ok = false;
            break;
          }
          if (second(item)) {
            // GEMM2's activations are GEMM1's output for this expert
            const int need = 4 * args.n_tiles * (tab.chunk_off[it.k + 1] - tab.chunk_off[it.k]);
            if (!wait_count_at_least(args.done1 + it.e, need, abort_flag)) {
              ok = false;
              break;
            }
            fence_proxy_async_global();  // generic-proxy stores -> the TMA reads below
          }
          const uint64_t policy =
              tab.chunk_off[it.k + 1] - tab.chunk_off[it.k] > 1 ? reused : once;
          // WS: operand codes only (the scale ring carries the scale tiles)
          const uint32_t bytes = WS ? (16u << amap) * 128u + NW * kTileBytes
                                    : (16u << amap) * 128u + NW * A.b_tile_bytes + SFT * 512u;
          const uint8_t* sfa = A.sfa + static_cast<int64_t>(it.prow0 >> 7) * A.sfa_tiles_k * 512;
          // the item's first 128-row weight tile; the next one (NW = 2)
          // follows num_kb tiles later
          const uint8_t* btile =
              A.b_tiles + (static_cast<int64_t>(it.e) * A.n_tiles + it.n_tile) * NW * A.num_kb *
                              A.b_tile_bytes;
          for (int kb = 0; kb < A.num_kb; ++kb) {
            if (!mbar_wait(&empty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            if (A.test_stall && blockIdx.x == 0 && skipped < 0) {
              // test hook: nothing ever completes this stage
              skipped = slots++;
              if (++stage == kStages) {
                stage = 0;
                phase ^= 1u;
              }
              continue;
            }
            uint8_t* sp = smem + stage * SBO;
            mbar_arrive_expect_tx(&full[stage], bytes);
            tma_load_2d(sp, &amaps[amap], &full[stage], kb * 128, it.prow0);
            if constexpr (NW == 1) {
              // weight tile codes + its scale tiles: one contiguous block
              bulk_load_hint(sp + A_BYTES, btile + static_cast<int64_t>(kb) * A.b_tile_bytes,
                             A.b_tile_bytes, &full[stage], policy);
            } else {
              // codes of both tiles back to back (one 256-row operand), then
              // their scale tiles
#pragma unroll
              for (int w = 0; w < NW; ++w) {
                const uint8_t* src =
                    btile + (static_cast<int64_t>(w) * A.num_kb + kb) * A.b_tile_bytes;
                bulk_load_hint(sp + A_BYTES + w * kTileBytes, src, kTileBytes, &full[stage],
                               policy);
                if constexpr (SFT > 0 && !WS)
                  bulk_load_hint(sp + kOffBsf + w * SFT * 512, src + kTileBytes, SFT * 512,
                                 &full[stage], policy);
              }
            }
            if constexpr (SFT > 0 && !WS)
              bulk_load(sp + kOffAsf, sfa + kb * SFT * 512, SFT * 512, &full[stage]);
            ++slots;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        // Before leaving, make sure no copy this thread issued is still in
        // flight (they all completed already unless the block gave up).
        for (int back = 1; back <= kStages && back <= slots; ++back) {
          const int idx = slots - back;
          if (idx == skipped) continue;
          mbar_wait(&full[idx % kStages], static_cast<uint32_t>((idx / kStages) & 1), nullptr);
        }
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (WS && warp == 3) {
      // ------------------------------------------------ scale producer
      // Fills the scale ring (both weight tiles' scale tiles and the
      // activation scale tiles of each K slice) as far ahead of the operand
      // ring as its slots allow; a slot is released once its scales are in
      // TMEM (or, without the stagers, once the MMA thread's copies of them
      // have completed).
      if (lane == 0) {
        const uint64_t once = l2_policy_evict_first();
        const uint64_t reused = l2_policy_evict_normal();
        int stage = 0;
        uint32_t phase = 0;
        int slots = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
          const GemmArgs& A = gargs(item);
          const Item it = map_item<NW == 2>(tab, args.E, A.n_tiles, local_item(item));
          const uint64_t policy =
              tab.chunk_off[it.k + 1] - tab.chunk_off[it.k] > 1 ? reused : once;
          const uint8_t* sfa = A.sfa + static_cast<int64_t>(it.prow0 >> 7) * A.sfa_tiles_k * 512;
          const uint8_t* btile =
              A.b_tiles + (static_cast<int64_t>(it.e) * A.n_tiles + it.n_tile) * NW * A.num_kb *
                              A.b_tile_bytes;
          for (int kb = 0; kb < A.num_kb; ++kb) {
            if (!mbar_wait(&sempty[stage], phase ^ 1u, abort_flag)) {
              ok = false;
              break;
            }
            uint8_t* sp = sring + stage * kSfSlot;
            mbar_arrive_expect_tx(&sfull[stage], kSfSlot);
#pragma unroll
            for (int w = 0; w < NW; ++w)
              bulk_load_hint(sp + w * SFT * 512,
                             btile + (static_cast<int64_t>(w) * A.num_kb + kb) * A.b_tile_bytes +
                                 kTileBytes,
                             SFT * 512, &sfull[stage], policy);
            bulk_load(sp + kOffAsf, sfa + kb * SFT * 512, SFT * 512, &sfull[stage]);
            ++slots;
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        for (int back = 1; back <= kStages && back <= slots; ++back) {
          const int idx = slots - back;
          mbar_wait(&sfull[idx % kStages], static_cast<uint32_t>((idx / kStages) & 1), nullptr);
        }
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (warp == 1) {
      // ------------------------------------------------ MMA issuer
      if (lane == 0) {
        uint32_t idesc;
        if constexpr (FMT == kFmtBF16) idesc = idesc_bf16(128, 128 * NW);
        else if constexpr (FMT == kFmtNVFP4) idesc = idesc_nvf4(128, 128 * NW);
        else idesc = 0;
        int stage = 0;
        uint32_t phase = 0;
        int local = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x, ++local) {
          const GemmArgs& A = gargs(item);
          const int buf = local % kBufs;
          const uint32_t use = static_cast<uint32_t>(local / kBufs);
          // A chunk of at most 32 rows keeps all its real accumulator rows in
          // TMEM lane quarter 0.  The MMA of each lane quarter reads both
          // operands' scales from that quarter's own lanes, so then only lanes
          // 0-31 need correct scales: two 512-byte scale tiles go in with one
          // non-broadcast 128x256b copy (the other lanes receive neighbouring
          // shared memory and only feed accumulator rows that are not stored).
          // Larger chunks broadcast every tile to all four quarters.
          const bool q0_only = NW == 1 && args.pair_scale_copies &&
                               map_item<NW == 2>(tab, args.E, A.n_tiles, local_item(item)).rows <= 32;
          if (!mbar_wait(&tempty[buf], (use & 1u) ^ 1u, abort_flag)) {
            ok = false;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem + buf * kAccCols;
          if constexpr (WS) {
            if (wstaged) {
              // The wide NVFP4 main loop, kept short: this thread's own time
              // per K slice (the wait, four MMA issues, the commit, the loop)
              // must stay below the tensor pipe's 262 ns for the pipe to stay
              // busy.  Descriptors advance by adding 16-byte units to the
              // start-address field (shared memory stays below 256 KiB, so
              // the field never carries).
              const uint64_t da0 = desc_sw128(smem_u32(smem));
              const uint32_t sf0 = tmem + kSfColBase;
              const int nkb = A.num_kb;
              for (int kb = 0; kb < nkb; ++kb) {
                // full counts the operand bytes and the stagers' reports
                if (!mbar_wait(&full[stage], phase, abort_flag)) {
                  ok = false;
                  break;
                }
                tc_fence_after();
                const uint64_t da = da0 + static_cast<uint64_t>(stage * (SBO >> 4));
                const uint64_t db = da + (A_BYTES >> 4);
                const uint32_t sfc = sf0 + stage * kSfColsPerStage;
                mma_nvf4(d_tmem, da, db, idesc, sfc + 32, sfc, kb != 0);
                mma_nvf4(d_tmem, da + 2, db + 2, idesc, sfc + 36, sfc + 8, 1u);
                mma_nvf4(d_tmem, da + 4, db + 4, idesc, sfc + 40, sfc + 16, 1u);
                mma_nvf4(d_tmem, da + 6, db + 6, idesc, sfc + 44, sfc + 24, 1u);
                tc_commit(&empty[stage]);
                if (++stage == kStages) {
                  stage = 0;
                  phase ^= 1u;
                }
              }
              if (ok) tc_commit(&tfull[buf]);
              continue;
            }
          }
          for (int kb = 0; kb < A.num_kb; ++kb) {
            // (WS without the stagers: the scale ring slot is waited for
            // separately)
            if (!mbar_wait(staged ? &sf_ready[stage] : &full[stage], phase, abort_flag) ||
                (WS && !wstaged && !mbar_wait(&sfull[stage], phase, abort_flag))) {
              ok = false;
              break;
            }
            tc_fence_after();
            uint8_t* sp = smem + stage * SBO;
            const uint32_t a_addr = smem_u32(sp), b_addr = smem_u32(sp + A_BYTES);
            uint8_t* sfbase = WS ? sring + stage * kSfSlot : sp;
            uint8_t* sf = sfbase + kOffBsf;  // weight scales, then activation scales
            const uint32_t sf_col = tmem + kSfColBase + stage * kSfColsPerStage;
            if constexpr (FMT == kFmtNVFP4 && NW == 2) {
              // without the stagers: the MMA thread copies the scale tiles
#pragma unroll
              for (int j = 0; j < 4; ++j) {
                tc_copy_sf(sf_col + j * 16, desc_sf(smem_u32(sfbase + kOffAsf + j * 512)));
                tc_copy_sf(sf_col + j * 16 + 8, desc_sf(smem_u32(sf + j * 512)));
                tc_copy_sf(sf_col + j * 16 + 12, desc_sf(smem_u32(sf + (SFT + j) * 512)));
              }
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_nvf4(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                         sf_col + j * 16, sf_col + j * 16 + 8, (kb | j) != 0);
            } else if constexpr (FMT == kFmtMXFP8 && NW == 2) {
              tc_copy_sf(sf_col, desc_sf(smem_u32(sf)));
              tc_copy_sf(sf_col + 4, desc_sf(smem_u32(sf + 512)));
              tc_copy_sf(sf_col + 8, desc_sf(smem_u32(sfbase + kOffAsf)));
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_mxf8(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32),
                         idesc_mxf8(128, 256, j), sf_col + 8, sf_col, (kb | j) != 0);
            } else if constexpr (FMT == kFmtNVFP4) {
              if (q0_only && staged) {
                // lanes 0-31 of the stage's scale columns were written by warp 0
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  mma_nvf4(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                           sf_col + j * 8, sf_col + j * 8 + 4, (kb | j) != 0);
              } else if (q0_only) {
                // columns: A scales of substeps 0-1 | 2-3, B scales 0-1 | 2-3
                const uint32_t sfa = smem_u32(sf + 4 * 512), sfb = smem_u32(sf);
                tc_copy_128x256b(sf_col, desc_sf_pair(sfa, 512));
                tc_copy_128x256b(sf_col + 8, desc_sf_pair(sfa + 1024, 512));
                tc_copy_128x256b(sf_col + 16, desc_sf_pair(sfb, 512));
                tc_copy_128x256b(sf_col + 24, desc_sf_pair(sfb + 1024, 512));
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  const uint32_t c = (j >> 1) * 8 + (j & 1) * 4;
                  mma_nvf4(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                           sf_col + c, sf_col + 16 + c, (kb | j) != 0);
                }
              } else {
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                  tc_copy_sf(sf_col + j * 8, desc_sf(smem_u32(sf + (4 + j) * 512)));
                  tc_copy_sf(sf_col + j * 8 + 4, desc_sf(smem_u32(sf + j * 512)));
                }
#pragma unroll
                for (int j = 0; j < 4; ++j)
                  mma_nvf4(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                           sf_col + j * 8, sf_col + j * 8 + 4, (kb | j) != 0);
              }
            } else if constexpr (FMT == kFmtMXFP8) {
              if (q0_only && staged) {
                // lanes 0-31 of the stage's scale columns were written by warp 0
              } else if (q0_only) {
                // columns 0-3: B scales, 4-7: A scales (tiles adjacent in smem)
                tc_copy_128x256b(sf_col, desc_sf_pair(smem_u32(sf), 512));
              } else {
                tc_copy_sf(sf_col, desc_sf(smem_u32(sf)));
                tc_copy_sf(sf_col + 4, desc_sf(smem_u32(sf + 512)));
              }
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_mxf8(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32),
                         idesc_mxf8(128, 128, j), sf_col + 4, sf_col, (kb | j) != 0);
            } else {
#pragma unroll
              for (int j = 0; j < 4; ++j)
                mma_bf16(d_tmem, desc_sw128(a_addr + j * 32), desc_sw128(b_addr + j * 32), idesc,
                         (kb | j) != 0);
            }
            tc_commit(&empty[stage]);
            if (WS && !wstaged) tc_commit(&sempty[stage]);  // its scale copies are done
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
          if (ok) tc_commit(&tfull[buf]);
        }
        // Every MMA this thread issued must finish before TMEM is released.
        tc_commit(drained);
        mbar_wait(drained, 0, nullptr);
        if (!ok) report_status(args.status, kStatusTimeout);
      }
    } else if (WS && warp >= kEpiWarp0 + 4 * NW) {
      // ------------------------------------------------ wide scale stagers
      // Warp w writes TMEM lane quarter q = w % 4 of each stage's 64 scale
      // columns: per 64-element substep j, the 256 weight rows' scales in
      // columns 8j..8j+7 (row n at column 8j + n/32, lane n % 32: every quarter
      // holds all of them), and its own 32 activation rows' scales in column
      // 32 + 4j + q (the MMA of quarter q reads column q of the four starting
      // at the activation scale address).  A stage's columns are free once
      // the MMAs of the stage's previous use have completed (its empty
      // barrier), its scales come from the scale ring, and the report goes
      // to the stage's full barrier, which the MMA thread waits on anyway:
      // the scales are staged while the operands are still in flight.
      if (wstaged) {
        const int q = warp & 3;
        int stage = 0;
        uint32_t phase = 0;
        bool ok = true;
        for (int item = blockIdx.x; item < total && ok; item += gridDim.x) {
          const GemmArgs& A = gargs(item);
          for (int kb = 0; kb < A.num_kb; ++kb) {
            const bool ready = mbar_wait(&sfull[stage], phase, abort_flag) &&
                               mbar_wait(&empty[stage], phase ^ 1u, abort_flag);
            if (!__all_sync(0xFFFFFFFFu, ready)) {
              ok = false;
              break;
            }
            tc_fence_after();
            const uint8_t* sp = sring + stage * kSfSlot;
            uint32_t v[32];
#pragma unroll
            for (int j = 0; j < 4; ++j) {
              const uint4 b0 = *reinterpret_cast<const uint4*>(sp + kOffBsf + j * 512 + lane * 16);
              const uint4 b1 =
                  *reinterpret_cast<const uint4*>(sp + kOffBsf + (SFT + j) * 512 + lane * 16);
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
              a4[j] = *reinterpret_cast<const uint32_t*>(sp + kOffAsf + j * 512 + lane * 16 + q * 4);
            // the ring slot has been read; the next bulk copy into it is an
            // async-proxy write after these generic-proxy reads
            asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
            __syncwarp();
            if (lane == 0) mbar_arrive(&sempty[stage]);
            const uint32_t col = tmem + (static_cast<uint32_t>(q * 32) << 16) + kSfColBase +
                                 stage * kSfColsPerStage;
            tmem_st32(col, v);
#pragma unroll
            for (int j = 0; j < 4; ++j) tmem_st1(col + 32 + 4 * j + q, a4[j]);
            tmem_st_wait();
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&full[stage]);
            if (++stage == kStages) {
              stage = 0;
              phase ^= 1u;
            }
          }
        }
        if (!ok && lane == 0) report_status(args.status, kStatusTimeout);
      }
    }
  } else {
    if constexpr (WS) regs_claim<kEpiRegs>();
    // ------------------------------------------------ epilogue warps
    // Warp w reads TMEM lane quarter w % 4 (rows 32q..) of accumulator
    // column group (w - 3) / 4 (one 128-column group per weight tile).
    const int q = warp & 3;
    const int grp = (warp - kEpiWarp0) >> 2;
    int local = 0;
    for (int item = blockIdx.x; item < total; item += gridDim.x, ++local) {
      const GemmArgs& A = gargs(item);
      const bool g2 = second(item);
      const Item it = map_item<NW == 2>(tab, args.E, A.n_tiles, local_item(item));
      const int buf = local % kBufs;
      const uint32_t use = static_cast<uint32_t>(local / kBufs);
      if (!mbar_wait(&tfull[buf], use & 1u, abort_flag)) {
        if (lane == 0) report_status(args.status, kStatusTimeout);
        break;
      }
      tc_fence_after();
      const int r = q * 32 + lane;
      const bool active = q * 32 < it.rows;
      const uint32_t taddr =
          tmem + (static_cast<uint32_t>(q * 32) << 16) + buf * kAccCols + grp * 128;
      const int64_t prow = it.prow0 + r;
      // batched format: expert e's rows go to rows e*M.. of the output
      const int64_t orow = A.out_rows_per_expert
                               ? static_cast<int64_t>(it.e) * A.out_rows_per_expert +
                                     (it.prow0 - tab.pad_off[it.k]) + r
                               : prow;
      const int n128 = it.n_tile * NW + grp;
      if constexpr (NW == 1) {
        if (active) {
          uint32_t carry[5];
#pragma unroll
          for (int p = 0; p < 2; ++p) {
            uint32_t v[64];
            if (g2) epilogue_load<2>(taddr, p, v);
            else epilogue_load<EPI>(taddr, p, v);
            tmem_ld_wait();
            epilogue_fence(v);
            if (g2) epilogue_round<FMT, 2>(v, p, r < it.rows, prow, orow, n128, A, carry);
            else epilogue_round<FMT, EPI>(v, p, r < it.rows, prow, orow, n128, A, carry);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (FUSED && !g2) {
          // this warp's rows of the item are stored: count them for GEMM2
          __threadfence();
          __syncwarp();
          if (lane == 0) atomicAdd(args.done1 + it.e, 1);
        }
      } else {
        uint32_t v[128];
        if (active) {
          epilogue_load<EPI>(taddr, 0, v);
          epilogue_load<EPI>(taddr, 1, v + 64);
          tmem_ld_wait();
          epilogue_fence(v);
          epilogue_fence(v + 64);
        }
        // the accumulator is free for the next item's MMAs from here on
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&tempty[buf]);
        if (active) {
          uint32_t carry[5];
          epilogue_round<FMT, EPI>(v, 0, r < it.rows, prow, orow, n128, A, carry);
          epilogue_round<FMT, EPI>(v + 64, 1, r < it.rows, prow, orow, n128, A, carry);
          if (EPI == 4 && A.gather_inv) combine_fused(r < it.rows, prow, n128, A);
        }
      }
    }
  }

  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

// Set once the launch allocation of a wide-stager instantiation has been
// checked against its register split.
template <int FMT, int EPI, int MROWS, int NW, bool FUSED>
bool& split_checked() {
  static bool ok = false;
  return ok;
}

template <int FMT, int EPI, int MROWS, int NW, bool FUSED = false>
cudaError_t launch_one(const GemmMaps& maps, const GemmArgs& args, const GemmMaps& maps2,
                       const GemmArgs& args2, int grid, cudaStream_t s) {
  if (wide_stager(FMT, NW) && !split_checked<FMT, EPI, MROWS, NW, FUSED>())
    return cudaErrorInvalidConfiguration;
  return launch_pdl(g_pdl_gemm, moe_gemm_kernel<FMT, EPI, MROWS, NW, FUSED>, dim3(grid),
                    dim3(gemm_threads(FMT, NW)), gemm_smem<FMT, MROWS, NW>(), s, maps, args,
                    maps2, args2);
}

template <int FMT, int EPI, int MROWS, int NW, bool FUSED = false>
cudaError_t set_smem() {
  cudaError_t e = cudaFuncSetAttribute(moe_gemm_kernel<FMT, EPI, MROWS, NW, FUSED>,
                                       cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       gemm_smem<FMT, MROWS, NW>());
  if (e != cudaSuccess || !wide_stager(FMT, NW)) return e;
  // The kernel's register split only balances at kSplitLaunchRegs registers
  // per thread; with fewer, the claiming warpgroups would wait forever.
  cudaFuncAttributes fa{};
  e = cudaFuncGetAttributes(&fa, moe_gemm_kernel<FMT, EPI, MROWS, NW, FUSED>);
  if (e != cudaSuccess) return e;
  if (fa.numRegs != kSplitLaunchRegs ||
      fa.numRegs * gemm_threads(FMT, NW) > 65536)
    return cudaErrorInvalidConfiguration;
  split_checked<FMT, EPI, MROWS, NW, FUSED>() = true;
  return cudaSuccess;
}

template <int FMT, int MROWS, int NW>
cudaError_t prepare_m() {
  cudaError_t e = set_smem<FMT, 1, MROWS, NW>();
  if (e == cudaSuccess) e = set_smem<FMT, 2, MROWS, NW>();
  if (e == cudaSuccess) e = set_smem<FMT, 3, MROWS, NW>();
  return e;
}

template <int FMT>
cudaError_t prepare_one() {
  cudaError_t e = prepare_m<FMT, 32, 1>();
  if (e == cudaSuccess) e = prepare_m<FMT, 64, 1>();
  if (e == cudaSuccess) e = prepare_m<FMT, 128, 1>();
  if (e == cudaSuccess) e = prepare_m<FMT, 128, 2>();
  if (e == cudaSuccess) e = set_smem<FMT, 4, 128, 2>();
  if (e == cudaSuccess) e = set_smem<FMT, 1, 32, 1, true>();
  if (e == cudaSuccess) e = set_smem<FMT, 3, 32, 1, true>();
  return e;
}

template <int FMT, int EPI>
cudaError_t launch_fmt(const GemmMaps& maps, const GemmArgs& args, int grid, int mrows, bool wide,
                       cudaStream_t s) {
  if (wide) return launch_one<FMT, EPI, 128, 2>(maps, args, maps, args, grid, s);
  if (mrows <= 32) return launch_one<FMT, EPI, 32, 1>(maps, args, maps, args, grid, s);
  if (mrows <= 64) return launch_one<FMT, EPI, 64, 1>(maps, args, maps, args, grid, s);
  return launch_one<FMT, EPI, 128, 1>(maps, args, maps, args, grid, s);
}

// epi 4: GEMM2 with the fused combine (wide launches only).  Its gather is
// compiled into its own kernel: inside the plain GEMM2 kernel it made the
// register allocator spill 172 bytes for every wide GEMM2 launch.
template <int FMT>
cudaError_t launch_epi(int epi, const GemmMaps& maps, const GemmArgs& args, int grid, int mrows,
                       bool wide, cudaStream_t s) {
  if (epi == 4)
    return wide ? launch_one<FMT, 4, 128, 2>(maps, args, maps, args, grid, s)
                : cudaErrorInvalidValue;
  return epi == 1   ? launch_fmt<FMT, 1>(maps, args, grid, mrows, wide, s)
         : epi == 3 ? launch_fmt<FMT, 3>(maps, args, grid, mrows, wide, s)
                    : launch_fmt<FMT, 2>(maps, args, grid, mrows, wide, s);
}

}  // namespace

cudaError_t gemm_prepare(int fmt) {
  return fmt == kFmtBF16 ? prepare_one<kFmtBF16>()
         : fmt == kFmtMXFP8 ? prepare_one<kFmtMXFP8>()
                            : prepare_one<kFmtNVFP4>();
}

cudaError_t launch_gemm(int fmt, int epi, const GemmMaps& maps, const GemmArgs& args, int grid,
                        int max_rows, bool wide, cudaStream_t s) {
  if (fmt == kFmtBF16) return launch_epi<kFmtBF16>(epi, maps, args, grid, max_rows, wide, s);
  if (fmt == kFmtMXFP8) return launch_epi<kFmtMXFP8>(epi, maps, args, grid, max_rows, wide, s);
  return launch_epi<kFmtNVFP4>(epi, maps, args, grid, max_rows, wide, s);
}

namespace {

template <int FMT, int EPI>
cudaError_t launch_fused_fmt(const GemmMaps& maps1, const GemmArgs& args1, const GemmMaps& maps2,
                             const GemmArgs& args2, int grid, int mrows, cudaStream_t s) {
  if (mrows > 32) return cudaErrorInvalidValue;  // decode-sized chunks only
  return launch_one<FMT, EPI, 32, 1, true>(maps1, args1, maps2, args2, grid, s);
}

template <int FMT>
cudaError_t launch_fused_epi(int epi1, const GemmMaps& maps1, const GemmArgs& args1,
                             const GemmMaps& maps2, const GemmArgs& args2, int grid, int mrows,
                             cudaStream_t s) {
  return epi1 == 3 ? launch_fused_fmt<FMT, 3>(maps1, args1, maps2, args2, grid, mrows, s)
                   : launch_fused_fmt<FMT, 1>(maps1, args1, maps2, args2, grid, mrows, s);
}

}  // namespace

cudaError_t launch_gemm_fused(int fmt, int epi1, const GemmMaps& maps1, const GemmArgs& args1,
                              const GemmMaps& maps2, const GemmArgs& args2, int grid,
                              int max_rows, cudaStream_t s) {
  if (fmt == kFmtBF16)
    return launch_fused_epi<kFmtBF16>(epi1, maps1, args1, maps2, args2, grid, max_rows, s);
  if (fmt == kFmtMXFP8)
    return launch_fused_epi<kFmtMXFP8>(epi1, maps1, args1, maps2, args2, grid, max_rows, s);
  return launch_fused_epi<kFmtNVFP4>(epi1, maps1, args1, maps2, args2, grid, max_rows, s);
}

}  // namespace moe
