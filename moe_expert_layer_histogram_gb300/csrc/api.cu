// api.cu -- host runtime behind the C ABI in include/moe.h.
//
// moe_create sizes and allocates every device buffer once for T_max tokens
// (the reference design also sizes its workspace once, by its maximum token
// count: MegaMoE kernel-drop workflow page, sec. 六, num_max_tokens), so a
// forward allocates nothing and only enqueues kernels on the caller's
// stream: routing + histogram, scan, scatter + activation quantisation,
// GEMM1 (+SwiGLU/requant), GEMM2, combine -- for T <= 16 one front-end
// kernel, one launch for both GEMMs and the combine.  E and K are fixed at create;
// every launch uses the handle's E (a global-vs-local expert-count mismatch
// broke the reference integration: PR #40082 report, sec. 风险与影响 item 3).
#include <cudaTypedefs.h>

#include <algorithm>
#include <cmath>
#include <cstdlib>
#include <cstring>
#include <string>
#include <vector>

#include "internal.h"
#include "moe.h"

using namespace moe;

thread_local bool moe::g_pdl_small = true;
thread_local bool moe::g_pdl_gemm = true;

struct moe_layer {
  moe_config cfg;
  int device = 0, num_sms = 0;
  int fmt = 0, H = 0, I = 0, E = 0, K = 0, Tmax = 0;
  int64_t Rmax = 0, Rpad = 0;
  int NBmax = 0;
  int xb = 0, hb = 0;                // bytes per row: GEMM1 / GEMM2 input
  int x_tiles_k = 0, h_tiles_k = 0;  // 128x4 scale tiles per 128-row block
  float clamp = INFINITY;
  int act = MOE_ACT_SWIGLU;
  int w13_rows = 0;                  // 2I (SwiGLU: gate and up) or I (ReLU^2)
  std::vector<void*> allocs;
  int32_t *ids = nullptr, *blockhist = nullptr, *prefix = nullptr;
  int32_t *offsets = nullptr, *pad_off = nullptr, *chunk_off = nullptr, *counts = nullptr;
  int32_t *perm = nullptr, *inv = nullptr;
  int combine = MOE_COMBINE_GATHER;
  float* acc = nullptr;              // in-kernel reduce: fp32 [Tmax, H], zero between forwards
  int32_t *acc_cnt = nullptr, *prow_slot = nullptr;
  int32_t* done1 = nullptr;          // fused decode GEMMs: per-expert GEMM1 completion counts
  int32_t* otab = nullptr;           // [4(E+1)] the GEMMs' item tables in the mixed order
  int mix_items = 1;                 // wide single-CTA GEMMs: single-chunk experts' items mixed in
  DecodeCtl* dctl = nullptr;         // single-launch decode: counters (zero between forwards)
  int single_launch = 1;             // T <= 16: the whole layer in one kernel
  int fused_gemms = 1;               // T <= 16: GEMM1 and GEMM2 in one launch
  int host_zero_copy = 1;            // moe_forward_host: kernels access pinned host buffers
  float* w = nullptr;
  uint8_t *xq = nullptr, *xsf = nullptr, *hq = nullptr, *hsf = nullptr, *y = nullptr;
  uint8_t *w13t = nullptr, *w2t = nullptr;  // prepared weight tiles
  int* status = nullptr;
  uint8_t *h_in = nullptr, *o_out = nullptr;
  float* l_in = nullptr;
  // moe_forward_host_async: streams for the input copies, the layer and the
  // output copies, and their events (created on first use); ev_user marks
  // the latest work on the layer enqueued on a caller's stream by the other
  // entry points
  cudaStream_t xi = nullptr, xo = nullptr, cs = nullptr;
  cudaEvent_t ev_in = nullptr, ev_front = nullptr, ev_comb = nullptr, ev_d2h = nullptr,
              ev_user = nullptr;
  GemmMaps maps1{}, maps2{};
  int pair_scale_copies = 1;
  int wide_tiles = -1;               // 0 off, 1 always, -1 for prefill-sized launches
  int stage_scales = 1;              // decode scales written by a warp, not copied
  int test_stall = 0;                // fault injection (moe_config.test_stall_gemm): GEMM1 times out
  int max_ctas = 0;                  // CTAs per GEMM launch (moe_config.max_ctas, else the SM count)
  int pair_clusters = 0;             // NVFP4 wide launches: co-resident CTA pairs (0: single CTAs)
  bool pdl_small = true;             // programmatic dependent launch of the small kernels
  bool pdl_gemm = true;              // ... of the GEMM kernels
  bool pdl_prefill = false;          // ... also for prefill-sized (wide) forwards
  bool weights_ready = false;
  int last_T = 0, last_launches = 0;
  std::vector<cudaEvent_t> tev;  // per-kernel timing events, 7 per forward
  int timing_max = 0, timing_rec = 0;
};

namespace {

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  if (!fn) {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  }
  return fn;
}

// 2-D byte tensor [rows, row_bytes], box of 128 bytes x box_rows, 128-byte
// swizzle (the layout the MMA descriptors expect) or none (data stored
// pre-swizzled).
bool make_map(CUtensorMap* m, void* base, uint64_t row_bytes, uint64_t rows, uint32_t box_rows,
              bool swizzle = true) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {row_bytes, rows};
  cuuint64_t strides[1] = {row_bytes};
  cuuint32_t box[2] = {128, box_rows};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE,
            swizzle ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Prepared weight tiles viewed as rows of 2 KiB (256 x 64-bit elements), box
// of 8 rows (16 KiB), no swizzle: the codes are stored pre-swizzled.
bool make_tile_map(CUtensorMap* m, void* base, uint64_t rows) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {256, rows};
  cuuint64_t strides[1] = {2048};
  cuuint32_t box[2] = {256, 8};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_UINT64, 2, base, dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
            CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Device allocations of moe_create.  moe_config.test_fail_alloc_at = n makes
// the n-th one fail, so tests can check that the error is reported and
// nothing leaks, without exhausting the GPU.
struct Allocator {
  moe_layer* L;
  int count = 0, fail_at = 0;
  Allocator(moe_layer* l, int fail) : L(l), fail_at(fail) {}
  template <class T>
  bool get(T** p, size_t bytes) {
    ++count;
    *p = nullptr;
    if (fail_at > 0 && count == fail_at) return false;
    void* q = nullptr;
    if (cudaMalloc(&q, std::max<size_t>(bytes, 256)) != cudaSuccess) {
      cudaGetLastError();
      return false;
    }
    L->allocs.push_back(q);
    *p = static_cast<T*>(q);
    return true;
  }
};

void free_all(moe_layer* L) {
  for (void* p : L->allocs) cudaFree(p);
  L->allocs.clear();
}

// Launches of more than kPairCopyMaxTokens tokens (mostly full 128-row
// chunks) use GEMM items of two weight tiles (N = 256), which halves the
// shared-memory traffic of the activation operand per FLOP.
//
// Chunks of at most 32 rows can take their block scales in with half as
// many TMEM copies (lanes 0-31 only).  Measured on GB300 this speeds up
// decode-sized launches (every chunk that small) by 10-15 %, but slows a
// prefill launch that mixes such chunks with full ones (Zipf-routed T=8192:
// GEMM2 +35 %), so it is used up to this many tokens.
constexpr int kPairCopyMaxTokens = 1024;

int64_t max_chunks(const moe_layer* L, int T) {
  const int64_t R = static_cast<int64_t>(T) * L->K;
  return std::min<int64_t>(L->E, R) + R / kRowBlock;
}

// Work that another entry point enqueues on the caller's stream s is
// ordered after the pipelined forwards' layer work (before_call), and the
// next pipelined forward after it (after_call).  No-ops until
// moe_forward_host_async has been used on the layer.
void before_call(const moe_layer* L, cudaStream_t s) {
  if (L->cs) cudaStreamWaitEvent(s, L->ev_comb, 0);
}
void after_call(const moe_layer* L, cudaStream_t s) {
  if (L->cs) cudaEventRecord(L->ev_user, s);
}

// Launch attributes of this forward's kernels (read by launch_pdl on this
// host thread): programmatic dependent launch for decode-sized forwards,
// plain stream order for wide (prefill) ones unless MOE_PDL_PREFILL=1.
void set_pdl(const moe_layer* L, bool wide) {
  const bool on = !wide || L->pdl_prefill;
  g_pdl_small = L->pdl_small && on;
  g_pdl_gemm = L->pdl_gemm && on;
}

// GEMM1 (+ the activation and re-quantisation) over the padded
// activation rows of the current tables.
// The item tables of a GEMM launch: by expert, or (mixed) the ones the
// scatter kernel wrote in the mixed order.
void set_tables(const moe_layer* L, bool mixed, GemmArgs& a) {
  if (mixed) {
    a.chunk_off = L->otab;
    a.pad_off = L->otab + (L->E + 1);
    a.counts = L->otab + (2 * L->E + 1);
    a.order = L->otab + (3 * L->E + 1);
  } else {
    a.chunk_off = L->chunk_off;
    a.pad_off = L->pad_off;
    a.counts = L->counts;
    a.order = nullptr;
  }
}

GemmArgs gemm1_args(const moe_layer* L, int pair, bool wide, bool mixed = false) {
  GemmArgs a{};
  set_tables(L, mixed, a);
  a.E = L->E;
  a.n_tiles = L->w13_rows / (wide ? 256 : 128);
  a.num_kb = L->xb / 128;
  a.sfa = L->xsf;
  a.sfa_tiles_k = L->x_tiles_k;
  a.b_tiles = L->w13t;
  a.b_tile_bytes = weight_tile_bytes(L->fmt);
  a.out = L->hq;
  a.out_ld = L->hb;
  a.out_sf = L->hsf;
  a.out_sf_tiles_k = L->h_tiles_k;
  a.clamp = L->clamp;
  a.pair_scale_copies = pair;
  a.stage_scales = L->stage_scales;
  a.test_stall = L->test_stall;
  a.out_rows_per_expert = 0;
  a.status = L->status;
  return a;
}

// GEMM2 into `out` (bf16, H per row): padded rows (rows_per_expert 0) or
// rows e*rows_per_expert + i (batched format).  reduce_out (routed forward
// with the in-kernel reduce): the bf16 layer output, summed by GEMM2's
// epilogue instead of the combine kernel.
GemmArgs gemm2_args(const moe_layer* L, int pair, bool wide, void* out, int rows_per_expert,
                    void* reduce_out, bool mixed = false) {
  GemmArgs a{};
  set_tables(L, mixed, a);
  a.E = L->E;
  a.n_tiles = L->H / (wide ? 256 : 128);
  a.num_kb = L->hb / 128;
  a.sfa = L->hsf;
  a.sfa_tiles_k = L->h_tiles_k;
  a.b_tiles = L->w2t;
  a.b_tile_bytes = weight_tile_bytes(L->fmt);
  a.out = static_cast<uint8_t*>(out);
  a.out_ld = static_cast<int64_t>(L->H) * 2;
  a.out_sf = nullptr;
  a.out_sf_tiles_k = 0;
  a.clamp = INFINITY;
  a.pair_scale_copies = pair;
  a.stage_scales = L->stage_scales;
  a.out_rows_per_expert = rows_per_expert;
  if (reduce_out && L->combine != MOE_COMBINE_GATHER) {
    a.acc = L->combine == MOE_COMBINE_REDUCE ? L->acc : nullptr;
    a.gather_inv = L->combine == MOE_COMBINE_FUSED ? L->inv : nullptr;
    a.acc_cnt = L->acc_cnt;
    a.prow_slot = L->prow_slot;
    a.topk_w = L->w;
    a.comb_out = static_cast<uint8_t*>(reduce_out);
    a.K = L->K;
    a.H = L->H;
  }
  a.status = L->status;
  return a;
}

// Wide NVFP4 items run on CTA pairs when the device has them: one launch of
// `clusters` pairs, each item covering up to two 128-row chunks.
cudaError_t launch_wide_or_pair(moe_layer* L, int epi, const GemmMaps& maps, const GemmArgs& a,
                                int64_t chunks, int max_rows, bool wide, cudaStream_t s) {
  if (wide && L->pair_clusters > 0) {
    const int clusters = static_cast<int>(
        std::min<int64_t>(std::min(L->pair_clusters, std::max(1, L->max_ctas / 2)),
                          (chunks + 1) / 2 * a.n_tiles));
    return launch_gemm_pair(epi, maps, a, clusters, s);
  }
  const int grid = static_cast<int>(std::min<int64_t>(L->max_ctas, chunks * a.n_tiles));
  // GEMM2 with the fused combine has a kernel of its own (epilogue kind 4)
  return launch_gemm(L->fmt, epi == 2 && a.gather_inv && wide ? 4 : epi, maps, a, grid, max_rows,
                     wide, s);
}

// max_rows bounds the rows of any expert (selects the activation tile height).
// mixed: the scatter kernel wrote the mixed-order tables (wide single-CTA
// launches of the routed forward).
cudaError_t run_gemm1(moe_layer* L, int64_t chunks, int max_rows, int pair, bool wide,
                      cudaStream_t s, bool mixed = false) {
  wide = wide && L->w13_rows % 256 == 0;
  const GemmArgs a = gemm1_args(L, pair, wide, mixed && wide);
  return launch_wide_or_pair(L, L->act == MOE_ACT_RELU2 ? 3 : 1, L->maps1, a, chunks, max_rows,
                             wide, s);
}

cudaError_t run_gemm2(moe_layer* L, int64_t chunks, int max_rows, int pair, bool wide, void* out,
                      int rows_per_expert, cudaStream_t s, void* reduce_out = nullptr,
                      bool mixed = false) {
  wide = wide && L->H % 256 == 0;
  const GemmArgs a = gemm2_args(L, pair, wide, out, rows_per_expert, reduce_out, mixed && wide);
  return launch_wide_or_pair(L, 2, L->maps2, a, chunks, max_rows, wide, s);
}

// Decode: GEMM1 and GEMM2 in one persistent launch (narrow items, chunks of
// at most 32 rows); the one-kernel front end has zeroed the per-expert
// counters.
cudaError_t run_gemms_fused(moe_layer* L, int64_t chunks, int max_rows, int pair,
                            void* reduce_out, cudaStream_t s) {
  GemmArgs a1 = gemm1_args(L, pair, false);
  a1.done1 = L->done1;
  const GemmArgs a2 = gemm2_args(L, pair, false, L->y, 0, reduce_out);
  const int grid = static_cast<int>(
      std::min<int64_t>(L->max_ctas, chunks * (a1.n_tiles + a2.n_tiles)));
  return launch_gemm_fused(L->fmt, L->act == MOE_ACT_RELU2 ? 3 : 1, L->maps1, a1, L->maps2, a2,
                           grid, max_rows, s);
}

// The device address of page-locked host memory, or nullptr when `p` is not
// page-locked host memory the device can address.
void* device_view(const void* p) {
  cudaPointerAttributes a{};
  if (cudaPointerGetAttributes(&a, p) != cudaSuccess) {
    cudaGetLastError();
    return nullptr;
  }
  return a.type == cudaMemoryTypeHost ? a.devicePointer : nullptr;
}

}  // namespace

extern "C" {

const char* moe_status_string(moe_status s) {
  switch (s) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape or format";
    case MOE_ERR_NO_WEIGHTS: return "weights not prepared";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "device allocation failed";
    case MOE_ERR_DEVICE_TIMEOUT: return "a kernel gave up a bounded wait";
    case MOE_ERR_NO_DEVICE: return "no usable sm_103 device";
  }
  return "unknown status";
}

moe_status moe_create(const moe_config* cfg, moe_layer** out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg) return MOE_ERR_INVALID_ARG;
  const moe_config c = *cfg;
  if (c.max_tokens < 1 || c.hidden < 1 || c.inter < 1 || c.num_experts < 1 || c.top_k < 1)
    return MOE_ERR_INVALID_ARG;
  if (c.format < MOE_FMT_BF16 || c.format > MOE_FMT_NVFP4) return MOE_ERR_INVALID_ARG;
  if (c.activation != MOE_ACT_SWIGLU && c.activation != MOE_ACT_RELU2) return MOE_ERR_INVALID_ARG;
  if (c.combine != MOE_COMBINE_GATHER && c.combine != MOE_COMBINE_REDUCE &&
      c.combine != MOE_COMBINE_FUSED)
    return MOE_ERR_INVALID_ARG;
  if (c.max_ctas < 0 || c.test_fail_alloc_at < 0 || c.test_stall_gemm < 0 || c.test_stall_gemm > 1)
    return MOE_ERR_INVALID_ARG;
  if (c.activation == MOE_ACT_RELU2 && c.clamp_limit > 0.0f && std::isfinite(c.clamp_limit))
    return MOE_ERR_UNSUPPORTED;
  const int kq = c.format == MOE_FMT_NVFP4 ? 256 : 128;
  if (c.hidden % kq || c.inter % kq || c.num_experts > kMaxExperts || c.top_k > kMaxTopK ||
      c.top_k > c.num_experts)
    return MOE_ERR_UNSUPPORTED;
  const int64_t Rmax = static_cast<int64_t>(c.max_tokens) * c.top_k;
  const int64_t Rpad =
      (Rmax + static_cast<int64_t>(kRowBlock - 1) * std::min<int64_t>(c.num_experts, Rmax) +
       kRowBlock - 1) / kRowBlock * kRowBlock;
  if (Rpad >= (int64_t(1) << 30)) return MOE_ERR_UNSUPPORTED;

  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  int major = 0, minor = 0, sms = 0;
  cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
  cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
  cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (major != 10 || minor != 3) return MOE_ERR_NO_DEVICE;
  if (gemm_prepare(c.format) != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_NO_DEVICE;
  }
  if (!encode_fn()) return MOE_ERR_NO_DEVICE;
  const char* pv = std::getenv("MOE_PAIR_SCALE_COPIES");

  moe_layer* L = new moe_layer;
  L->cfg = c;
  L->device = dev;
  {
    const char* v = std::getenv("MOE_DISABLE_PDL");
    const std::string off = v ? v : "";
    L->pdl_small = !(off == "1" || off == "small");
    L->pdl_gemm = !(off == "1" || off == "gemm");
    const char* pp = std::getenv("MOE_PDL_PREFILL");
    L->pdl_prefill = pp && pp[0] == '1';
  }
  L->num_sms = sms;
  L->fmt = c.format;
  L->H = c.hidden;
  L->I = c.inter;
  L->E = c.num_experts;
  L->K = c.top_k;
  L->Tmax = c.max_tokens;
  L->Rmax = Rmax;
  L->Rpad = Rpad;
  L->NBmax = (c.max_tokens + kTokensPerRouteBlock - 1) / kTokensPerRouteBlock;
  L->clamp = (c.clamp_limit > 0.0f && std::isfinite(c.clamp_limit)) ? c.clamp_limit : INFINITY;
  L->act = c.activation;
  L->combine = c.combine;
  L->w13_rows = c.activation == MOE_ACT_RELU2 ? c.inter : 2 * c.inter;
  // MOE_PAIR_SCALE_COPIES=0 turns the decode-sized scale-copy path off.
  L->pair_scale_copies = !(pv && pv[0] == '0');
  // MOE_WIDE_TILES=0|1: never / always use the N = 256 GEMM items (default:
  // for launches of more than kPairCopyMaxTokens tokens).
  if (const char* wv = std::getenv("MOE_WIDE_TILES")) L->wide_tiles = wv[0] == '0' ? 0 : 1;
  // MOE_SCALE_STAGER=0: decode chunks copy their scales with tcgen05.cp
  // (lanes 0-31 through 128x256b copies) instead of a staging warp.
  if (const char* sv = std::getenv("MOE_SCALE_STAGER")) L->stage_scales = sv[0] != '0';
  // Fault injection for the bounded waits (tests only, through the config):
  // one CTA of every GEMM1 launch leaves one stage unloaded; its waits give
  // up after 2 s and moe_get_status reports MOE_ERR_DEVICE_TIMEOUT.
  L->test_stall = c.test_stall_gemm == 1;
  L->max_ctas = c.max_ctas > 0 ? std::min(c.max_ctas, sms) : sms;
  // NVFP4 wide (prefill) launches on CTA pairs with MOE_PAIR_CTAS=1 (off by
  // default: measured slower than single CTAs so far).
  if (L->fmt == MOE_FMT_NVFP4) {
    const char* pv2 = std::getenv("MOE_PAIR_CTAS");
    if (pv2 && pv2[0] == '1' && gemm_pair_prepare(&L->pair_clusters) != cudaSuccess) {
      cudaGetLastError();
      delete L;
      return MOE_ERR_NO_DEVICE;
    }
  }
  // MOE_SINGLE_LAUNCH=0: decode batches use the three-launch path (front
  // end, both GEMMs in one launch, combine) instead of the single kernel.
  if (const char* sv1 = std::getenv("MOE_SINGLE_LAUNCH")) L->single_launch = sv1[0] != '0';
  if (decode_prepare(L->fmt) != cudaSuccess) {
    cudaGetLastError();
    delete L;
    return MOE_ERR_NO_DEVICE;
  }
  // MOE_FUSED_GEMMS=0: decode launches keep GEMM1 and GEMM2 separate.
  if (const char* fv = std::getenv("MOE_FUSED_GEMMS")) L->fused_gemms = fv[0] != '0';
  // MOE_HOST_ZERO_COPY=0: moe_forward_host always copies through device buffers.
  if (const char* zv = std::getenv("MOE_HOST_ZERO_COPY")) L->host_zero_copy = zv[0] != '0';
  // MOE_MIX_ITEMS=0: wide GEMM launches take their items in plain expert
  // order instead of mixing the single-chunk experts' items in.
  if (const char* mv = std::getenv("MOE_MIX_ITEMS")) L->mix_items = mv[0] != '0';
  const int H = L->H, I = L->I, E = L->E;
  if (L->fmt == MOE_FMT_NVFP4) {
    L->xb = H / 2; L->hb = I / 2; L->x_tiles_k = H / 64; L->h_tiles_k = I / 64;
  } else if (L->fmt == MOE_FMT_MXFP8) {
    L->xb = H; L->hb = I; L->x_tiles_k = H / 128; L->h_tiles_k = I / 128;
  } else {
    L->xb = 2 * H; L->hb = 2 * I; L->x_tiles_k = 0; L->h_tiles_k = 0;
  }
  const size_t rblocks = static_cast<size_t>(Rpad / kRowBlock);
  Allocator A(L, c.test_fail_alloc_at);
  bool ok = A.get(&L->ids, Rmax * 4) && A.get(&L->w, Rmax * 4) &&
            A.get(&L->blockhist, static_cast<size_t>(L->NBmax) * E * 4) &&
            A.get(&L->prefix, static_cast<size_t>(L->NBmax) * E * 4) &&
            A.get(&L->offsets, (E + 1) * 4) && A.get(&L->pad_off, (E + 1) * 4) &&
            A.get(&L->chunk_off, (E + 1) * 4) && A.get(&L->counts, E * 4) &&
            A.get(&L->perm, Rmax * 4) && A.get(&L->inv, Rmax * 4) &&
            A.get(&L->xq, static_cast<size_t>(Rpad) * L->xb) &&
            A.get(&L->xsf, rblocks * L->x_tiles_k * 512) &&
            A.get(&L->hq, static_cast<size_t>(Rpad) * L->hb) &&
            A.get(&L->hsf, rblocks * L->h_tiles_k * 512) &&
            A.get(&L->y, static_cast<size_t>(Rpad) * H * 2) &&
            A.get(&L->w13t, static_cast<size_t>(E) * (L->w13_rows / 128) * (L->xb / 128) *
                                weight_tile_bytes(L->fmt)) &&
            A.get(&L->w2t, static_cast<size_t>(E) * (H / 128) * (L->hb / 128) *
                               weight_tile_bytes(L->fmt)) &&
            A.get(&L->status, 16) &&
            A.get(&L->h_in, static_cast<size_t>(L->Tmax) * H * 2) &&
            A.get(&L->l_in, static_cast<size_t>(L->Tmax) * E * 4) &&
            A.get(&L->o_out, static_cast<size_t>(L->Tmax) * H * 2) &&
            A.get(&L->done1, static_cast<size_t>(E) * 4) &&
            A.get(&L->dctl, sizeof(DecodeCtl)) &&
            A.get(&L->otab, static_cast<size_t>(E + 1) * 4 * 4);
  const bool reduce = L->combine == MOE_COMBINE_REDUCE;
  const bool counted = L->combine != MOE_COMBINE_GATHER;  // reduce or fused combine
  ok = ok && (!reduce || A.get(&L->acc, static_cast<size_t>(L->Tmax) * H * 4));
  ok = ok && (!counted || (A.get(&L->acc_cnt, static_cast<size_t>(L->Tmax) * (H / 128) * 4) &&
                           A.get(&L->prow_slot, static_cast<size_t>(Rpad) * 4)));
  if (!ok) {
    free_all(L);
    delete L;
    return MOE_ERR_OOM;
  }
  // Padding rows are never written by a forward; start them at zero.
  ok = cudaMemset(L->xq, 0, static_cast<size_t>(Rpad) * L->xb) == cudaSuccess &&
       cudaMemset(L->hq, 0, static_cast<size_t>(Rpad) * L->hb) == cudaSuccess &&
       cudaMemset(L->y, 0, static_cast<size_t>(Rpad) * H * 2) == cudaSuccess &&
       cudaMemset(L->status, 0, 16) == cudaSuccess &&
       cudaMemset(L->dctl, 0, sizeof(DecodeCtl)) == cudaSuccess &&
       (!reduce || cudaMemset(L->acc, 0, static_cast<size_t>(L->Tmax) * H * 4) == cudaSuccess) &&
       (!counted ||
        cudaMemset(L->acc_cnt, 0, static_cast<size_t>(L->Tmax) * (H / 128) * 4) == cudaSuccess);
  for (int i = 0; i < 4 && ok; ++i) {
    ok = make_map(&L->maps1.a[i], L->xq, L->xb, Rpad, 16u << i) &&
         make_map(&L->maps2.a[i], L->hq, L->hb, Rpad, 16u << i);
  }
  // NVFP4 weight tiles (18 KiB: 16 KiB of codes, 2 KiB of scales) as rows
  // of 2 KiB: the codes of tile t are rows 9t .. 9t+7, one box of 8 rows
  if (L->fmt == MOE_FMT_NVFP4)
    ok = ok &&
         make_tile_map(&L->maps1.b, L->w13t,
                       static_cast<uint64_t>(E) * (L->w13_rows / 128) * (L->xb / 128) *
                           weight_tile_bytes(L->fmt) / 2048) &&
         make_tile_map(&L->maps2.b, L->w2t,
                       static_cast<uint64_t>(E) * (H / 128) * (L->hb / 128) *
                           weight_tile_bytes(L->fmt) / 2048);
  ok = ok && cudaDeviceSynchronize() == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    free_all(L);
    delete L;
    return MOE_ERR_CUDA;
  }
  *out = L;
  return MOE_OK;
}

moe_status moe_prepare_weights(moe_layer* L, const void* w13, const void* w13_sf,
                               const float* w13_gs, const void* w2, const void* w2_sf,
                               const float* w2_gs, void* stream) {
  if (!L || !w13 || !w2) return MOE_ERR_INVALID_ARG;
  if (L->fmt != MOE_FMT_BF16 && (!w13_sf || !w2_sf)) return MOE_ERR_INVALID_ARG;
  if (L->fmt == MOE_FMT_NVFP4 && (!w13_gs || !w2_gs)) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  before_call(L, s);
  const int E = L->E, H = L->H, I = L->I;
  cudaError_t e = launch_tile_weights(L->fmt, static_cast<const uint8_t*>(w13),
                                      static_cast<const uint8_t*>(w13_sf), w13_gs, L->w13t, E,
                                      L->w13_rows, L->xb, L->x_tiles_k * 4,
                                      L->act == MOE_ACT_RELU2 ? 0 : I, s);
  if (e == cudaSuccess)
    e = launch_tile_weights(L->fmt, static_cast<const uint8_t*>(w2),
                            static_cast<const uint8_t*>(w2_sf), w2_gs, L->w2t, E, H, L->hb,
                            L->h_tiles_k * 4, 0, s);
  after_call(L, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  L->weights_ready = true;
  return MOE_OK;
}

// The kernels move activations with 16-byte vector accesses and read the
// logits as fp32.
bool io_aligned(const void* hidden, const void* logits, const void* out) {
  return ((reinterpret_cast<uintptr_t>(hidden) | reinterpret_cast<uintptr_t>(out)) & 15) == 0 &&
         (reinterpret_cast<uintptr_t>(logits) & 3) == 0;
}

}  // extern "C"

namespace {

// The routed forward on stream s.  front_done (if any) is recorded once the
// kernels that read `hidden` and `logits` have been enqueued; s waits for
// before_out (if any) before the first kernel that writes `out`.
moe_status forward_impl(moe_layer* L, const void* hidden, const float* logits, void* out, int T,
                        cudaStream_t s, cudaEvent_t front_done, cudaEvent_t before_out) {
  const int E = L->E, K = L->K, H = L->H;
  const int NB = (T + kTokensPerRouteBlock - 1) / kTokensPerRouteBlock;
  cudaEvent_t* ev = nullptr;
  if (L->timing_rec < L->timing_max) ev = &L->tev[static_cast<size_t>(L->timing_rec++) * 7];
  auto mark = [&](int i) {
    if (ev) cudaEventRecord(ev[i], s);
  };
  mark(0);
  cudaError_t e;
  int launches = 4;
  const bool small = T <= kSmallFrontTokens;
  const bool wide = L->wide_tiles == 1 || (L->wide_tiles < 0 && T > kPairCopyMaxTokens);
  // single-chunk experts' items mixed into the wide single-CTA GEMMs (the
  // CTA-pair kernels map items by expert)
  const bool mixed = L->mix_items && wide && !small && L->pair_clusters == 0;
  set_pdl(L, wide);
  // (the fused combine has the decode kernel's own combine for T <= 16)
  if (small && L->single_launch && L->fused_gemms && L->combine != MOE_COMBINE_REDUCE &&
      (L->stage_scales || L->fmt == MOE_FMT_BF16)) {
    // the whole layer in one launch (timed as GEMM1)
    GemmArgs a1 = gemm1_args(L, 1, false);
    const GemmArgs a2 = gemm2_args(L, 1, false, L->y, 0, nullptr);
    DecodeArgs d{};
    d.logits = logits;
    d.hidden = hidden;
    d.T = T;
    d.K = K;
    d.H = H;
    d.ids = L->ids;
    d.counts = L->counts;
    d.offsets = L->offsets;
    d.pad_off = L->pad_off;
    d.chunk_off = L->chunk_off;
    d.perm = L->perm;
    d.inv = L->inv;
    d.w = L->w;
    d.xq = L->xq;
    d.xsf = L->xsf;
    d.out = static_cast<uint8_t*>(out);
    d.ctl = L->dctl;
    const int64_t chunks = max_chunks(L, T);
    const int grid = static_cast<int>(
        std::min<int64_t>(L->max_ctas, chunks * (a1.n_tiles + a2.n_tiles)));
    mark(1);
    mark(2);
    mark(3);
    if (before_out) cudaStreamWaitEvent(s, before_out, 0);
    e = launch_decode(L->fmt, L->act == MOE_ACT_RELU2 ? 3 : 1, L->maps1, a1, L->maps2, a2, d,
                      grid, s);
    if (front_done) cudaEventRecord(front_done, s);
    mark(4);
    mark(5);
    mark(6);
    if (e != cudaSuccess) return MOE_ERR_CUDA;
    L->last_T = T;
    L->last_launches = 1;
    return MOE_OK;
  }
  if (small) {
    // one kernel for routing .. GEMM1 input (timed as the routing kernel)
    e = launch_small_front(L->fmt, logits, T, E, K, hidden, H, L->ids, L->w, L->counts,
                           L->offsets, L->pad_off, L->chunk_off, L->perm, L->inv, L->prow_slot,
                           L->done1, L->xq, L->xsf, s);
    mark(1);
    mark(2);
  } else {
    e = launch_route(logits, T, E, K, L->ids, L->w, L->blockhist, s);
    mark(1);
    if (e == cudaSuccess) e = launch_expert_scan(L->blockhist, NB, E, L->prefix, L->counts, s);
    mark(2);
    if (e == cudaSuccess)
      e = launch_scatter_quant(L->fmt, L->ids, T, E, K, hidden, H, L->prefix, L->counts,
                               L->offsets, L->pad_off, L->chunk_off, L->perm, L->inv,
                               L->prow_slot, mixed ? L->otab : nullptr, L->xq, L->xsf, s);
    launches = 6;
  }
  if (front_done) cudaEventRecord(front_done, s);
  mark(3);
  const int64_t chunks = max_chunks(L, T);
  const int pair = L->pair_scale_copies && T <= kPairCopyMaxTokens;
  // the fused combine runs in wide (prefill) GEMM2 launches only; narrower
  // launches keep the combine kernel (their GEMM2 kernels carry no gather)
  const bool fused_combine = L->combine == MOE_COMBINE_FUSED && wide && H % 256 == 0;
  void* reduce_out = L->combine == MOE_COMBINE_REDUCE || fused_combine ? out : nullptr;
  // decode: both GEMMs in one launch (for larger T the split measured faster)
  if (before_out && reduce_out) cudaStreamWaitEvent(s, before_out, 0);  // GEMM2 writes out
  if (small && !wide && L->fused_gemms) {
    // one launch for both GEMMs (timed as GEMM1)
    if (e == cudaSuccess) e = run_gemms_fused(L, chunks, T, pair, reduce_out, s);
    --launches;
    mark(4);
  } else {
    if (e == cudaSuccess) e = run_gemm1(L, chunks, T, pair, wide, s, mixed);
    mark(4);
    if (e == cudaSuccess) e = run_gemm2(L, chunks, T, pair, wide, L->y, 0, s, reduce_out, mixed);
  }
  mark(5);
  // with the in-kernel reduce or the fused combine GEMM2 has written `out` already
  if (e == cudaSuccess && reduce_out == nullptr) {
    if (before_out) cudaStreamWaitEvent(s, before_out, 0);
    e = launch_combine(L->y, L->inv, L->w, T, K, H, out, s);
  }
  else
    --launches;
  mark(6);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  L->last_T = T;
  L->last_launches = launches;
  return MOE_OK;
}

}  // namespace

extern "C" {

moe_status moe_forward(moe_layer* L, const void* hidden, const float* logits, void* out, int T,
                       void* stream) {
  if (!L || T < 0 || T > L->Tmax) return MOE_ERR_INVALID_ARG;
  if (T == 0) {
    L->last_T = 0;
    L->last_launches = 0;
    return MOE_OK;
  }
  if (!hidden || !logits || !out || !io_aligned(hidden, logits, out)) return MOE_ERR_INVALID_ARG;
  if (!L->weights_ready) return MOE_ERR_NO_WEIGHTS;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  before_call(L, s);
  const moe_status st = forward_impl(L, hidden, logits, out, T, s, nullptr, nullptr);
  after_call(L, s);
  return st;
}

moe_status moe_forward_batched(moe_layer* L, const void* hidden, const int32_t* counts, int M,
                               void* out, void* stream) {
  if (!L || M < 0) return MOE_ERR_INVALID_ARG;
  if (M == 0) return MOE_OK;
  if (!hidden || !counts || !out || !io_aligned(hidden, counts, out)) return MOE_ERR_INVALID_ARG;
  if (!L->weights_ready) return MOE_ERR_NO_WEIGHTS;
  const int64_t mpad = (static_cast<int64_t>(M) + kRowBlock - 1) / kRowBlock * kRowBlock;
  if (mpad * L->E > L->Rpad) return MOE_ERR_UNSUPPORTED;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int64_t chunks = mpad / kRowBlock * L->E;
  // every chunk holds at most 32 rows when M <= 32: the lanes-0-31 scale copies apply
  const int pair = L->pair_scale_copies && M <= 32;
  const bool wide = L->wide_tiles == 1 || (L->wide_tiles < 0 && M >= 256);
  set_pdl(L, wide);
  before_call(L, s);
  cudaError_t e = launch_batched_quant(L->fmt, hidden, counts, M, L->E, L->H, L->counts,
                                       L->offsets, L->pad_off, L->chunk_off, L->xq, L->xsf,
                                       L->status, s);
  if (e == cudaSuccess) e = run_gemm1(L, chunks, M, pair, wide, s);
  if (e == cudaSuccess) e = run_gemm2(L, chunks, M, pair, wide, out, M, s);
  after_call(L, s);
  if (e != cudaSuccess) return MOE_ERR_CUDA;
  L->last_T = 0;
  L->last_launches = 3;
  return MOE_OK;
}

moe_status moe_forward_host(moe_layer* L, const void* hidden_host, const float* logits_host,
                            void* out_host, int T, void* stream) {
  if (!L || T < 0 || T > L->Tmax) return MOE_ERR_INVALID_ARG;
  if (T == 0) return moe_forward(L, nullptr, nullptr, nullptr, 0, stream);
  if (!hidden_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (!L->weights_ready) return MOE_ERR_NO_WEIGHTS;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // (synchronous: a pipeline of moe_forward_host_async steps on the layer
  // finishes first, since this call reuses its device buffers)
  if (L->cs && (cudaStreamSynchronize(L->xi) != cudaSuccess ||
                cudaStreamSynchronize(L->cs) != cudaSuccess ||
                cudaStreamSynchronize(L->xo) != cudaSuccess))
    return MOE_ERR_CUDA;
  // Page-locked host buffers the device can address (on a Grace-Blackwell
  // node over NVLink-C2C) are read and written by the kernels in place: the
  // front end reads the hidden states and logits, the combine writes the
  // output, with no separate copies.  Other host memory is copied.
  void* hd = L->host_zero_copy ? device_view(hidden_host) : nullptr;
  void* ld = L->host_zero_copy ? device_view(logits_host) : nullptr;
  void* od = L->host_zero_copy ? device_view(out_host) : nullptr;
  if (hd && ld && od && io_aligned(hd, ld, od)) {
    moe_status st = moe_forward(L, hd, static_cast<const float*>(ld), od, T, stream);
    if (st != MOE_OK) return st;
    return cudaStreamSynchronize(s) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
  }
  const size_t hb = static_cast<size_t>(T) * L->H * 2, lb = static_cast<size_t>(T) * L->E * 4;
  if (cudaMemcpyAsync(L->h_in, hidden_host, hb, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(L->l_in, logits_host, lb, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return MOE_ERR_CUDA;
  moe_status st = moe_forward(L, L->h_in, L->l_in, L->o_out, T, stream);
  if (st != MOE_OK) return st;
  if (cudaMemcpyAsync(out_host, L->o_out, hb, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaStreamSynchronize(s) != cudaSuccess)
    return MOE_ERR_CUDA;
  return MOE_OK;
}

moe_status moe_forward_host_async(moe_layer* L, const void* hidden_host, const float* logits_host,
                                  void* out_host, int T, void* stream) {
  if (!L || T < 0 || T > L->Tmax) return MOE_ERR_INVALID_ARG;
  if (T == 0) return moe_forward(L, nullptr, nullptr, nullptr, 0, stream);
  if (!hidden_host || !logits_host || !out_host) return MOE_ERR_INVALID_ARG;
  if (!L->weights_ready) return MOE_ERR_NO_WEIGHTS;
  if (!L->cs) {
    bool ok = true;
    for (cudaStream_t* x : {&L->xi, &L->xo, &L->cs})
      ok = ok && cudaStreamCreateWithFlags(x, cudaStreamNonBlocking) == cudaSuccess;
    for (cudaEvent_t* e : {&L->ev_in, &L->ev_front, &L->ev_comb, &L->ev_d2h, &L->ev_user})
      ok = ok && cudaEventCreateWithFlags(e, cudaEventDisableTiming) == cudaSuccess;
    if (!ok) {
      cudaGetLastError();
      return MOE_ERR_CUDA;
    }
  }
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // Decode-sized steps whose buffers the GPU can address in place (pinned
  // memory over NVLink-C2C) skip the copies: the single-launch decode kernel
  // reads the inputs and writes the output in host memory, and a step costs
  // the host one launch instead of three copies besides.
  if (L->host_zero_copy && T <= kSmallFrontTokens) {
    void* hd = device_view(hidden_host);
    void* ld = device_view(logits_host);
    void* od = device_view(out_host);
    if (hd && ld && od && io_aligned(hd, ld, od)) {
      if (cudaStreamWaitEvent(L->cs, L->ev_user, 0) != cudaSuccess) return MOE_ERR_CUDA;
      moe_status st = forward_impl(L, hd, static_cast<const float*>(ld), od, T, L->cs, nullptr,
                                   nullptr);
      if (st != MOE_OK) return st;
      return cudaEventRecord(L->ev_comb, L->cs) == cudaSuccess &&
                     cudaStreamWaitEvent(s, L->ev_comb, 0) == cudaSuccess
                 ? MOE_OK
                 : MOE_ERR_CUDA;
    }
  }
  const size_t hb = static_cast<size_t>(T) * L->H * 2, lb = static_cast<size_t>(T) * L->E * 4;
  // The input copies wait until the previous step's front end has read
  // h_in and l_in; the layer waits for them and for the latest work other
  // entry points enqueued on the layer; its output kernel waits until the
  // previous step's output copy has read o_out.  (Waiting on an event that
  // was never recorded is a no-op.)
  bool ok = cudaStreamWaitEvent(L->xi, L->ev_front, 0) == cudaSuccess &&
            cudaMemcpyAsync(L->h_in, hidden_host, hb, cudaMemcpyHostToDevice, L->xi) ==
                cudaSuccess &&
            cudaMemcpyAsync(L->l_in, logits_host, lb, cudaMemcpyHostToDevice, L->xi) ==
                cudaSuccess &&
            cudaEventRecord(L->ev_in, L->xi) == cudaSuccess &&
            cudaStreamWaitEvent(L->cs, L->ev_in, 0) == cudaSuccess &&
            cudaStreamWaitEvent(L->cs, L->ev_user, 0) == cudaSuccess;
  if (!ok) return MOE_ERR_CUDA;
  moe_status st = forward_impl(L, L->h_in, L->l_in, L->o_out, T, L->cs, L->ev_front, L->ev_d2h);
  if (st != MOE_OK) return st;
  // the caller's stream completes once out_host holds the result; nothing
  // of the layer waits on the caller's stream, so consecutive steps overlap
  ok = cudaEventRecord(L->ev_comb, L->cs) == cudaSuccess &&
       cudaStreamWaitEvent(L->xo, L->ev_comb, 0) == cudaSuccess &&
       cudaMemcpyAsync(out_host, L->o_out, hb, cudaMemcpyDeviceToHost, L->xo) == cudaSuccess &&
       cudaEventRecord(L->ev_d2h, L->xo) == cudaSuccess &&
       cudaStreamWaitEvent(s, L->ev_d2h, 0) == cudaSuccess;
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_debug_routing(moe_layer* L, int32_t* topk_ids, float* topk_w, int32_t* offsets,
                             int32_t* perm, void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t R = static_cast<size_t>(L->last_T) * L->K;
  before_call(L, s);
  bool ok = true;
  if (topk_ids && R) ok &= cudaMemcpyAsync(topk_ids, L->ids, R * 4, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  if (topk_w && R) ok &= cudaMemcpyAsync(topk_w, L->w, R * 4, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  if (offsets && R)
    ok &= cudaMemcpyAsync(offsets, L->offsets, (L->E + 1) * 4, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  if (perm && R) ok &= cudaMemcpyAsync(perm, L->perm, R * 4, cudaMemcpyDeviceToDevice, s) == cudaSuccess;
  after_call(L, s);
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_debug_act_quant(moe_layer* L, uint8_t* codes, uint8_t* scales, void* stream) {
  if (!L || !codes || !scales) return MOE_ERR_INVALID_ARG;
  if (L->fmt == MOE_FMT_BF16) return MOE_ERR_UNSUPPORTED;
  if (L->last_T == 0) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  before_call(L, s);
  const bool ok = launch_debug_act(L->fmt, L->inv, L->last_T, L->K, L->H, L->xq, L->xsf, codes,
                                   scales, s) == cudaSuccess;
  after_call(L, s);
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_debug_weight_tiles(moe_layer* L, int which, int expert, void* dst,
                                  size_t dst_bytes, void* stream) {
  if (!L || !dst || (which != 13 && which != 2) || expert < 0 || expert >= L->E)
    return MOE_ERR_INVALID_ARG;
  if (!L->weights_ready) return MOE_ERR_NO_WEIGHTS;
  const int rows = which == 13 ? L->w13_rows : L->H;
  const int row_bytes = which == 13 ? L->xb : L->hb;
  const size_t per_expert =
      static_cast<size_t>(rows / 128) * (row_bytes / 128) * weight_tile_bytes(L->fmt);
  if (dst_bytes != per_expert) return MOE_ERR_INVALID_ARG;
  const uint8_t* src = (which == 13 ? L->w13t : L->w2t) + per_expert * expert;
  return cudaMemcpyAsync(dst, src, per_expert, cudaMemcpyDefault,
                         static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_CUDA;
}

moe_status moe_debug_intermediates(moe_layer* L, float* h, float* y, void* stream) {
  if (!L) return MOE_ERR_INVALID_ARG;
  const int R = L->last_T * L->K;
  if (R == 0 || (!h && !y)) return MOE_OK;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  before_call(L, s);
  const bool ok = launch_debug_rows(L->fmt, L->offsets, L->pad_off, L->E, R, L->I, L->H, L->hq,
                                    L->hsf, L->y, h, y, s) == cudaSuccess;
  after_call(L, s);
  return ok ? MOE_OK : MOE_ERR_CUDA;
}

moe_status moe_get_status(moe_layer* L) {
  if (!L) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return MOE_ERR_CUDA;
  }
  int v = 0;
  if (cudaMemcpy(&v, L->status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess)
    return MOE_ERR_CUDA;
  if (v != 0) {
    cudaMemset(L->status, 0, sizeof(int));
    return v == kStatusBadCount ? MOE_ERR_INVALID_ARG : MOE_ERR_DEVICE_TIMEOUT;
  }
  return MOE_OK;
}

moe_status moe_timing_start(moe_layer* L, int max_forwards) {
  if (!L || max_forwards < 1) return MOE_ERR_INVALID_ARG;
  for (cudaEvent_t e : L->tev) cudaEventDestroy(e);
  L->tev.assign(static_cast<size_t>(max_forwards) * 7, nullptr);
  for (auto& e : L->tev)
    if (cudaEventCreate(&e) != cudaSuccess) {
      cudaGetLastError();
      for (cudaEvent_t x : L->tev)
        if (x) cudaEventDestroy(x);
      L->tev.clear();
      L->timing_max = L->timing_rec = 0;
      return MOE_ERR_CUDA;
    }
  L->timing_max = max_forwards;
  L->timing_rec = 0;
  return MOE_OK;
}

moe_status moe_timing_stop(moe_layer* L, float* kernel_ms, int* forwards) {
  if (!L) return MOE_ERR_INVALID_ARG;
  moe_status st = MOE_OK;
  float sum[6] = {0, 0, 0, 0, 0, 0};
  const int n = L->timing_rec;
  if (n > 0 && cudaEventSynchronize(L->tev[static_cast<size_t>(n) * 7 - 1]) != cudaSuccess)
    st = MOE_ERR_CUDA;
  for (int f = 0; f < n && st == MOE_OK; ++f)
    for (int k = 0; k < 6; ++k) {
      float ms = 0.0f;
      if (cudaEventElapsedTime(&ms, L->tev[f * 7 + k], L->tev[f * 7 + k + 1]) != cudaSuccess) {
        st = MOE_ERR_CUDA;
        break;
      }
      sum[k] += ms;
    }
  for (cudaEvent_t e : L->tev) cudaEventDestroy(e);
  L->tev.clear();
  L->timing_max = L->timing_rec = 0;
  if (st != MOE_OK) cudaGetLastError();
  if (kernel_ms)
    for (int k = 0; k < 6; ++k) kernel_ms[k] = sum[k];
  if (forwards) *forwards = n;
  return st;
}

int moe_last_launch_count(const moe_layer* L) { return L ? L->last_launches : 0; }

int moe_gemm_ctas(const moe_layer* L, int wide) {
  if (!L) return 0;
  if (wide && L->pair_clusters > 0)
    return 2 * std::min(L->pair_clusters, std::max(1, L->max_ctas / 2));
  return L->max_ctas;
}

void moe_destroy(moe_layer* L) {
  if (!L) return;
  cudaDeviceSynchronize();
  for (cudaEvent_t e : L->tev) cudaEventDestroy(e);
  for (cudaEvent_t e : {L->ev_in, L->ev_front, L->ev_comb, L->ev_d2h, L->ev_user})
    if (e) cudaEventDestroy(e);
  for (cudaStream_t x : {L->xi, L->xo, L->cs})
    if (x) cudaStreamDestroy(x);
  free_all(L);
  delete L;
}

}  // extern "C"
