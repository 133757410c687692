// route_static.cu -- routing and expert permutation for callers that cannot
// allocate device memory.
//
// moe_create allocates every buffer a layer needs.  Some callers cannot do
// that: a serving framework whose caching allocator has already reserved the
// whole GPU, or a latency-critical caller that cannot accept the device-wide
// synchronisation cudaMalloc/cudaFree may cause.  For them this file offers
// the routing + histogram / scan / scatter step as one entry point that
// allocates nothing.  The caller passes the router logits and the output
// buffers; the per-block histograms and bases the step needs live in one
// file-scope device array of fixed size (kStaticScratchInts int32, 256 KiB),
// which every GPU that loads this library holds until the process exits.
//
// Device code could name the array directly, but host code must not pass its
// name to a kernel: on the host the name is only a stand-in, not a device
// address.  The entry point therefore looks the address up once per device
// (cudaGetSymbolAddress, with that device current) on its first call there.
//
// All calls share the array and it keeps the previous call's contents.
// Every entry a call reads is written earlier in that same call, so nothing
// has to be cleared between calls; but two calls whose kernels overlap on the
// GPU (different streams, or different host threads without ordering) race
// on the array and produce garbage.
#include <mutex>

#include "internal.h"
#include "moe.h"
#include "route_token.cuh"

namespace moe {

namespace {

constexpr int kStaticMaxTokens = 4096;
constexpr int kStaticBlockTokens = 64;
constexpr int kStaticMaxBlocks = kStaticMaxTokens / kStaticBlockTokens;  // 64
// [blocks][experts] histogram, then [blocks][experts] first row per block
constexpr int kStaticScratchInts = 2 * kStaticMaxBlocks * kMaxExperts;   // 65536

static __device__ __align__(256) int32_t g_static_scratch[kStaticScratchInts];

constexpr unsigned kAll = 0xFFFFFFFFu;

// One warp per token (route_token, the same router moe_forward uses); block
// b counts its 64 tokens' slots per expert.
__global__ void __launch_bounds__(256) static_route_kernel(const float* __restrict__ logits, int T,
                                                           int E, int K, int32_t* __restrict__ ids,
                                                           float* __restrict__ w,
                                                           int32_t* __restrict__ hist_out) {
  __shared__ int hist[kMaxExperts];
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist[e] = 0;
  __syncthreads();
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  for (int i = warp; i < kStaticBlockTokens; i += 8) {
    const int t = blockIdx.x * kStaticBlockTokens + i;
    if (t >= T) break;
    int my_i;
    float my_w;
    route_token<kMaxExperts / 32>(logits + static_cast<int64_t>(t) * E, E, K, lane, &my_i, &my_w);
    if (lane < K) {
      ids[static_cast<int64_t>(t) * K + lane] = my_i;
      w[static_cast<int64_t>(t) * K + lane] = my_w;
      atomicAdd(&hist[my_i], 1);
    }
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x) hist_out[blockIdx.x * E + e] = hist[e];
}

// One block, thread e = expert: offsets (exclusive scan of the per-expert
// counts) and the first permuted row of each (block, expert) pair.
__global__ void __launch_bounds__(kMaxExperts) static_scan_kernel(const int32_t* __restrict__ hist,
                                                                  int NB, int E,
                                                                  int32_t* __restrict__ offsets,
                                                                  int32_t* __restrict__ base) {
  __shared__ int wsum[kMaxExperts / 32];
  const int e = threadIdx.x, lane = e & 31, warp = e >> 5;
  int c = 0;
  if (e < E)
    for (int b = 0; b < NB; ++b) c += hist[b * E + e];
  int inc = c;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kAll, inc, off);
    if (lane >= off) inc += o;
  }
  if (lane == 31) wsum[warp] = inc;
  __syncthreads();
  int ex = inc - c;
  for (int w2 = 0; w2 < warp; ++w2) ex += wsum[w2];
  if (e < E) {
    offsets[e] = ex;
    if (e == E - 1) offsets[E] = ex + c;
    int run = ex;
    for (int b = 0; b < NB; ++b) {
      base[b * E + e] = run;
      run += hist[b * E + e];
    }
  }
}

// Block b walks its slots in order and gives each the next row of its
// expert (stable in the slot index t*K + k).
__global__ void __launch_bounds__(32) static_rank_kernel(const int32_t* __restrict__ ids, int T,
                                                         int E, int K,
                                                         const int32_t* __restrict__ base,
                                                         int32_t* __restrict__ perm) {
  __shared__ int cnt[kMaxExperts];
  const int lane = threadIdx.x;
  for (int e = lane; e < E; e += 32) cnt[e] = 0;
  __syncwarp();
  const int tok0 = blockIdx.x * kStaticBlockTokens;
  const int ntok = min(kStaticBlockTokens, T - tok0);
  for (int i = 0; i < ntok; ++i) {
    if (lane < K) {
      const int64_t s = static_cast<int64_t>(tok0 + i) * K + lane;
      const int e = ids[s];
      const int r = cnt[e];
      cnt[e] = r + 1;  // the K experts of one token are distinct
      perm[base[blockIdx.x * E + e] + r] = static_cast<int32_t>(s);
    }
    __syncwarp();
  }
}

// Device address of g_static_scratch per device, looked up once.
constexpr int kMaxDevices = 64;
std::mutex g_scratch_mu;
int32_t* g_scratch_ptr[kMaxDevices] = {};

cudaError_t static_scratch(int32_t** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_scratch_mu);
  if (!g_scratch_ptr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_static_scratch);
    if (e != cudaSuccess) return e;
    g_scratch_ptr[dev] = static_cast<int32_t*>(p);
  }
  *out = g_scratch_ptr[dev];
  return cudaSuccess;
}

}  // namespace

}  // namespace moe

// Every pointer is read or written as 32-bit words by the kernels.
static bool aligned4(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 3) == 0; }

extern "C" moe_status moe_route_permute_static(const float* router_logits, int T, int E, int K,
                                               int32_t* topk_ids, float* topk_w,
                                               int32_t* offsets, int32_t* perm, void* stream) {
  using namespace moe;
  if (T < 0 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
  if (T > kStaticMaxTokens || E > kMaxExperts || K > kMaxTopK) return MOE_ERR_UNSUPPORTED;
  if (T == 0) return MOE_OK;
  if (!router_logits || !topk_ids || !topk_w || !offsets || !perm) return MOE_ERR_INVALID_ARG;
  if (!aligned4(router_logits) || !aligned4(topk_ids) || !aligned4(topk_w) ||
      !aligned4(offsets) || !aligned4(perm))
    return MOE_ERR_INVALID_ARG;
  int32_t* scratch = nullptr;
  if (static_scratch(&scratch) != cudaSuccess) {
    cudaGetLastError();  // the failed look-up's own error, not a sticky one
    return MOE_ERR_CUDA;
  }
  int32_t* hist = scratch;
  int32_t* base = scratch + kStaticMaxBlocks * kMaxExperts;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const int NB = (T + kStaticBlockTokens - 1) / kStaticBlockTokens;
  // each launch reports its own error; an earlier, unrelated error of the
  // context is neither reported here nor cleared
  cudaError_t e = launch_pdl(false, static_route_kernel, dim3(NB), dim3(256), 0, s, router_logits,
                             T, E, K, topk_ids, topk_w, hist);
  if (e == cudaSuccess)
    e = launch_pdl(false, static_scan_kernel, dim3(1), dim3(kMaxExperts), 0, s, hist, NB, E,
                   offsets, base);
  if (e == cudaSuccess)
    e = launch_pdl(false, static_rank_kernel, dim3(NB), dim3(32), 0, s, topk_ids, T, E, K, base,
                   perm);
  return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
