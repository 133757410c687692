// route_token.cuh -- one warp routes one token: the K largest router logits
// in the total order (value descending, lower expert index first on ties,
// -0.0 equal to +0.0) and the softmax of those K values.  Shared by the
// layer's routing kernels and the no-allocation routing entry point, so
// both compute exactly the same ids and weights.
//
// Routing is the first step of the fused layer, which the b12x integration
// runs with both expert GEMMs and the reduction in one call (PR #40082
// report, sec. 实现拆解 item 1).
#pragma once

#include <cstdint>

namespace moe {

// Order-preserving 32-bit key of a router logit: larger value -> larger
// key, -0.0 and +0.0 the same key, every finite or infinite value >= 1 (0
// marks an empty slot).  NaN logits are not supported.
__device__ __forceinline__ uint32_t logit_key(float x) {
  uint32_t b = __float_as_uint(x);
  if (b == 0x80000000u) b = 0u;  // -0.0 == +0.0
  return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_logit(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k);
}

// Lane l holds logits l, l+32, ... (MAXJ of them, E <= 32 MAXJ).  Each of
// the K rounds takes the warp's largest key (redux.sync max), then the
// lowest expert index holding it (redux.sync min), and removes that entry;
// then the softmax of the K selected values.  Lane k < K receives the k-th
// expert in *id and its softmax weight in *wt; the other lanes receive
// weight 0.
template <int MAXJ>
__device__ __forceinline__ void route_token(const float* __restrict__ l, int E, int K, int lane,
                                            int* id, float* wt) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  float my_v = 0.0f;
  int my_i = 0;
  {
    uint32_t key[MAXJ];
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = lane + 32 * j;
      key[j] = e < E ? logit_key(__ldg(l + e)) : 0u;
    }
    for (int k = 0; k < K; ++k) {
      uint32_t m = 0u;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j) m = max(m, key[j]);
      const uint32_t wmax = __reduce_max_sync(kAll, m);
      uint32_t idx = 0xFFFFFFFFu;
#pragma unroll
      for (int j = MAXJ - 1; j >= 0; --j)
        if (key[j] == wmax) idx = static_cast<uint32_t>(lane + 32 * j);
      const uint32_t widx = __reduce_min_sync(kAll, idx);
      if (static_cast<int>(widx & 31u) == lane) {
#pragma unroll
        for (int j = 0; j < MAXJ; ++j)
          if (static_cast<uint32_t>(j) == (widx >> 5)) key[j] = 0u;
      }
      if (lane == k) {
        my_v = key_logit(wmax);
        my_i = static_cast<int>(widx);
      }
    }
  }
  const float m = __shfl_sync(kAll, my_v, 0);
  const float ex = lane < K ? expf(my_v - m) : 0.0f;
  float sum = ex;
#pragma unroll
  for (int off = 16; off; off >>= 1) sum += __shfl_xor_sync(kAll, sum, off);
  *id = my_i;
  *wt = ex / sum;
}

}  // namespace moe
