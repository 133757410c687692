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

#include <cfloat>
#include <climits>
#include <cstdint>

namespace moe {

// Lane l holds logits l, l+32, ... (MAXJ of them, E <= 32 MAXJ); K rounds of
// a warp arg-max in the total order, then the softmax of the K selected
// values.  Lane k < K receives the k-th expert in *id and its softmax weight
// in *wt; the other lanes receive weight 0.
template <int MAXJ>
__device__ __forceinline__ void route_token(const float* __restrict__ l, int E, int K, int lane,
                                            int* id, float* wt) {
  constexpr unsigned kAll = 0xFFFFFFFFu;
  float my_v = 0.0f;
  int my_i = 0;
  {
    float v[MAXJ];
    uint32_t avail = 0;
#pragma unroll
    for (int j = 0; j < MAXJ; ++j) {
      const int e = lane + 32 * j;
      v[j] = -FLT_MAX;
      if (e < E) {
        v[j] = __ldg(l + e);
        avail |= 1u << j;
      }
    }
    for (int k = 0; k < K; ++k) {
      float bv = -FLT_MAX;
      int bi = INT_MAX;
#pragma unroll
      for (int j = 0; j < MAXJ; ++j)
        if (((avail >> j) & 1u) && (bi == INT_MAX || v[j] > bv)) {
          bv = v[j];
          bi = lane + 32 * j;
        }
#pragma unroll
      for (int off = 16; off; off >>= 1) {
        const float ov = __shfl_xor_sync(kAll, bv, off);
        const int oi = __shfl_xor_sync(kAll, bi, off);
        const bool take = oi != INT_MAX && (bi == INT_MAX || ov > bv || (ov == bv && oi < bi));
        if (take) {
          bv = ov;
          bi = oi;
        }
      }
      if ((bi & 31) == lane) avail &= ~(1u << (bi >> 5));
      if (lane == k) {
        my_v = bv;
        my_i = bi;
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
