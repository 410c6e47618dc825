// topk.cuh - the router's selection and weighting step for one token, done
// by one warp (DeepSeek-V4 EP article, section 3.2): pre_k rounds of a warp
// argmax under (logit descending, lower expert id first), then the weights
// from max-subtracted exponentials of the chosen logits. Shared by the SIMT
// and tensor-core gate kernels.
#pragma once

#include <cfloat>
#include <cstdint>

#include "common.cuh"

namespace moe {
namespace topk {

constexpr int kRouterRenorm = 0;

// Ranking rule: a beats b if a has the larger logit, or equal logits and the
// lower expert id.
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Each lane holds NJ (logit, expert id) pairs; padding uses -inf and an id
// >= E. Selects the top pre_k (or k, for renorm) by repeated warp argmax and
// writes slots j < k of token t.
template <int NJ>
__device__ __forceinline__ void warp_select_and_weigh(const float (&v)[NJ], const int (&id)[NJ],
                                                      int k, int pre_k, int router, int t,
                                                      int32_t* __restrict__ topk_idx,
                                                      float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  bool taken[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) taken[j] = false;
  float sel_v[kMaxTopK];
  int sel_i[kMaxTopK];
  const int rounds = (router == kRouterRenorm) ? k : pre_k;
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    sel_v[s] = -FLT_MAX;
    sel_i[s] = 0x7fffffff;
    if (s < rounds) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (!taken[j] && beats(v[j], id[j], bv, bi)) {
          bv = v[j];
          bi = id[j];
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (beats(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
      sel_v[s] = bv;
      sel_i[s] = bi;
#pragma unroll
      for (int j = 0; j < NJ; ++j)
        if (id[j] == bi) taken[j] = true;
    }
  }
  // weights: max-subtracted exponentials of the chosen logits
  const float m = sel_v[0];
  float den = 0.f;
  float ex[kMaxTopK];
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    ex[s] = (s < rounds) ? expf(sel_v[s] - m) : 0.f;
    den += ex[s];
  }
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    if (s < k && lane == s) {
      topk_idx[static_cast<size_t>(t) * k + s] = sel_i[s];
      topk_w[static_cast<size_t>(t) * k + s] = ex[s] / den;
    }
  }
}


}  // namespace topk
}  // namespace moe
