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

// The same selection and weights for G tokens at once in one warp: token g's
// logits in v[g] (padding as above), written when valid[g]. The G tokens'
// butterflies are interleaved (the one-token form is bound by shuffle
// latency); the arithmetic per token, and so every result, is that of
// warp_select_and_weigh.
template <int NJ, int G>
__device__ __forceinline__ void warp_select_and_weigh_g(const float (&v)[G][NJ],
                                                        const int (&id)[G][NJ], int k, int pre_k,
                                                        int router, const int (&t)[G],
                                                        const bool (&valid)[G],
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  static_assert(NJ <= 32, "taken bits");
  const int lane = threadIdx.x & 31;
  uint32_t taken[G];
#pragma unroll
  for (int g = 0; g < G; ++g) taken[g] = 0u;
  float sel_v[G][kMaxTopK];
  int sel_i[G][kMaxTopK];
  const int rounds = (router == kRouterRenorm) ? k : pre_k;
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
#pragma unroll
    for (int g = 0; g < G; ++g) {
      sel_v[g][s] = -FLT_MAX;
      sel_i[g][s] = 0x7fffffff;
    }
    if (s < rounds) {
      float bv[G];
      int bi[G];
#pragma unroll
      for (int g = 0; g < G; ++g) {
        bv[g] = -INFINITY;
        bi[g] = 0x7fffffff;
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          if (!((taken[g] >> j) & 1u) && beats(v[g][j], id[g][j], bv[g], bi[g])) {
            bv[g] = v[g][j];
            bi[g] = id[g][j];
          }
      }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
          const float ov = __shfl_xor_sync(0xffffffffu, bv[g], off);
          const int oi = __shfl_xor_sync(0xffffffffu, bi[g], off);
          if (beats(ov, oi, bv[g], bi[g])) {
            bv[g] = ov;
            bi[g] = oi;
          }
        }
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        sel_v[g][s] = bv[g];
        sel_i[g][s] = bi[g];
#pragma unroll
        for (int j = 0; j < NJ; ++j)
          if (id[g][j] == bi[g]) taken[g] |= 1u << j;
      }
    }
  }
#pragma unroll
  for (int g = 0; g < G; ++g) {
    const float m = sel_v[g][0];
    float den = 0.f;
    float ex[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      ex[s] = (s < rounds) ? expf(sel_v[g][s] - m) : 0.f;
      den += ex[s];
    }
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      if (valid[g] && s < k && lane == s) {
        topk_idx[static_cast<size_t>(t[g]) * k + s] = sel_i[g][s];
        topk_w[static_cast<size_t>(t[g]) * k + s] = ex[s] / den;
      }
    }
  }
}

// One thread per token: scan the token's E logits (row[e], e ascending) and
// keep the best kMaxTopK in a sorted list; the weights as above. Experts
// arrive in increasing id, so a logit equal to one already listed ranks
// after it and the insertion test is a strict `>`. The same ranking and the
// same weight arithmetic as the warp forms, without a warp-wide argmax per
// round (the warp forms spend ~1k instructions a token at pre_k = 8).
__device__ __forceinline__ void thread_select_and_weigh(const float* row, int E, int k, int pre_k,
                                                        int router, int t,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  float sv[kMaxTopK];
  int si[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sv[j] = -INFINITY;
    si[j] = 0x7fffffff;
  }
  for (int e = 0; e < E; ++e) {
    const float v = row[e];
    if (v > sv[kMaxTopK - 1]) {
      // shift the entries below the insertion point down by one
#pragma unroll
      for (int j = kMaxTopK - 1; j > 0; --j) {
        const bool down = v > sv[j - 1];
        const bool here = !down && v > sv[j];
        sv[j] = down ? sv[j - 1] : (here ? v : sv[j]);
        si[j] = down ? si[j - 1] : (here ? e : si[j]);
      }
      if (v > sv[0]) {
        sv[0] = v;
        si[0] = e;
      }
    }
  }
  const int rounds = (router == kRouterRenorm) ? k : pre_k;
  const float m = sv[0];
  float den = 0.f;
  float ex[kMaxTopK];
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    ex[s] = (s < rounds) ? expf(sv[s] - m) : 0.f;
    den += ex[s];
  }
#pragma unroll
  for (int s = 0; s < kMaxTopK; ++s) {
    if (s < k) {
      topk_idx[static_cast<size_t>(t) * k + s] = si[s];
      topk_w[static_cast<size_t>(t) * k + s] = ex[s] / den;
    }
  }
}

}  // namespace topk
}  // namespace moe
