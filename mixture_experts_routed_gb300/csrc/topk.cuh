// topk.cuh - the router's selection and weighting step for one token
// (DeepSeek-V4 EP article, section 3.2): the top pre_k (or k) logits under
// (logit descending, lower expert id first), then the weights from
// max-subtracted exponentials of the chosen logits. The group-limited mode
// first drops every expert outside the topk_group groups with the best mean
// probability (the node limit of the DeepSeek V3/V4 parallel-strategy
// article, EP section). Soft gating weights every expert instead. Two
// forms: one warp per token (SIMT gate kernels) and one thread per token
// (tensor-core gate).
#pragma once

#include <cfloat>
#include <cstdint>

#include "common.cuh"

namespace moe {
namespace topk {

constexpr int kRouterRenorm = 0;
constexpr int kRouterPrek = 1;
constexpr int kRouterGroup = 2;
constexpr int kRouterSoft = 3;

// Ranking rule: a beats b if a has the larger value, or equal values and the
// lower id (expert or group).
__device__ __forceinline__ bool beats(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

// Selection rounds: the pre_k softmax router ranks pre_k experts, the others k.
__device__ __forceinline__ int rounds_of(const RouterSpec& rs) {
  return rs.mode == kRouterPrek ? rs.pre_k : rs.k;
}

// Group-limited mode, warp form: the lanes hold NJ (logit, id) pairs each
// (padding: -inf and an id >= E). Group g (experts g*gs .. g*gs+gs-1, gs =
// E/n_group) scores sum_e exp(L_e - L_max), which ranks the groups as their
// mean probability does (common factors dropped). Experts outside the
// topk_group best groups (ties: lower group id) get -inf, so the following
// top-k sees only the kept groups.
template <int NJ>
__device__ __forceinline__ void warp_group_limit(float (&v)[NJ], const int (&id)[NJ], int E,
                                                 const RouterSpec& rs) {
  const int lane = threadIdx.x & 31;
  const int ng = rs.n_group, gs = E / ng;
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j) m = fmaxf(m, v[j]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float ex[NJ];
  int grp[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    const bool real = id[j] < E;
    ex[j] = real ? expf(v[j] - m) : 0.f;
    grp[j] = real ? id[j] / gs : -1;
  }
  float mine = 0.f;  // lane g < ng: group g's score
  for (int g = 0; g < ng; ++g) {
    float s = 0.f;
#pragma unroll
    for (int j = 0; j < NJ; ++j) s += (grp[j] == g) ? ex[j] : 0.f;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) s += __shfl_xor_sync(0xffffffffu, s, off);
    if (lane == g) mine = s;
  }
  int rank = 0;  // groups that beat this lane's group
  for (int g = 0; g < ng; ++g) {
    const float o = __shfl_sync(0xffffffffu, mine, g);
    rank += beats(o, g, mine, lane) ? 1 : 0;
  }
  const uint32_t keep = __ballot_sync(0xffffffffu, lane < ng && rank < rs.topk_group);
#pragma unroll
  for (int j = 0; j < NJ; ++j)
    if (grp[j] >= 0 && !((keep >> grp[j]) & 1u)) v[j] = -INFINITY;
}

// Warp form: each lane holds NJ (logit, expert id) pairs; padding uses -inf
// and an id >= E. Selects the top rounds_of(rs) by repeated warp argmax and
// writes slots j < k of token t.
template <int NJ>
__device__ __forceinline__ void warp_select_and_weigh(const float (&v)[NJ], const int (&id)[NJ],
                                                      const RouterSpec& rs, int t,
                                                      int32_t* __restrict__ topk_idx,
                                                      float* __restrict__ topk_w) {
  const int lane = threadIdx.x & 31;
  const int k = rs.k;
  bool taken[NJ];
#pragma unroll
  for (int j = 0; j < NJ; ++j) taken[j] = false;
  float sel_v[kMaxTopK];
  int sel_i[kMaxTopK];
  const int rounds = rounds_of(rs);
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

// Group-limited mode, thread form: the bit mask of the kept groups of one
// logits row (same scores and ranking as warp_group_limit).
__device__ __forceinline__ uint32_t thread_group_keep(const float* row, int E,
                                                      const RouterSpec& rs) {
  const int ng = rs.n_group, gs = E / ng;
  float m = -INFINITY;
  for (int e = 0; e < E; ++e) m = fmaxf(m, row[e]);
  float sg[kMaxGroups];
  for (int g = 0; g < ng; ++g) {
    float s = 0.f;
    for (int e = g * gs; e < (g + 1) * gs; ++e) s += expf(row[e] - m);
    sg[g] = s;
  }
  uint32_t keep = 0u;
  for (int g = 0; g < ng; ++g) {
    int rank = 0;
    for (int h = 0; h < ng; ++h) rank += beats(sg[h], h, sg[g], g) ? 1 : 0;
    if (rank < rs.topk_group) keep |= 1u << g;
  }
  return keep;
}

// Thread form: one thread per token scans the token's E logits (row[e], e
// ascending; in the group-limited mode only the kept groups' experts) and
// keeps the best kMaxTopK in a sorted list; the weights as above. Experts
// arrive in increasing id, so a logit equal to one already listed ranks
// after it and the insertion test is a strict `>`. The same ranking and the
// same weight arithmetic as the warp form, without a warp-wide argmax per
// round (the warp form spends ~1k instructions a token at pre_k = 8).
__device__ __forceinline__ void thread_select_and_weigh(const float* row, int E,
                                                        const RouterSpec& rs, int t,
                                                        int32_t* __restrict__ topk_idx,
                                                        float* __restrict__ topk_w) {
  const int k = rs.k;
  const bool grouped = rs.mode == kRouterGroup;
  const int ng = grouped ? rs.n_group : 1, gs = E / ng;
  const uint32_t keep = grouped ? thread_group_keep(row, E, rs) : 1u;
  float sv[kMaxTopK];
  int si[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sv[j] = -INFINITY;
    si[j] = 0x7fffffff;
  }
  for (int g = 0; g < ng; ++g) {
    if (!((keep >> g) & 1u)) continue;
    for (int e = g * gs; e < (g + 1) * gs; ++e) {
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
  }
  const int rounds = rounds_of(rs);
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

// G threads per token (G = 2 or 4 consecutive lanes of a warp, `h` = lane
// % G; every lane of the warp calls this; E a multiple of G): thread h keeps
// the best kMaxTopK of experts [h E/G, (h+1) E/G) by insertion (ascending
// ids, strict >: equal logits keep the lower id first); the sorted lists are
// merged pairwise at shuffle distance 1, then 2, each merge a bitonic step
// (element s against the partner's 7-s) and an 8-element bitonic sort under
// `beats`, which gives exactly the list one thread would keep over all E.
// Weights as thread_select_and_weigh (written by h = 0). Not for the
// group-limited or soft routers.
template <int G>
__device__ __forceinline__ void group_select_and_weigh(const float* row, int E,
                                                       const RouterSpec& rs, int t, int h,
                                                       bool active,
                                                       int32_t* __restrict__ topk_idx,
                                                       float* __restrict__ topk_w) {
  static_assert(G == 2 || G == 4, "2 or 4 threads per token");
  float sv[kMaxTopK];
  int si[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    sv[j] = -INFINITY;
    si[j] = 0x7fffffff;
  }
  const int hw = E / G;
  for (int e = h * hw; e < (h + 1) * hw; ++e) {
    const float v = row[e];
    if (v > sv[kMaxTopK - 1]) {
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
  // bitonic merges with the partner's list: c[s] = better of (mine[s],
  // partner[7 - s]) holds the best kMaxTopK of both as a bitonic sequence,
  // sorted again by three half-cleaner stages
#pragma unroll
  for (int dist = 1; dist < G; dist <<= 1) {
    float cv[kMaxTopK];
    int ci[kMaxTopK];
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      const float pv = __shfl_xor_sync(0xffffffffu, sv[kMaxTopK - 1 - s], dist);
      const int pi = __shfl_xor_sync(0xffffffffu, si[kMaxTopK - 1 - s], dist);
      const bool mine = beats(sv[s], si[s], pv, pi);
      cv[s] = mine ? sv[s] : pv;
      ci[s] = mine ? si[s] : pi;
    }
#pragma unroll
    for (int stride = kMaxTopK / 2; stride > 0; stride >>= 1) {
#pragma unroll
      for (int s = 0; s < kMaxTopK; ++s) {
        if ((s & stride) == 0) {
          const int o = s + stride;
          if (beats(cv[o], ci[o], cv[s], ci[s])) {
            const float tv = cv[s];
            const int ti = ci[s];
            cv[s] = cv[o];
            ci[s] = ci[o];
            cv[o] = tv;
            ci[o] = ti;
          }
        }
      }
    }
#pragma unroll
    for (int s = 0; s < kMaxTopK; ++s) {
      sv[s] = cv[s];
      si[s] = ci[s];
    }
  }
  if (!active || h != 0) return;
  const int k = rs.k;
  const int rounds = rounds_of(rs);
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

// Soft gating (Deepseek-MoE sync-tax article, section 3.3), warp form: lane
// values v[j] for experts id[j] (padding: id >= E); z = (L + g) / tau with
// the token's Gumbel samples g; w = exp(z - max z) / sum; slot j = expert j
// of a [T, E] routing.
template <int NJ>
__device__ __forceinline__ void warp_soft_weigh(const float (&v)[NJ], const int (&id)[NJ], int E,
                                                const RouterSpec& rs, int t,
                                                int32_t* __restrict__ topk_idx,
                                                float* __restrict__ topk_w) {
  const float* g = rs.noise + static_cast<size_t>(t) * E;
  float z[NJ];
  float m = -INFINITY;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    z[j] = (id[j] < E) ? (v[j] + __ldg(g + id[j])) / rs.tau : -INFINITY;
    m = fmaxf(m, z[j]);
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
  float ex[NJ];
  float den = 0.f;
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    ex[j] = (id[j] < E) ? expf(z[j] - m) : 0.f;
    den += ex[j];
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) den += __shfl_xor_sync(0xffffffffu, den, off);
#pragma unroll
  for (int j = 0; j < NJ; ++j) {
    if (id[j] < E) {
      topk_idx[static_cast<size_t>(t) * E + id[j]] = id[j];
      topk_w[static_cast<size_t>(t) * E + id[j]] = ex[j] / den;
    }
  }
}

// Soft gating, thread form (one thread per token, logits row in shared
// memory): the same arithmetic, with the sum in expert order.
__device__ __forceinline__ void thread_soft_weigh(const float* row, int E, const RouterSpec& rs,
                                                  int t, int32_t* __restrict__ topk_idx,
                                                  float* __restrict__ topk_w) {
  const float* g = rs.noise + static_cast<size_t>(t) * E;
  float m = -INFINITY;
  for (int e = 0; e < E; ++e) m = fmaxf(m, (row[e] + __ldg(g + e)) / rs.tau);
  float den = 0.f;
  for (int e = 0; e < E; ++e) den += expf((row[e] + __ldg(g + e)) / rs.tau - m);
  for (int e = 0; e < E; ++e) {
    topk_idx[static_cast<size_t>(t) * E + e] = e;
    topk_w[static_cast<size_t>(t) * E + e] = expf((row[e] + __ldg(g + e)) / rs.tau - m) / den;
  }
}

}  // namespace topk
}  // namespace moe
