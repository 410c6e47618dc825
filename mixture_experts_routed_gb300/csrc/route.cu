// route.cu - gate projection fused with the router (DeepSeek-V4 EP article,
// sections 2.1 and 3.2): per token, logits L = x W_g + b in fp32, then a
// warp-level partial top-pre_k by repeated warp argmax (larger logit first,
// lower expert id on ties), then the weights:
//   renorm:        w_j = exp(L_j - L_max) / sum_{i<k} exp(L_i - L_max)
//                  (= the full max-subtracted softmax of the chosen experts
//                  divided by their sum)
//   pre_k softmax: w_j = exp(L_j - L_max) / sum_{i<pre_k} exp(L_i - L_max)
// The logits never go to HBM unless the caller asks for them.
//
// Two gate GEMM shapes:
//  * E <= 32 ("narrow"): 4 warps per token split the hidden dimension; each
//    thread accumulates its slice for all E experts, a butterfly reduces
//    inside each warp and the 4 warp partials are added in warp order.
//  * E > 32 ("wide"): a CTA computes a 32-token x E tile from shared-memory
//    staged x and W_g; each thread owns 4 tokens x E/32 experts, accumulates
//    32-long K chunks and folds them into the total with compensated
//    (Kahan) summation, which keeps |L - L_fp64| ~1e-7 at d = 7168.
#include <cfloat>
#include <cstdint>
#include <cstddef>
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRouterRenorm = 0;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

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

// ---------------------------------------------------------------- narrow
// E <= 32. A CTA of 4 warps handles TPB tokens; its 128 threads stride the
// hidden dimension in 16-byte vectors of x (thread i takes vectors i, i+128,
// ...), so each thread sums a d/128 slice for every expert and token. W_g
// rows are read as 16-byte vectors when a row is a whole number of them
// (VW), else element by element. Partial sums: butterfly inside each warp
// (identical bits on every lane), then the 4 warp partials are added in warp
// order, so the result does not depend on scheduling.
template <typename Tin, int NE, int TPB, bool VW>
__global__ void __launch_bounds__(128) route_narrow_kernel(
    const Tin* __restrict__ x, const Tin* __restrict__ Wg, const float* __restrict__ bias, int T,
    int d, int E, int k, int pre_k, int router, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, float* __restrict__ logits) {
  constexpr int VEC = 16 / sizeof(Tin);  // elements per 16-byte load
  __shared__ float part[4][TPB][NE];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TPB;

  float acc[TPB][NE];
#pragma unroll
  for (int q = 0; q < TPB; ++q)
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[q][e] = 0.f;

  const int nvec = d / VEC;
  for (int c = threadIdx.x; c < nvec; c += 128) {
    uint4 raw[TPB];
#pragma unroll
    for (int q = 0; q < TPB; ++q)
      raw[q] = (t0 + q < T) ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t0 + q) * d) + c)
                            : make_uint4(0, 0, 0, 0);
#pragma unroll
    for (int i = 0; i < VEC; ++i) {
      const Tin* wrow = Wg + static_cast<size_t>(c * VEC + i) * E;
      float wv[NE];
      if constexpr (VW) {
        constexpr int PER = 16 / sizeof(Tin);
#pragma unroll
        for (int v = 0; v < NE / PER; ++v) {
          if (v * PER < E) {
            const uint4 u = __ldg(reinterpret_cast<const uint4*>(wrow) + v);
            const Tin* ue = reinterpret_cast<const Tin*>(&u);
#pragma unroll
            for (int j = 0; j < PER; ++j) wv[v * PER + j] = to_f32(ue[j]);
          } else {
#pragma unroll
            for (int j = 0; j < PER; ++j) wv[v * PER + j] = 0.f;
          }
        }
      } else {
#pragma unroll
        for (int e = 0; e < NE; ++e) wv[e] = (e < E) ? to_f32(__ldg(wrow + e)) : 0.f;
      }
#pragma unroll
      for (int q = 0; q < TPB; ++q) {
        const float xi = to_f32(reinterpret_cast<const Tin*>(&raw[q])[i]);
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[q][e] = fmaf(xi, wv[e], acc[q][e]);
      }
    }
  }
#pragma unroll
  for (int q = 0; q < TPB; ++q)
#pragma unroll
    for (int e = 0; e < NE; ++e) {
#pragma unroll
      for (int off = 16; off > 0; off >>= 1)
        acc[q][e] += __shfl_xor_sync(0xffffffffu, acc[q][e], off);
    }
#pragma unroll
  for (int q = 0; q < TPB; ++q)
#pragma unroll
    for (int e = 0; e < NE; ++e)
      if (e == lane) part[w][q][e] = acc[q][e];
  __syncthreads();

  // warp q selects for token t0 + q; lane e owns expert e
  for (int q = w; q < TPB; q += 4) {
    const int t = t0 + q;
    if (t >= T) break;
    float mine = -INFINITY;
    if (lane < E) {
      mine = ((part[0][q][lane] + part[1][q][lane]) + part[2][q][lane]) + part[3][q][lane];
      mine += bias ? __ldg(bias + lane) : 0.f;
      if (logits) logits[static_cast<size_t>(t) * E + lane] = mine;
    }
    float v[1] = {mine};
    int id[1] = {lane < E ? lane : 0x7fffffff};
    warp_select_and_weigh<1>(v, id, k, pre_k, router, t, topk_idx, topk_w);
  }
}

// ---------------------------------------------------------------- wide
// CTA = 256 threads, 32 tokens x (32 * EPT) experts. Thread (ty, tx):
// tokens 4*ty .. 4*ty+3, experts tx + 32*j (j < EPT).
constexpr int kWideTokens = 32;
constexpr int kWideBK = 32;

template <typename Tin, int EPT>
__global__ void __launch_bounds__(256) route_wide_kernel(
    const Tin* __restrict__ x, const Tin* __restrict__ Wg, const float* __restrict__ bias, int T,
    int d, int E, int k, int pre_k, int router, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, float* __restrict__ logits) {
  constexpr int EP = 32 * EPT;  // padded expert count
  __shared__ __align__(16) float xs[kWideBK][kWideTokens];
  __shared__ __align__(16) float ws[kWideBK * EP > kWideTokens * EP ? kWideBK * EP : kWideTokens * EP];

  const int tid = threadIdx.x;
  const int tx = tid & 31;
  const int ty = tid >> 5;
  const int t0 = blockIdx.x * kWideTokens;

  float tot[4][EPT], comp[4][EPT];
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EPT; ++j) tot[i][j] = comp[i][j] = 0.f;

  for (int k0 = 0; k0 < d; k0 += kWideBK) {
    // x tile [32 tokens][32 k] -> xs[k][token]; 4 elements per thread
    {
      const int r = tid >> 3;           // token within tile
      const int c = (tid & 7) * 4;      // k within chunk
      const int t = t0 + r;
#pragma unroll
      for (int i = 0; i < 4; ++i)
        xs[c + i][r] = (t < T) ? to_f32(x[static_cast<size_t>(t) * d + k0 + c + i]) : 0.f;
    }
    // W_g tile [32 k][EP experts]
    for (int idx = tid; idx < kWideBK * EP; idx += 256) {
      const int r = idx / EP, e = idx % EP;
      ws[idx] = (e < E) ? to_f32(Wg[static_cast<size_t>(k0 + r) * E + e]) : 0.f;
    }
    __syncthreads();
    float acc[4][EPT];
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < EPT; ++j) acc[i][j] = 0.f;
#pragma unroll 8
    for (int kk = 0; kk < kWideBK; ++kk) {
      const float4 a = *reinterpret_cast<const float4*>(&xs[kk][ty * 4]);
      float b[EPT];
#pragma unroll
      for (int j = 0; j < EPT; ++j) b[j] = ws[kk * EP + tx + 32 * j];
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        acc[0][j] = fmaf(a.x, b[j], acc[0][j]);
        acc[1][j] = fmaf(a.y, b[j], acc[1][j]);
        acc[2][j] = fmaf(a.z, b[j], acc[2][j]);
        acc[3][j] = fmaf(a.w, b[j], acc[3][j]);
      }
    }
    // compensated fold of the chunk sums into the totals
#pragma unroll
    for (int i = 0; i < 4; ++i)
#pragma unroll
      for (int j = 0; j < EPT; ++j) {
        const float y = acc[i][j] - comp[i][j];
        const float s = tot[i][j] + y;
        comp[i][j] = (s - tot[i][j]) - y;
        tot[i][j] = s;
      }
    __syncthreads();
  }

  // logits tile -> shared (reusing ws as [32 tokens][EP])
  float* Ls = ws;
#pragma unroll
  for (int i = 0; i < 4; ++i)
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tx + 32 * j;
      const int r = ty * 4 + i;
      float val = -INFINITY;
      if (e < E) val = tot[i][j] + (bias ? __ldg(bias + e) : 0.f);
      Ls[r * EP + e] = val;
      if (logits && e < E && t0 + r < T) logits[static_cast<size_t>(t0 + r) * E + e] = val;
    }
  __syncthreads();

  // 8 warps x 4 tokens: select and weigh
#pragma unroll 1
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    const int t = t0 + r;
    if (t >= T) break;
    float v[EPT];
    int id[EPT];
#pragma unroll
    for (int j = 0; j < EPT; ++j) {
      const int e = tx + 32 * j;
      v[j] = Ls[r * EP + e];
      id[j] = (e < E) ? e : 0x7fffffff;
    }
    warp_select_and_weigh<EPT>(v, id, k, pre_k, router, t, topk_idx, topk_w);
  }
}

template <typename Tin>
cudaError_t launch_route_t(const Tin* x, const Tin* Wg, const float* bias, int T, int d, int E,
                           int k, int pre_k, int router, int32_t* topk_idx, float* topk_w,
                           float* logits, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (E <= 32) {
    const bool vw = (reinterpret_cast<uintptr_t>(Wg) % 16 == 0) &&
                    ((E * static_cast<int>(sizeof(Tin))) % 16 == 0);
    const int tpb = (T >= 4096) ? 2 : 1;
    const dim3 block(128);
#define MOE_NARROW(NE, TPB, VW)                                                          \
  route_narrow_kernel<Tin, NE, TPB, VW><<<dim3(ceil_div(T, TPB)), block, 0, s>>>(      \
      x, Wg, bias, T, d, E, k, pre_k, router, topk_idx, topk_w, logits)
#define MOE_NARROW_E(TPB, VW) \
  do {                        \
    if (E <= 8)               \
      MOE_NARROW(8, TPB, VW); \
    else if (E <= 16)         \
      MOE_NARROW(16, TPB, VW);\
    else                      \
      MOE_NARROW(32, TPB, VW);\
  } while (0)
    if (tpb == 1) {
      if (vw) MOE_NARROW_E(1, true); else MOE_NARROW_E(1, false);
    } else {
      if (vw) MOE_NARROW_E(2, true); else MOE_NARROW_E(2, false);
    }
#undef MOE_NARROW_E
#undef MOE_NARROW
  } else {
    const dim3 grid(ceil_div(T, kWideTokens)), block(256);
#define MOE_WIDE(EPT)                                                                        \
  route_wide_kernel<Tin, EPT><<<grid, block, 0, s>>>(x, Wg, bias, T, d, E, k, pre_k, router, \
                                                     topk_idx, topk_w, logits)
    if (E <= 64)
      MOE_WIDE(2);
    else if (E <= 128)
      MOE_WIDE(4);
    else
      MOE_WIDE(8);
#undef MOE_WIDE
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(int dtype, const void* x, const void* Wg, const float* bias, int T,
                         int d, int E, int k, int pre_k, int router, int32_t* topk_idx,
                         float* topk_w, float* logits, cudaStream_t s) {
  if (dtype == 0)
    return launch_route_t<float>(static_cast<const float*>(x), static_cast<const float*>(Wg),
                                 bias, T, d, E, k, pre_k, router, topk_idx, topk_w, logits, s);
  return launch_route_t<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(x),
                                       static_cast<const __nv_bfloat16*>(Wg), bias, T, d, E, k,
                                       pre_k, router, topk_idx, topk_w, logits, s);
}

}  // namespace moe
