// combine.cu - weighted sum of each token's k expert outputs back in token
// order (Deepseek-MoE sync-tax article, section 2.3):
//   out[t] = sum_{j=0..k-1} w[t, j] * Y[pos[t*k + j]]
// 128 threads per token; each owns 4-float columns, issues the k row loads
// together and accumulates in fp32 in increasing j with no atomics, so the
// result is bitwise reproducible. A pos outside [0, R) adds nothing and flags
// kErrBadIndex.
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

// 128 threads per token, two tokens per CTA; each thread owns float4
// columns c, c+128, ... and keeps U = 8/KMAX of them (8 row loads) in flight.
template <int DT, int KMAX>  // DT 0: fp32 out, 1: bf16 out; k <= KMAX
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ pos,
                                                      const float* __restrict__ w, int T, int d,
                                                      int k, int R, void* __restrict__ out,
                                                      uint32_t* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int tl = threadIdx.x & 127;
  const int t = blockIdx.x * 2 + (threadIdx.x >> 7);
  if (t >= T) return;
  int p[KMAX];
  float wt[KMAX];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < KMAX; ++j) {
    p[j] = -1;
    wt[j] = 0.f;
    if (j < k) {
      const int q = __ldg(pos + static_cast<size_t>(t) * k + j);
      if (q >= 0 && q < R) {
        p[j] = q;
        wt[j] = __ldg(w + static_cast<size_t>(t) * k + j);
      } else {
        bad = true;
      }
    }
  }
  if (bad && tl == 0) atomicOr(err, kErrBadIndex);

  const int nv = d / 4;
  const float4* yv = reinterpret_cast<const float4*>(y);
  if constexpr (KMAX <= 8) {
    // 8 / KMAX float4 columns of each of the k rows in flight per thread:
    // more CTAs per SM (fewer registers) beat deeper per-thread batches
    // (measured)
    constexpr int U = 8 / KMAX > 0 ? 8 / KMAX : 1;
    for (int c0 = tl; c0 < nv; c0 += 128 * U) {
      float4 rows[U][KMAX];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 128;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (p[j] >= 0 && c < nv) rows[u][j] = __ldg(yv + static_cast<size_t>(p[j]) * nv + c);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 128;
        if (c >= nv) break;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (p[j] >= 0) {
            acc.x = fmaf(wt[j], rows[u][j].x, acc.x);
            acc.y = fmaf(wt[j], rows[u][j].y, acc.y);
            acc.z = fmaf(wt[j], rows[u][j].z, acc.z);
            acc.w = fmaf(wt[j], rows[u][j].w, acc.w);
          }
        }
        if constexpr (DT == 0) {
          reinterpret_cast<float4*>(out)[static_cast<size_t>(t) * nv + c] = acc;
        } else {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
          uint2 uu;
          uu.x = *reinterpret_cast<const uint32_t*>(&lo);
          uu.y = *reinterpret_cast<const uint32_t*>(&hi);
          reinterpret_cast<uint2*>(out)[static_cast<size_t>(t) * nv + c] = uu;
        }
      }
    }
  } else {
    // k > 8: the rows in batches of 8 (the fp32 sum still runs j = 0, 1, ...,
    // k-1 in order); all 16 at once took 176 registers, one CTA per SM
    constexpr int U = 8 / KMAX > 0 ? 8 / KMAX : 1;
    constexpr int JB = KMAX < 8 ? KMAX : 8;
    for (int c0 = tl; c0 < nv; c0 += 128 * U) {
      float4 acc[U];
#pragma unroll
      for (int u = 0; u < U; ++u) acc[u] = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll(KMAX > 8 ? 1 : 2)
      for (int jb = 0; jb < KMAX; jb += JB) {
        float4 rows[U][JB];
#pragma unroll
        for (int u = 0; u < U; ++u) {
          const int c = c0 + u * 128;
#pragma unroll
          for (int jj = 0; jj < JB; ++jj) {
            const int j = jb + jj;
            int pj = -1;
#pragma unroll
            for (int q = 0; q < KMAX; ++q) pj = (q == j) ? p[q] : pj;
            if (pj >= 0 && c < nv) rows[u][jj] = __ldg(yv + static_cast<size_t>(pj) * nv + c);
          }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
#pragma unroll
          for (int jj = 0; jj < JB; ++jj) {
            const int j = jb + jj;
            int pj = -1;
            float wj = 0.f;
#pragma unroll
            for (int q = 0; q < KMAX; ++q) {
              pj = (q == j) ? p[q] : pj;
              wj = (q == j) ? wt[q] : wj;
            }
            if (pj >= 0) {
              acc[u].x = fmaf(wj, rows[u][jj].x, acc[u].x);
              acc[u].y = fmaf(wj, rows[u][jj].y, acc[u].y);
              acc[u].z = fmaf(wj, rows[u][jj].z, acc[u].z);
              acc[u].w = fmaf(wj, rows[u][jj].w, acc[u].w);
            }
          }
        }
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 128;
        if (c >= nv) break;
        if constexpr (DT == 0) {
          reinterpret_cast<float4*>(out)[static_cast<size_t>(t) * nv + c] = acc[u];
        } else {
          const __nv_bfloat162 lo = __floats2bfloat162_rn(acc[u].x, acc[u].y);
          const __nv_bfloat162 hi = __floats2bfloat162_rn(acc[u].z, acc[u].w);
          uint2 uu;
          uu.x = *reinterpret_cast<const uint32_t*>(&lo);
          uu.y = *reinterpret_cast<const uint32_t*>(&hi);
          reinterpret_cast<uint2*>(out)[static_cast<size_t>(t) * nv + c] = uu;
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_combine(int dtype, const float* y, const int32_t* pos, const float* w, int T,
                           int d, int k, int R, void* out, uint32_t* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(ceil_div(T, 2)), block(256);
#define MOE_COMBINE(DT, KM) \
  return launch_pdl(combine_kernel<DT, KM>, grid, block, 0, s, y, pos, w, T, d, k, R, out, err)
  if (dtype == 0) {
    if (k <= 2) MOE_COMBINE(0, 2);
    if (k <= 4) MOE_COMBINE(0, 4);
    if (k <= 8) MOE_COMBINE(0, 8);
    MOE_COMBINE(0, 16);
  }
  if (k <= 2) MOE_COMBINE(1, 2);
  if (k <= 4) MOE_COMBINE(1, 4);
  if (k <= 8) MOE_COMBINE(1, 8);
  MOE_COMBINE(1, 16);
#undef MOE_COMBINE
}

}  // namespace moe
