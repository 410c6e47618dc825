// combine.cu - weighted sum of each token's k expert outputs back in token
// order (Deepseek-MoE sync-tax article, section 2.3):
//   out[t] = sum_{j=0..k-1} w[t, j] * Y[pos[t*k + j]]
// One warp per token; each lane owns 4-float columns, issues the k row loads
// together and accumulates in fp32 in increasing j with no atomics, so the
// result is bitwise reproducible. A pos outside [0, R) adds nothing and flags
// kErrBadIndex.
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

template <int DT>  // 0: fp32 out, 1: bf16 out
__global__ void __launch_bounds__(256) combine_kernel(const float* __restrict__ y,
                                                      const int32_t* __restrict__ pos,
                                                      const float* __restrict__ w, int T, int d,
                                                      int k, int R, void* __restrict__ out,
                                                      uint32_t* __restrict__ err) {
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * (blockDim.x / 32) + (threadIdx.x >> 5);
  if (t >= T) return;
  int p[kMaxTopK];
  float wt[kMaxTopK];
  bool bad = false;
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
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
  if (bad && lane == 0) atomicOr(err, kErrBadIndex);

  const int nv = d / 4;
  const float4* yv = reinterpret_cast<const float4*>(y);
  for (int c = lane; c < nv; c += 32) {
    float4 rows[kMaxTopK];
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j)
      if (p[j] >= 0) rows[j] = __ldg(yv + static_cast<size_t>(p[j]) * nv + c);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (p[j] >= 0) {
        acc.x = fmaf(wt[j], rows[j].x, acc.x);
        acc.y = fmaf(wt[j], rows[j].y, acc.y);
        acc.z = fmaf(wt[j], rows[j].z, acc.z);
        acc.w = fmaf(wt[j], rows[j].w, acc.w);
      }
    }
    if constexpr (DT == 0) {
      reinterpret_cast<float4*>(out)[static_cast<size_t>(t) * nv + c] = acc;
    } else {
      const __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(acc.z, acc.w);
      uint2 u;
      u.x = *reinterpret_cast<const uint32_t*>(&lo);
      u.y = *reinterpret_cast<const uint32_t*>(&hi);
      reinterpret_cast<uint2*>(out)[static_cast<size_t>(t) * nv + c] = u;
    }
  }
}

}  // namespace

cudaError_t launch_combine(int dtype, const float* y, const int32_t* pos, const float* w, int T,
                           int d, int k, int R, void* out, uint32_t* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(ceil_div(T, 8)), block(256);
  if (dtype == 0)
    combine_kernel<0><<<grid, block, 0, s>>>(y, pos, w, T, d, k, R, out, err);
  else
    combine_kernel<1><<<grid, block, 0, s>>>(y, pos, w, T, d, k, R, out, err);
  return cudaGetLastError();
}

}  // namespace moe
