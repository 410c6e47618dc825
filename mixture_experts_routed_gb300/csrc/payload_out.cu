// payload_out.cu - FP8 expert-output payload (Deepseek-MoE sync-tax article,
// section 3.1: each expert output vector is quantised on its own, from its
// min and max, by an affine map) and the combine that consumes it.
//
// quantise, per routed row r of the fp32 expert outputs y:
//   zero = mx/2 + mn/2, half = mx/2 - mn/2   (one fp32 rounding each)
//   s = half / 448 (fp32 IEEE division; 1 for a constant row)
//   q = E4M3(fp32(y - zero) / s), round to nearest even, saturating
// so [mn, mx] spans [-448, 448] and the row decodes as q * s + zero.
// combine, per token t: out[t] = sum_{j<k} w[t,j] * (q[p] * s[p] + zero[p]),
// p = pos[t*k + j], j ascending, fp32, no atomics.
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kRowsPerCta = 8;  // one warp per row

// Four values of a row -> four E4M3 bytes of fp32(v - zero) / s (the IEEE
// quotient; FAST: from y = RN(1/s) and two residual corrections, the same
// bits), element 0 in the lowest byte.
template <bool FAST>
__device__ __forceinline__ uint32_t quant4(float4 a, float zero, float s, float y) {
  const float x0 = __fsub_rn(a.x, zero), x1 = __fsub_rn(a.y, zero);
  const float x2 = __fsub_rn(a.z, zero), x3 = __fsub_rn(a.w, zero);
  const float2 lo = FAST ? make_float2(quotient_rn(x0, s, y), quotient_rn(x1, s, y))
                         : make_float2(__fdiv_rn(x0, s), __fdiv_rn(x1, s));
  const float2 hi = FAST ? make_float2(quotient_rn(x2, s, y), quotient_rn(x3, s, y))
                         : make_float2(__fdiv_rn(x2, s), __fdiv_rn(x3, s));
  const uint32_t b0 = __nv_cvt_float2_to_fp8x2(lo, __NV_SATFINITE, __NV_E4M3);
  const uint32_t b1 = __nv_cvt_float2_to_fp8x2(hi, __NV_SATFINITE, __NV_E4M3);
  return b0 | (b1 << 16);
}

// Pass 2 of quantize_out_kernel for one row (one warp); the division form
// (scales outside [2^-64, 2^64] only) keeps one load in flight per lane.
template <bool FAST>
__device__ __forceinline__ void quant_row_out(const float4* __restrict__ row, int nv, int lane,
                                              float zero, float s, uint32_t* __restrict__ out) {
  const float y = FAST ? __frcp_rn(s) : 0.f;
  constexpr int U = FAST ? 4 : 1;
  for (int v0 = lane; v0 < nv; v0 += 32 * U) {
    float4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + 32 * u < nv) a[u] = __ldg(row + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nv) break;
      out[v] = quant4<FAST>(a[u], zero, s, y);
    }
  }
}

// Pass 1 reads the row for its min and max, pass 2 reads it again (from L2:
// the row was read a moment before) and writes 4 E4M3 bytes per float4.
// The quotients come from one reciprocal per row and two residual
// corrections (quotient_rn), bit for bit the IEEE division.
__global__ void __launch_bounds__(256) quantize_out_kernel(const float* __restrict__ y, int R,
                                                           int d, uint8_t* __restrict__ yq,
                                                           float* __restrict__ ys,
                                                           float* __restrict__ yz) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int r = blockIdx.x * kRowsPerCta + (threadIdx.x >> 5);
  if (r >= R) return;
  const int nv = d / 4;
  const float4* row = reinterpret_cast<const float4*>(y + static_cast<size_t>(r) * d);
  constexpr int U = 4;  // float4 loads in flight per lane
  float mn = INFINITY, mx = -INFINITY;
  for (int v0 = lane; v0 < nv; v0 += 32 * U) {
    float4 a[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + 32 * u < nv) a[u] = __ldg(row + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < U; ++u) {
      if (v0 + 32 * u >= nv) break;
      mn = fminf(fminf(mn, a[u].x), fminf(a[u].y, fminf(a[u].z, a[u].w)));
      mx = fmaxf(fmaxf(mx, a[u].x), fmaxf(a[u].y, fmaxf(a[u].z, a[u].w)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  const float hmx = __fmul_rn(mx, 0.5f), hmn = __fmul_rn(mn, 0.5f);
  const float zero = __fadd_rn(hmx, hmn);
  const float half = __fsub_rn(hmx, hmn);
  const float s = (half == 0.f) ? 1.f : __fdiv_rn(half, 448.f);
  uint32_t* out = reinterpret_cast<uint32_t*>(yq + static_cast<size_t>(r) * d);
  if (quotient_scale_ok(s))  // s is uniform across the warp
    quant_row_out<true>(row, nv, lane, zero, s, out);
  else
    quant_row_out<false>(row, nv, lane, zero, s, out);
  if (lane == 0) {
    ys[r] = s;
    yz[r] = zero;
  }
}

// One CTA of 256 threads per row, the row held in registers (NV float4 per
// thread, d <= 1024 NV): one read of y, min/max by warp shuffles and a
// shared-memory pass over the 8 warps, then the same per-value arithmetic
// as quantize_out_kernel.
template <int NV>
__global__ void __launch_bounds__(256) quantize_out_cta_kernel(const float* __restrict__ y, int R,
                                                               int d, uint8_t* __restrict__ yq,
                                                               float* __restrict__ ys,
                                                               float* __restrict__ yz) {
  __shared__ float red[2][8];
  pdl_wait();
  pdl_trigger();
  const int r = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int nv = d / 4;
  const float4* row = reinterpret_cast<const float4*>(y + static_cast<size_t>(r) * d);
  float4 a[NV];
  float mn = INFINITY, mx = -INFINITY;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = tid + 256 * i;
    if (v < nv) {
      a[i] = __ldg(row + v);
      mn = fminf(fminf(mn, a[i].x), fminf(a[i].y, fminf(a[i].z, a[i].w)));
      mx = fmaxf(fmaxf(mx, a[i].x), fmaxf(a[i].y, fmaxf(a[i].z, a[i].w)));
    }
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    mn = fminf(mn, __shfl_xor_sync(0xffffffffu, mn, off));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
  }
  if (lane == 0) {
    red[0][w] = mn;
    red[1][w] = mx;
  }
  __syncthreads();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    mn = fminf(mn, red[0][i]);
    mx = fmaxf(mx, red[1][i]);
  }
  const float hmx = __fmul_rn(mx, 0.5f), hmn = __fmul_rn(mn, 0.5f);
  const float zero = __fadd_rn(hmx, hmn);
  const float half = __fsub_rn(hmx, hmn);
  const float s = (half == 0.f) ? 1.f : __fdiv_rn(half, 448.f);
  uint32_t* out = reinterpret_cast<uint32_t*>(yq + static_cast<size_t>(r) * d);
  const bool fast = quotient_scale_ok(s);  // uniform across the CTA
  const float yr = fast ? __frcp_rn(s) : 0.f;
#pragma unroll
  for (int i = 0; i < NV; ++i) {
    const int v = tid + 256 * i;
    if (v < nv) out[v] = fast ? quant4<true>(a[i], zero, s, yr) : quant4<false>(a[i], zero, s, yr);
  }
  if (tid == 0) {
    ys[r] = s;
    yz[r] = zero;
  }
}

// Two E4M3 bytes (element 0 in the low byte) -> two floats, exactly (every
// E4M3 value is a half value).
__device__ __forceinline__ float2 e4m3x2_to_float2(uint16_t b) {
  const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(b), __NV_E4M3);
  return __half22float2(*reinterpret_cast<const __half2*>(&hr));
}

// 128 threads per token, two tokens per CTA; each thread owns 16-byte
// columns c, c+128, ... (16 values) of the k payload rows and keeps U of
// them in flight.
template <int DT, int KMAX>  // DT 0: fp32 out, 1: bf16 out; k <= KMAX
__global__ void __launch_bounds__(256) combine_fp8_kernel(
    const uint8_t* __restrict__ yq, const float* __restrict__ ys, const float* __restrict__ yz,
    const int32_t* __restrict__ pos, const float* __restrict__ w, int T, int d, int k, int R,
    void* __restrict__ out, uint32_t* __restrict__ err) {
  pdl_wait();
  pdl_trigger();
  const int tl = threadIdx.x & 127;
  const int t = blockIdx.x * 2 + (threadIdx.x >> 7);
  if (t >= T) return;
  const int nv = d / 16;
  const uint4* qv = reinterpret_cast<const uint4*>(yq);
  if constexpr (KMAX <= 4) {
    int p[KMAX];
    float wt[KMAX], sc[KMAX], zr[KMAX];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < KMAX; ++j) {
      p[j] = -1;
      wt[j] = 0.f;
      sc[j] = 0.f;
      zr[j] = 0.f;
      if (j < k) {
        const int q = __ldg(pos + static_cast<size_t>(t) * k + j);
        if (q >= 0 && q < R) {
          p[j] = q;
          wt[j] = __ldg(w + static_cast<size_t>(t) * k + j);
          sc[j] = __ldg(ys + q);
          zr[j] = __ldg(yz + q);
        } else {
          bad = true;
        }
      }
    }
    if (bad && tl == 0) atomicOr(err, kErrBadIndex);

    constexpr int U = 8 / KMAX > 0 ? 8 / KMAX : 1;
    for (int c0 = tl; c0 < nv; c0 += 128 * U) {
      uint4 rows[U][KMAX];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 128;
#pragma unroll
        for (int j = 0; j < KMAX; ++j)
          if (p[j] >= 0 && c < nv) rows[u][j] = __ldg(qv + static_cast<size_t>(p[j]) * nv + c);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int c = c0 + u * 128;
        if (c >= nv) break;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll
        for (int j = 0; j < KMAX; ++j) {
          if (p[j] < 0) continue;
          const uint32_t wd[4] = {rows[u][j].x, rows[u][j].y, rows[u][j].z, rows[u][j].w};
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const float2 f = e4m3x2_to_float2(static_cast<uint16_t>(wd[h >> 1] >> (16 * (h & 1))));
            acc[2 * h] = fmaf(wt[j], fmaf(f.x, sc[j], zr[j]), acc[2 * h]);
            acc[2 * h + 1] = fmaf(wt[j], fmaf(f.y, sc[j], zr[j]), acc[2 * h + 1]);
          }
        }
        if constexpr (DT == 0) {
          float4* o = reinterpret_cast<float4*>(out) + (static_cast<size_t>(t) * nv + c) * 4;
#pragma unroll
          for (int q = 0; q < 4; ++q)
            o[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
        } else {
          uint4 uu[2];
          uint32_t* pu = &uu[0].x;
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * h], acc[2 * h + 1]);
            pu[h] = *reinterpret_cast<const uint32_t*>(&b);
          }
          uint4* o = reinterpret_cast<uint4*>(out) + (static_cast<size_t>(t) * nv + c) * 2;
          o[0] = uu[0];
          o[1] = uu[1];
        }
      }
    }
  } else {
    // k > 4: rows in batches of 4, each batch's position, weight, scale and
    // zero read per column block (all k of each in registers took ~190
    // registers at k = 16); the fp32 sum still runs j = 0..k-1 in order
    bool bad = false;
    for (int j = 0; j < k; ++j) {
      const int q = __ldg(pos + static_cast<size_t>(t) * k + j);
      bad |= !(q >= 0 && q < R);
    }
    if (bad && tl == 0) atomicOr(err, kErrBadIndex);
    constexpr int JB = 4;
    for (int c = tl; c < nv; c += 128) {
      float acc[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) acc[i] = 0.f;
#pragma unroll 1
      for (int jb = 0; jb < k; jb += JB) {
        int pj[JB];
        float wj[JB], sj[JB], zj[JB];
        uint4 rows[JB];
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          const int j = jb + jj;
          pj[jj] = -1;
          wj[jj] = sj[jj] = zj[jj] = 0.f;
          if (j < k) {
            const int q = __ldg(pos + static_cast<size_t>(t) * k + j);
            if (q >= 0 && q < R) {
              pj[jj] = q;
              wj[jj] = __ldg(w + static_cast<size_t>(t) * k + j);
              sj[jj] = __ldg(ys + q);
              zj[jj] = __ldg(yz + q);
            }
          }
        }
#pragma unroll
        for (int jj = 0; jj < JB; ++jj)
          if (pj[jj] >= 0) rows[jj] = __ldg(qv + static_cast<size_t>(pj[jj]) * nv + c);
#pragma unroll
        for (int jj = 0; jj < JB; ++jj) {
          if (pj[jj] < 0) continue;
          const uint32_t wd[4] = {rows[jj].x, rows[jj].y, rows[jj].z, rows[jj].w};
#pragma unroll
          for (int h = 0; h < 8; ++h) {
            const float2 f = e4m3x2_to_float2(static_cast<uint16_t>(wd[h >> 1] >> (16 * (h & 1))));
            acc[2 * h] = fmaf(wj[jj], fmaf(f.x, sj[jj], zj[jj]), acc[2 * h]);
            acc[2 * h + 1] = fmaf(wj[jj], fmaf(f.y, sj[jj], zj[jj]), acc[2 * h + 1]);
          }
        }
      }
      if constexpr (DT == 0) {
        float4* o = reinterpret_cast<float4*>(out) + (static_cast<size_t>(t) * nv + c) * 4;
#pragma unroll
        for (int q = 0; q < 4; ++q)
          o[q] = make_float4(acc[4 * q], acc[4 * q + 1], acc[4 * q + 2], acc[4 * q + 3]);
      } else {
        uint4 uu[2];
        uint32_t* pu = &uu[0].x;
#pragma unroll
        for (int h = 0; h < 8; ++h) {
          const __nv_bfloat162 b = __floats2bfloat162_rn(acc[2 * h], acc[2 * h + 1]);
          pu[h] = *reinterpret_cast<const uint32_t*>(&b);
        }
        uint4* o = reinterpret_cast<uint4*>(out) + (static_cast<size_t>(t) * nv + c) * 2;
        o[0] = uu[0];
        o[1] = uu[1];
      }
    }
  }
}

}  // namespace

cudaError_t launch_quantize_out(const float* y, int R, int d, uint8_t* yq, float* ys, float* yz,
                                cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  // rows of more than 1024 values: a CTA per row, the row in registers (the
  // warp-per-row kernel's second read misses L2 once many rows are in
  // flight); short rows: a warp per row, whose re-read hits L2
  if (d > 1024 && d <= 2048)
    return launch_pdl(quantize_out_cta_kernel<2>, dim3(R), dim3(256), 0, s, y, R, d, yq, ys, yz);
  if (d > 2048 && d <= 4096)
    return launch_pdl(quantize_out_cta_kernel<4>, dim3(R), dim3(256), 0, s, y, R, d, yq, ys, yz);
  if (d > 4096 && d <= 8192)
    return launch_pdl(quantize_out_cta_kernel<8>, dim3(R), dim3(256), 0, s, y, R, d, yq, ys, yz);
  return launch_pdl(quantize_out_kernel, dim3(ceil_div(R, kRowsPerCta)), dim3(256), 0, s, y, R, d,
                    yq, ys, yz);
}

cudaError_t launch_combine_fp8(int dtype, const uint8_t* yq, const float* ys, const float* yz,
                               const int32_t* pos, const float* w, int T, int d, int k, int R,
                               void* out, uint32_t* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  const dim3 grid(ceil_div(T, 2)), block(256);
#define MOE_COMBINE8(DT, KM)                                                                    \
  return launch_pdl(combine_fp8_kernel<DT, KM>, grid, block, 0, s, yq, ys, yz, pos, w, T, d, k, \
                    R, out, err)
  if (dtype == 0) {
    if (k <= 2) MOE_COMBINE8(0, 2);
    if (k <= 4) MOE_COMBINE8(0, 4);
    if (k <= 8) MOE_COMBINE8(0, 8);
    MOE_COMBINE8(0, 16);
  }
  if (k <= 2) MOE_COMBINE8(1, 2);
  if (k <= 4) MOE_COMBINE8(1, 4);
  if (k <= 8) MOE_COMBINE8(1, 8);
  MOE_COMBINE8(1, 16);
#undef MOE_COMBINE8
}

}  // namespace moe
