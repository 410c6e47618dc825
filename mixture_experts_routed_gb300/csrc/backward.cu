// backward.cu - kernels of the layer's backward pass (DeepSeek-V4 EP article,
// section 2.1: in backpropagation the gradient goes back only to the
// activated experts; Deepseek-MoE sync-tax article, section 2.4: the backward
// exchange mirrors the dispatch). Given dout = dl/dout:
//
//   combine_bwd    dY[pos(t,j)] = w[t,j] dout[t],  dw[t,j] = <dout[t], Y[pos(t,j)]>;
//                  bf16 layers also keep, per routed row p, dout[t] itself and
//                  w[t,j] (the dH GEMM takes the weight out of its sum)
//   router_bwd     dL[t] from dw[t] through the router's softmax Jacobian
//   gemm_nt        out[r] = A[r] . W[e]^T (row r of expert e's segment; W[e]
//                  is [N][K] row-major), optionally times SiLU'(Z) in place
//   gemm_tn        out[e] = A_e^T . B_e over the segment's rows (ragged K)
//   bias_bwd       db[e] = sum_t dL[t, e]
//   undispatch     dx[t] = dx_gate[t] + sum_j dX_perm[pos(t,j)]
//
// Every sum runs in a fixed order (no atomics on data): the results are
// bitwise reproducible. The gate's GEMMs, and every GEMM of fp32 layers, are
// SIMT fp32 FMA here (128 x 128 tiles, 8 x 8 per thread); bf16 layers run
// the experts' GEMMs on the tensor cores (gemm_tc.cu, wgrad_tc.cu) with the
// operand split below.
#include <algorithm>
#include <cstdint>
#include <cuda_bf16.h>

#include "common.cuh"

namespace moe {
namespace {

// router modes, as RouterSpec::mode
constexpr int kRouterModePrek = 1;
constexpr int kRouterModeSoft = 3;

__device__ __forceinline__ float ld_f32(const float* p, size_t i) { return __ldg(p + i); }
__device__ __forceinline__ float ld_f32(const __nv_bfloat16* p, size_t i) {
  return __bfloat162float(p[i]);
}
// four consecutive values from a 4-aligned index
__device__ __forceinline__ float4 ld_f32x4(const float* p, size_t i) {
  return __ldg(reinterpret_cast<const float4*>(p + i));
}
__device__ __forceinline__ float4 ld_f32x4(const __nv_bfloat16* p, size_t i) {
  const uint2 u = __ldg(reinterpret_cast<const uint2*>(p + i));
  const float2 a = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.x));
  const float2 b = __bfloat1622float2(*reinterpret_cast<const __nv_bfloat162*>(&u.y));
  return make_float4(a.x, a.y, b.x, b.y);
}
// four consecutive elements copied bit for bit
__device__ __forceinline__ void copy4(float* dst, const float* src) {
  *reinterpret_cast<float4*>(dst) = __ldg(reinterpret_cast<const float4*>(src));
}
__device__ __forceinline__ void copy4(__nv_bfloat16* dst, const __nv_bfloat16* src) {
  *reinterpret_cast<uint2*>(dst) = __ldg(reinterpret_cast<const uint2*>(src));
}
// v = hi + lo, hi = bf16(v), lo = bf16(v - hi), for two values packed
__device__ __forceinline__ void split2(float a, float b, uint32_t* hi, uint32_t* lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  *hi = *reinterpret_cast<const uint32_t*>(&h);
  *lo = *reinterpret_cast<const uint32_t*>(&l);
}

// ---------------------------------------------------------------- combine
// One CTA of 128 threads per token: the k rows of dY (or, bf16 layers, the
// split of dY or of w H), the dout rows, and the k dot products
// (warp butterflies, then the 4 warp partials in warp order).
template <typename Tout>
__global__ void __launch_bounds__(128) combine_bwd_kernel(
    const Tout* __restrict__ dout, const float* __restrict__ y, const int32_t* __restrict__ pos,
    const float* __restrict__ w, int T, int d, int k, int R, float* __restrict__ dY,
    __nv_bfloat16* __restrict__ dYs, const __nv_bfloat16* __restrict__ h, int f,
    __nv_bfloat16* __restrict__ hs, Tout* __restrict__ doutp, float* __restrict__ wr,
    float* __restrict__ dw, uint32_t* __restrict__ err,
    uint32_t* __restrict__ zero, int nzero, int32_t* __restrict__ seg01,
    int32_t* __restrict__ segk, int nsegk, int chunk) {
  __shared__ float red[4][kMaxFanout];
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wp = tid >> 5;
  if (t == 0) {
    if (tid < nzero && zero != nullptr) zero[tid] = 0u;
    if (tid == 0) {
      seg01[0] = 0;
      seg01[1] = T;
    }
    // token chunks of the gate's split weight gradient: [i chunk, (i+1) chunk)
    if (segk != nullptr && tid <= nsegk) segk[tid] = min(tid * chunk, T);
  }
  for (int j = 0; j < k; ++j) {
    const int p = __ldg(pos + static_cast<size_t>(t) * k + j);
    const bool ok = p >= 0 && p < R;
    if (!ok && tid == 0) atomicOr(err, kErrBadIndex);
    const float wt = ok ? __ldg(w + static_cast<size_t>(t) * k + j) : 0.f;
    if (ok && wr != nullptr && tid == 0) wr[p] = wt;
    float part = 0.f;
    if (ok) {
      // four columns per thread (d is a multiple of 64)
      for (int c = tid * 4; c < d; c += 512) {
        const float4 g = ld_f32x4(dout, static_cast<size_t>(t) * d + c);
        if (doutp != nullptr) copy4(doutp + static_cast<size_t>(p) * d + c, dout + static_cast<size_t>(t) * d + c);
        const float4 v = make_float4(wt * g.x, wt * g.y, wt * g.z, wt * g.w);
        if (dY != nullptr) *reinterpret_cast<float4*>(dY + static_cast<size_t>(p) * d + c) = v;
        if (dYs != nullptr) {
          // bf16 split for the tensor-core GEMMs: v = hi + lo to ~2^-17
          uint2 hi, lo;
          split2(v.x, v.y, &hi.x, &lo.x);
          split2(v.z, v.w, &hi.y, &lo.y);
          *reinterpret_cast<uint2*>(dYs + static_cast<size_t>(p) * 2 * d + c) = hi;
          *reinterpret_cast<uint2*>(dYs + static_cast<size_t>(p) * 2 * d + d + c) = lo;
        }
        const float4 yv = ld_f32x4(y, static_cast<size_t>(p) * d + c);
        part = fmaf(g.x, yv.x, part);
        part = fmaf(g.y, yv.y, part);
        part = fmaf(g.z, yv.z, part);
        part = fmaf(g.w, yv.w, part);
      }
    }
    if (ok && hs != nullptr) {
      // H'[p] = w H[p] split for the tensor-core weight gradient dW2 =
      // sum_r H'_r^T dout_r (bf16 parts v = hi + lo to ~2^-17, [R][2f])
      for (int c = tid * 4; c < f; c += 512) {
        const float4 hv = ld_f32x4(h, static_cast<size_t>(p) * f + c);
        uint2 hi, lo;
        split2(wt * hv.x, wt * hv.y, &hi.x, &lo.x);
        split2(wt * hv.z, wt * hv.w, &hi.y, &lo.y);
        *reinterpret_cast<uint2*>(hs + static_cast<size_t>(p) * 2 * f + c) = hi;
        *reinterpret_cast<uint2*>(hs + static_cast<size_t>(p) * 2 * f + f + c) = lo;
      }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) part += __shfl_xor_sync(0xffffffffu, part, off);
    if (lane == 0) red[wp][j] = part;
  }
  __syncthreads();
  if (tid < k) dw[static_cast<size_t>(t) * k + tid] = ((red[0][tid] + red[1][tid]) + red[2][tid]) +
                                                       red[3][tid];
}

// ---------------------------------------------------------------- router
// One warp per token; lane l owns experts l, l + 32, ... (up to 8 of them).
constexpr int kRB_NJ = kMaxExperts / 32;

__device__ __forceinline__ bool beats_b(float va, int ia, float vb, int ib) {
  return va > vb || (va == vb && ia < ib);
}

__global__ void __launch_bounds__(256) router_bwd_kernel(
    const float* __restrict__ L, const int32_t* __restrict__ idx, const float* __restrict__ w,
    const float* __restrict__ dw, int T, int E, int k, int mode, int pre_k, float tau,
    float* __restrict__ dL, __nv_bfloat16* __restrict__ dLs) {
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31;
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const float* Lt = L + static_cast<size_t>(t) * E;
  float g[kRB_NJ];
#pragma unroll
  for (int jj = 0; jj < kRB_NJ; ++jj) g[jj] = 0.f;
  if (mode == kRouterModePrek) {
    // the pre_k largest logits (logit desc, id asc), as the forward chose them
    float v[kRB_NJ];
    bool taken[kRB_NJ];
#pragma unroll
    for (int jj = 0; jj < kRB_NJ; ++jj) {
      const int e = lane + 32 * jj;
      v[jj] = e < E ? Lt[e] : -INFINITY;
      taken[jj] = e >= E;
    }
    const int pk = min(pre_k, E);
    float pv[kMaxTopK];
    int pi[kMaxTopK];
    for (int r = 0; r < pk; ++r) {
      float bv = -INFINITY;
      int bi = 0x7fffffff;
#pragma unroll
      for (int jj = 0; jj < kRB_NJ; ++jj)
        if (!taken[jj] && beats_b(v[jj], lane + 32 * jj, bv, bi)) {
          bv = v[jj];
          bi = lane + 32 * jj;
        }
#pragma unroll
      for (int off = 16; off > 0; off >>= 1) {
        const float ov = __shfl_xor_sync(0xffffffffu, bv, off);
        const int oi = __shfl_xor_sync(0xffffffffu, bi, off);
        if (beats_b(ov, oi, bv, bi)) {
          bv = ov;
          bi = oi;
        }
      }
#pragma unroll
      for (int jj = 0; jj < kRB_NJ; ++jj)
        if (lane + 32 * jj == bi) taken[jj] = true;
      pv[r] = bv;
      pi[r] = bi;
    }
    // q = softmax over the pre_k; w_j = q_j for the first k
    const float m = pv[0];
    float q[kMaxTopK], den = 0.f;
    for (int r = 0; r < pk; ++r) {
      q[r] = expf(pv[r] - m);
      den += q[r];
    }
    float s = 0.f;
    for (int r = 0; r < pk; ++r) {
      q[r] = q[r] / den;
      if (r < k) s = fmaf(__ldg(dw + static_cast<size_t>(t) * k + r), q[r], s);
    }
    for (int r = 0; r < pk; ++r) {
      const float gr = r < k ? __ldg(dw + static_cast<size_t>(t) * k + r) : 0.f;
      const float val = q[r] * (gr - s);
#pragma unroll
      for (int jj = 0; jj < kRB_NJ; ++jj)
        if (lane + 32 * jj == pi[r]) g[jj] = val;
    }
  } else {
    // renormalised / group-limited: softmax over the chosen set; soft
    // gating: over all experts (slot j = expert j), divided by tau
    float s = 0.f;
    for (int j = 0; j < k; ++j)
      s = fmaf(__ldg(w + static_cast<size_t>(t) * k + j), __ldg(dw + static_cast<size_t>(t) * k + j),
               s);
    const float inv_tau = mode == kRouterModeSoft ? 1.f / tau : 1.f;
    for (int j = 0; j < k; ++j) {
      const int e = __ldg(idx + static_cast<size_t>(t) * k + j);
      const float val = __ldg(w + static_cast<size_t>(t) * k + j) *
                        (__ldg(dw + static_cast<size_t>(t) * k + j) - s) * inv_tau;
#pragma unroll
      for (int jj = 0; jj < kRB_NJ; ++jj)
        if (lane + 32 * jj == e) g[jj] = val;
    }
  }
#pragma unroll
  for (int jj = 0; jj < kRB_NJ; ++jj) {
    const int e = lane + 32 * jj;
    if (e < E) {
      dL[static_cast<size_t>(t) * E + e] = g[jj];
      if (dLs != nullptr) {
        // [T][2E] = [hi | lo] for the tensor-core gate GEMMs
        const __nv_bfloat16 hi = __float2bfloat16_rn(g[jj]);
        dLs[static_cast<size_t>(t) * 2 * E + e] = hi;
        dLs[static_cast<size_t>(t) * 2 * E + E + e] =
            __float2bfloat16_rn(g[jj] - __bfloat162float(hi));
      }
    }
  }
}

// ---------------------------------------------------------------- GEMMs
// 128 x 128 CTA tiles, 256 threads with 8 x 8 outputs each: thread (ty, tx)
// owns rows {4 ty .. 4 ty + 3, 64 + 4 ty .. 64 + 4 ty + 3} and the same
// columns from tx, so its shared-memory reads are float4s at distinct banks.
// K steps of 8, the next step's tiles loaded into registers while the
// current one is multiplied (two shared-memory buffers). 64 x 64 tiles with
// 4 x 4 per thread reached ~0.28 of the fp32 FMA peak (GB300).
constexpr int BM = 128, BN = 128, BK = 8;

// m-tile index -> (expert, rows) over the segments; returns -1 for no tile,
// -2 for bad offsets
__device__ __forceinline__ int find_tile(const int32_t* offsets, int E, int R, int mt, int* r0,
                                         int* r1, int* lo_out) {
  if (offsets[0] != 0) return -2;
  for (int e = 0; e < E; ++e) {
    const int lo = offsets[e], hi = offsets[e + 1];
    if (hi < lo || hi > R) return -2;
    const int tiles = (hi - lo + BM - 1) / BM;
    if (mt < tiles) {
      *r0 = lo + mt * BM;
      *r1 = min(*r0 + BM, hi);
      *lo_out = lo;
      return e;
    }
    mt -= tiles;
  }
  return -1;
}

// acc += As[buf] (BK x 128) ^T . Bs[buf] (BK x 128) for this thread's 8 x 8
__device__ __forceinline__ void mma_tile(const float (*As)[BM + 4], const float (*Bs)[BN + 4],
                                         int tx, int ty, float (&acc)[8][8]) {
#pragma unroll
  for (int kk = 0; kk < BK; ++kk) {
    const float4 a0 = *reinterpret_cast<const float4*>(&As[kk][ty * 4]);
    const float4 a1 = *reinterpret_cast<const float4*>(&As[kk][64 + ty * 4]);
    const float4 b0 = *reinterpret_cast<const float4*>(&Bs[kk][tx * 4]);
    const float4 b1 = *reinterpret_cast<const float4*>(&Bs[kk][64 + tx * 4]);
    const float a[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
    const float b[8] = {b0.x, b0.y, b0.z, b0.w, b1.x, b1.y, b1.z, b1.w};
#pragma unroll
    for (int i = 0; i < 8; ++i)
#pragma unroll
      for (int j = 0; j < 8; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
  }
}

// the tile row / column of this thread's output i (0..7)
__device__ __forceinline__ int sub_idx(int t, int i) { return (i < 4 ? 0 : 64) + t * 4 + (i & 3); }

// out[r, n] = sum_k A[r, k] W[e][n][k] for the rows r of expert e's segment;
// A fp32 [R, K]; W [E][N][K] (TW). SILU: out holds Z on entry and gets
// acc * SiLU'(Z) (each element read and written by the same thread).
// Loads: thread q takes row q / 2 of the A and W tiles, k half (q & 1) * 4.
template <typename TW, bool SILU>
__global__ void __launch_bounds__(256) gemm_nt_kernel(const float* __restrict__ A,
                                                      const TW* __restrict__ W, int E, int R,
                                                      int K, int N,
                                                      const int32_t* __restrict__ offsets,
                                                      float* __restrict__ out,
                                                      uint32_t* __restrict__ err) {
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Ws[2][BK][BN + 4];
  __shared__ int s_e, s_r0, s_r1;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  if (tid == 0) {
    int r0 = 0, r1 = 0, lo = 0;
    const int e = find_tile(offsets, E, R, blockIdx.x, &r0, &r1, &lo);
    if (e == -2 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(err, kErrBadIndex);
    s_e = e;
    s_r0 = r0;
    s_r1 = r1;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int row0 = s_r0, nrows = s_r1 - s_r0, n0 = blockIdx.y * BN;
  const float* Ae = A + static_cast<size_t>(row0) * K;
  const TW* We = W + static_cast<size_t>(e) * N * K;
  const int tx = tid & 15, ty = tid >> 4;
  const int lr = tid >> 1, lk = (tid & 1) * 4;
  float ra[4], rw[4];
  auto load = [&](int k0) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      const int kk = k0 + lk + u;
      ra[u] = (lr < nrows && kk < K) ? __ldg(Ae + static_cast<size_t>(lr) * K + kk) : 0.f;
      rw[u] = (n0 + lr < N && kk < K) ? ld_f32(We, static_cast<size_t>(n0 + lr) * K + kk) : 0.f;
    }
  };
  auto store = [&](int buf) {
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      As[buf][lk + u][lr] = ra[u];
      Ws[buf][lk + u][lr] = rw[u];
    }
  };
  float acc[8][8] = {};
  load(0);
  store(0);
  __syncthreads();
  int buf = 0;
  for (int k0 = 0; k0 < K; k0 += BK) {
    const bool more = k0 + BK < K;
    if (more) load(k0 + BK);
    mma_tile(As[buf], Ws[buf], tx, ty, acc);
    if (more) store(buf ^ 1);
    __syncthreads();
    buf ^= 1;
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = sub_idx(ty, i);
    if (r >= nrows) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + sub_idx(tx, j);
      if (n >= N) continue;
      float* o = out + static_cast<size_t>(row0 + r) * N + n;
      float v = acc[i][j];
      if (SILU) {
        const float z = *o;
        const float sg = 1.f / (1.f + expf(-z));
        v *= sg * (1.f + z * (1.f - sg));
      }
      *o = v;
    }
  }
}

// out[e][m][n] = sum over the rows r of expert e's segment of A[a(r)][m] B[r][n]
// (a(r) = r, or r - offsets[e] when A is shared by every expert); A [*, M]
// (TA), B fp32 [R, N]; out [E][M][N] fp32. An expert with no rows gets zeros.
// Loads: thread q takes k row q / 32 of the tiles, columns (q & 31) * 4 ..+3.
template <typename TA>
__global__ void __launch_bounds__(256) gemm_tn_kernel(const TA* __restrict__ A, int a_shared,
                                                      const float* __restrict__ B, int R, int M,
                                                      int N, const int32_t* __restrict__ offsets,
                                                      float* __restrict__ out,
                                                      uint32_t* __restrict__ err) {
  __shared__ __align__(16) float As[2][BK][BM + 4];
  __shared__ __align__(16) float Bs[2][BK][BN + 4];
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, e = blockIdx.z;
  const int m0 = blockIdx.x * BM, n0 = blockIdx.y * BN;
  int lo = __ldg(offsets + e), hi = __ldg(offsets + e + 1);
  if (lo < 0 || hi < lo || hi > R) {
    if (tid == 0 && blockIdx.x == 0 && blockIdx.y == 0) atomicOr(err, kErrBadIndex);
    lo = hi = 0;
  }
  const int abase = a_shared ? lo : 0;
  const int tx = tid & 15, ty = tid >> 4;
  const int lkr = tid >> 5, lc = (tid & 31) * 4;
  float ra[4], rb[4];
  auto load = [&](int r0) {
    const int r = r0 + lkr;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      ra[u] = (r < hi && m0 + lc + u < M) ? ld_f32(A, static_cast<size_t>(r - abase) * M + m0 + lc + u)
                                          : 0.f;
      rb[u] = (r < hi && n0 + lc + u < N) ? __ldg(B + static_cast<size_t>(r) * N + n0 + lc + u)
                                          : 0.f;
    }
  };
  auto store = [&](int buf) {
    *reinterpret_cast<float4*>(&As[buf][lkr][lc]) = make_float4(ra[0], ra[1], ra[2], ra[3]);
    *reinterpret_cast<float4*>(&Bs[buf][lkr][lc]) = make_float4(rb[0], rb[1], rb[2], rb[3]);
  };
  float acc[8][8] = {};
  if (lo < hi) {
    load(lo);
    store(0);
    __syncthreads();
    int buf = 0;
    for (int r0 = lo; r0 < hi; r0 += BK) {
      const bool more = r0 + BK < hi;
      if (more) load(r0 + BK);
      mma_tile(As[buf], Bs[buf], tx, ty, acc);
      if (more) store(buf ^ 1);
      __syncthreads();
      buf ^= 1;
    }
  }
  float* oe = out + static_cast<size_t>(e) * M * N;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int m = m0 + sub_idx(ty, i);
    if (m >= M) continue;
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int n = n0 + sub_idx(tx, j);
      if (n < N) oe[static_cast<size_t>(m) * N + n] = acc[i][j];
    }
  }
}

// ---------------------------------------------------------------- tensor-core GEMM operands
// bf16 layers run the experts' backward GEMMs on the tensor cores in bf16
// with every fp32 operand split in two: v = hi + lo with hi = bf16(v), lo =
// bf16(v - hi) (a 16-bit significand, error ~2^-17 |v|); the GEMMs take both
// parts against the same bf16 weight or activation, so the products are
// exact and the sums fp32.

// ---------------------------------------------------------------- bias, dx
// Partial sums of db[e] = sum_t dL[t, e] over token chunk c = blockIdx.y
// ([c chunk, (c+1) chunk)). A CTA of 32 warps takes 32 experts (lane =
// expert, so each warp reads 128 contiguous bytes of a row of dL); warp w
// sums the chunk's tokens t = w mod 32 in ascending order, then warp 0 adds
// the 32 partials in warp order: a fixed order, bitwise reproducible.
__global__ void __launch_bounds__(1024) bias_bwd_kernel(const float* __restrict__ dL, int T, int E,
                                                        int chunk, float* __restrict__ part) {
  __shared__ float red[32][33];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int e = blockIdx.x * 32 + lane;
  const int t0 = blockIdx.y * chunk, t1 = min(t0 + chunk, T);
  float s = 0.f;
  if (e < E)
    for (int t = t0 + w; t < t1; t += 32) s += __ldg(dL + static_cast<size_t>(t) * E + e);
  red[w][lane] = s;
  __syncthreads();
  if (w == 0 && e < E) {
    float tot = 0.f;
    for (int i = 0; i < 32; ++i) tot += red[i][lane];
    part[static_cast<size_t>(blockIdx.y) * E + e] = tot;
  }
}

// out[i] = sum over s < S of part[s][i], s ascending; two independent jobs
// (blockIdx.y), each skipped when its S is 0.
struct ReduceJob {
  const float* part;
  int S;
  size_t n;
  float* out;
};
__global__ void __launch_bounds__(256) reduce_partials_kernel(ReduceJob a, ReduceJob b) {
  pdl_wait();
  pdl_trigger();
  const ReduceJob j = blockIdx.y == 0 ? a : b;
  if (j.S == 0) return;
  for (size_t i = blockIdx.x * static_cast<size_t>(blockDim.x) + threadIdx.x; i < j.n;
       i += static_cast<size_t>(gridDim.x) * blockDim.x) {
    float v = 0.f;
    for (int s = 0; s < j.S; ++s) v += __ldg(j.part + static_cast<size_t>(s) * j.n + i);
    j.out[i] = v;
  }
}

// dx[t] = dx_gate[t] + sum_j dX_perm[pos(t, j)], j ascending; 128 threads per token.
__global__ void __launch_bounds__(128) undispatch_kernel(const float* __restrict__ dxg,
                                                         const float* __restrict__ dxp,
                                                         const int32_t* __restrict__ pos, int T,
                                                         int d, int k, int R,
                                                         float* __restrict__ dx) {
  pdl_wait();
  pdl_trigger();
  const int t = blockIdx.x;
  // four columns per thread (d is a multiple of 64): 16-byte loads and stores
  for (int c = threadIdx.x * 4; c < d; c += 512) {
    float4 v = __ldg(reinterpret_cast<const float4*>(dxg + static_cast<size_t>(t) * d + c));
    for (int j = 0; j < k; ++j) {
      const int p = __ldg(pos + static_cast<size_t>(t) * k + j);
      if (p >= 0 && p < R) {
        const float4 a = __ldg(reinterpret_cast<const float4*>(dxp + static_cast<size_t>(p) * d + c));
        v.x += a.x;
        v.y += a.y;
        v.z += a.z;
        v.w += a.w;
      }
    }
    *reinterpret_cast<float4*>(dx + static_cast<size_t>(t) * d + c) = v;
  }
}

}  // namespace

cudaError_t launch_combine_bwd(int dtype, const void* dout, const float* y, const int32_t* pos,
                               const float* w, int T, int d, int k, int R, float* dY, void* dYs,
                               const void* h, int f, void* hs, void* doutp, float* wr, float* dw,
                               uint32_t* err, uint32_t* zero, int nzero, int32_t* seg01,
                               int32_t* segk, int nsegk, int chunk, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  if (hs != nullptr && (dtype != 1 || h == nullptr || f % 4 != 0)) return cudaErrorInvalidValue;
  __nv_bfloat16* ys = static_cast<__nv_bfloat16*>(dYs);
  const __nv_bfloat16* hb = static_cast<const __nv_bfloat16*>(h);
  __nv_bfloat16* hsb = static_cast<__nv_bfloat16*>(hs);
  if (dtype == 0)
    return launch_pdl(combine_bwd_kernel<float>, dim3(T), dim3(128), 0, s,
                      static_cast<const float*>(dout), y, pos, w, T, d, k, R, dY, ys, hb, f, hsb,
                      static_cast<float*>(doutp), wr, dw, err, zero, nzero, seg01, segk, nsegk,
                      chunk);
  return launch_pdl(combine_bwd_kernel<__nv_bfloat16>, dim3(T), dim3(128), 0, s,
                    static_cast<const __nv_bfloat16*>(dout), y, pos, w, T, d, k, R, dY, ys, hb,
                    f, hsb, static_cast<__nv_bfloat16*>(doutp), wr, dw, err, zero, nzero, seg01,
                    segk, nsegk, chunk);
}

cudaError_t launch_router_bwd(const float* L, const int32_t* idx, const float* w, const float* dw,
                              int T, int E, int k, int mode, int pre_k, float tau, float* dL,
                              void* dLs, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(router_bwd_kernel, dim3(ceil_div(T, 8)), dim3(256), 0, s, L, idx, w, dw, T, E,
                    k, mode, pre_k, tau, dL, static_cast<__nv_bfloat16*>(dLs));
}

cudaError_t launch_gemm_nt(int wdtype, bool silu, const float* A, const void* W, int E, int R,
                           int K, int N, const int32_t* offsets, float* out, uint32_t* err,
                           cudaStream_t s) {
  if (R == 0) return cudaSuccess;
  const dim3 grid(ceil_div(R, BM) + E, ceil_div(N, BN)), block(256);
  if (wdtype == 0)
    return silu ? launch_pdl(gemm_nt_kernel<float, true>, grid, block, 0, s, A,
                             static_cast<const float*>(W), E, R, K, N, offsets, out, err)
                : launch_pdl(gemm_nt_kernel<float, false>, grid, block, 0, s, A,
                             static_cast<const float*>(W), E, R, K, N, offsets, out, err);
  return silu ? launch_pdl(gemm_nt_kernel<__nv_bfloat16, true>, grid, block, 0, s, A,
                           static_cast<const __nv_bfloat16*>(W), E, R, K, N, offsets, out, err)
              : launch_pdl(gemm_nt_kernel<__nv_bfloat16, false>, grid, block, 0, s, A,
                           static_cast<const __nv_bfloat16*>(W), E, R, K, N, offsets, out, err);
}

cudaError_t launch_gemm_tn(int adtype, const void* A, int a_shared, const float* B, int E, int R,
                           int M, int N, const int32_t* offsets, float* out, uint32_t* err,
                           cudaStream_t s) {
  if (E == 0) return cudaSuccess;
  const dim3 grid(ceil_div(M, BM), ceil_div(N, BN), E), block(256);
  if (adtype == 0)
    return launch_pdl(gemm_tn_kernel<float>, grid, block, 0, s, static_cast<const float*>(A),
                      a_shared, B, R, M, N, offsets, out, err);
  return launch_pdl(gemm_tn_kernel<__nv_bfloat16>, grid, block, 0, s,
                    static_cast<const __nv_bfloat16*>(A), a_shared, B, R, M, N, offsets, out, err);
}

cudaError_t launch_bias_bwd(const float* dL, int T, int E, int chunk, int nchunk, float* part,
                            cudaStream_t s) {
  if (T == 0 || E == 0) return cudaSuccess;
  return launch_pdl(bias_bwd_kernel, dim3(ceil_div(E, 32), nchunk), dim3(1024), 0, s, dL, T, E,
                    chunk, part);
}

cudaError_t launch_reduce_partials(const float* pa, int Sa, size_t na, float* oa, const float* pb,
                                   int Sb, size_t nb, float* ob, cudaStream_t s) {
  if (Sa == 0 && Sb == 0) return cudaSuccess;
  const size_t n = na > nb ? na : nb;
  const int blocks = static_cast<int>(std::min<size_t>((n + 255) / 256, 152 * 8));
  return launch_pdl(reduce_partials_kernel, dim3(blocks > 0 ? blocks : 1, 2), dim3(256), 0, s,
                    ReduceJob{pa, Sa, na, oa}, ReduceJob{pb, Sb, nb, ob});
}

cudaError_t launch_undispatch(const float* dxg, const float* dxp, const int32_t* pos, int T, int d,
                              int k, int R, float* dx, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  return launch_pdl(undispatch_kernel, dim3(T), dim3(128), 0, s, dxg, dxp, pos, T, d, k, R, dx);
}

}  // namespace moe
