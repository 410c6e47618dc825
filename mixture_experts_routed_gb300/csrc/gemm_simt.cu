// gemm_simt.cu - grouped expert GEMM in fp32 FMA, for fp32 layers (the
// tensor cores have no full-fp32 input path; tf32 would miss a 1e-5 bound).
// Same contract as the tensor-core kernel: for every expert e, rows
// [offsets[e], offsets[e+1]) of A (or, shared, rows 0.. of A for every
// expert) times W[e] (K x N, row-major), with
//   epi 0: out = SiLU(acc) (and zout = acc when zout is non-null)
//   epi 1: out = acc
// CTA tile 64 x 64, K step 16, 256 threads with 4 x 4 outputs each. The grid
// covers an upper bound of the m-tiles; each CTA finds its (expert, m-tile)
// from the offsets and exits if it has none.
#include <cstdint>

#include "common.cuh"

namespace moe {
namespace {

constexpr int BM = 64, BN = 64, BK = 16;

template <int EPI>
__global__ void __launch_bounds__(256) gemm_simt_kernel(const float* __restrict__ A, int a_shared,
                                                        int R,
                                                        const float* __restrict__ W, int E,
                                                        int K, int N,
                                                        const int32_t* __restrict__ offsets,
                                                        float* __restrict__ out,
                                                        uint32_t* __restrict__ err,
                                                        float* __restrict__ zout) {
  __shared__ float As[BK][BM + 4];
  __shared__ float Bs[BK][BN];
  __shared__ int s_e, s_row0, s_row1, s_lo;
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x;
  if (tid == 0) {
    // m-tile index -> (expert, rows)
    int mt = blockIdx.x, e_found = -1, r0 = 0, r1 = 0, seg_lo = 0;
    bool ok = offsets[0] == 0;
    for (int e = 0; e < E && ok; ++e) {
      const int lo = offsets[e], hi = offsets[e + 1];
      if (hi < lo || hi > R) { ok = false; break; }
      const int tiles = (hi - lo + BM - 1) / BM;
      if (e_found < 0 && mt < tiles) {
        e_found = e;
        seg_lo = lo;
        r0 = lo + mt * BM;
        r1 = min(r0 + BM, hi);
      }
      mt -= tiles;
    }
    if (!ok) {
      if (blockIdx.x == 0 && blockIdx.y == 0) atomicOr(err, kErrBadIndex);
      e_found = -1;
    }
    s_e = e_found;
    s_row0 = r0;
    s_row1 = r1;
    s_lo = seg_lo;
  }
  __syncthreads();
  const int e = s_e;
  if (e < 0) return;
  const int row0 = s_row0, nrows = s_row1 - s_row0;
  const int n0 = blockIdx.y * BN;
  // shared A: every expert reads rows 0.. of A (row r of the segment -> r - lo)
  const float* Ae = A + static_cast<size_t>(row0 - (a_shared ? s_lo : 0)) * K;
  const float* We = W + static_cast<size_t>(e) * K * N;

  const int tx = tid & 15, ty = tid >> 4;  // 16 x 16 threads, 4 x 4 each
  float acc[4][4] = {};
  for (int k0 = 0; k0 < K; k0 += BK) {
    // A tile: 64 rows x 16 k (4 per thread)
    for (int q = tid; q < BM * BK; q += 256) {
      const int r = q / BK, kk = q % BK;
      As[kk][r] = (r < nrows) ? Ae[static_cast<size_t>(r) * K + k0 + kk] : 0.f;
    }
    // B tile: 16 k x 64 n
    for (int q = tid; q < BK * BN; q += 256) {
      const int kk = q / BN, n = q % BN;
      Bs[kk][n] = (n0 + n < N) ? We[static_cast<size_t>(k0 + kk) * N + n0 + n] : 0.f;
    }
    __syncthreads();
#pragma unroll
    for (int kk = 0; kk < BK; ++kk) {
      float a[4], b[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) a[i] = As[kk][ty * 4 + i];
#pragma unroll
      for (int j = 0; j < 4; ++j) b[j] = Bs[kk][tx * 4 + j];
#pragma unroll
      for (int i = 0; i < 4; ++i)
#pragma unroll
        for (int j = 0; j < 4; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
    __syncthreads();
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = ty * 4 + i;
    if (r >= nrows) continue;
#pragma unroll
    for (int j = 0; j < 4; ++j) {
      const int n = n0 + tx * 4 + j;
      if (n >= N) continue;
      float v = acc[i][j];
      if (EPI == 0) {
        if (zout != nullptr) zout[static_cast<size_t>(row0 + r) * N + n] = v;
        v = v / (1.f + expf(-v));
      }
      out[static_cast<size_t>(row0 + r) * N + n] = v;
    }
  }
}

}  // namespace

cudaError_t launch_gemm_simt(int epi, const float* A, int a_shared, int R, const float* W, int E,
                             int K, int N, const int32_t* offsets, float* out, uint32_t* err,
                             cudaStream_t s, float* zout) {
  if (R == 0) return cudaSuccess;
  const dim3 grid(ceil_div(R, BM) + E, ceil_div(N, BN)), block(256);
  return launch_pdl(epi == 0 ? gemm_simt_kernel<0> : gemm_simt_kernel<1>, grid, block, 0, s, A,
                    a_shared, R, W, E, K, N, offsets, out, err, epi == 0 ? zout : nullptr);
}

}  // namespace moe
