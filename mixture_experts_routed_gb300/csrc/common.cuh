// common.cuh - internal declarations shared by the kernel translation units
// and the C-ABI layer (moe_abi.cu). Nothing here is exported.
#pragma once

#include <cstddef>
#include <cstdint>
#include <utility>
#include <cuda_runtime.h>

namespace moe {

// ---------------------------------------------------------------- launch
// Programmatic dependent launch: every kernel of the layer is launched with
// programmatic stream serialisation, so its CTAs may be scheduled while the
// previous kernel in the stream is still draining. Each kernel calls
// pdl_wait() before its first global-memory access (read or write); it
// returns once the previous grid has completed and its writes are visible,
// which by induction orders it after every earlier kernel of the stream.
// pdl_trigger() lets the next kernel be scheduled (it takes effect once
// every CTA of this grid has issued it or exited).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ------------------------------------------------------------ quotient
// x / s rounded to nearest even (the IEEE quotient) without a division per
// element. With y = RN(1/s) (one correctly rounded reciprocal per row),
// q = RN(x y) is within two ulps of x / s; a correction
// q <- RN(q + RN(x - s q) y), the residual from one FMA, brings it within
// one ulp, and by Markstein's theorem (P. Markstein, IBM J. Res. Dev. 34(1),
// 1990; Muller et al., Handbook of Floating-Point Arithmetic, ch. 4) a second
// one then gives the correctly rounded quotient: once q is within one ulp,
// the residual is exact. The callers take this path only for s in
// [2^-64, 2^64] (y normal). The theorem wants no underflow: for quotients
// of magnitude 2^-11 or more the exact residual x - s q is a multiple of
// ulp(s) ulp(q) >= 2^-121, so normal or zero; smaller quotients lie below
// the first E4M3 rounding boundary (2^-10), where the code is +-0 whatever
// their last bits, and the sign of x is kept.
// CLAMP: quotients of magnitude above 1024 (the first product says so to
// within 2^-22) saturate to +-448 in E4M3 either way and are returned as
// +-1024, which keeps the corrections away from overflow; without it the
// caller guarantees |x| <= 448 s (x within the row's absmax, s = amax / 448
// rounded). For finite x.
__device__ __forceinline__ bool quotient_scale_ok(float s) {
  return s >= 0x1p-64f && s <= 0x1p64f;
}
template <bool CLAMP = true>
__device__ __forceinline__ float quotient_rn(float x, float s, float y) {
  float q = __fmul_rn(x, y);
  const bool big = CLAMP && fabsf(q) > 1024.f;
  float r = __fmaf_rn(-s, q, x);
  q = __fmaf_rn(r, y, q);
  r = __fmaf_rn(-s, q, x);
  q = __fmaf_rn(r, y, q);
  return copysignf(big ? 1024.f : q, x);
}

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t s, Args&&... args) {
  cudaLaunchConfig_t lc = {};
  lc.gridDim = grid;
  lc.blockDim = block;
  lc.dynamicSmemBytes = smem;
  lc.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 1;
  return cudaLaunchKernelEx(&lc, kernel, std::forward<Args>(args)...);
}

// Bits of the device error word (the first 4 bytes of the workspace).
constexpr uint32_t kErrBadIndex = 1u;
constexpr uint32_t kErrTimeout = 2u;

// Tile counters of the two expert GEMMs: 32-bit words of the workspace's
// first 256-byte block (after the error word), zeroed before each layer.
constexpr size_t kGemmCounterOffset = 64;
constexpr int kNumGemmCounters = 2;

// Bound on any device-side wait (mbarrier): 2 s of wall time.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// Dispatch works on chunks of this many tokens (one CTA per chunk).
constexpr int kDispatchTokensPerChunk = 8;

constexpr int kMaxExperts = 256;
constexpr int kMaxTopK = 8;

// Router parameters, as in moe_config_t. mode: 0 renormalised top-k, 1
// softmax over the pre_k largest logits, 2 group-limited top-k (the k best
// experts inside the topk_group best of n_group groups of consecutive ids),
// 3 soft gating (softmax((L + noise) / tau) over all E experts, k = E).
struct RouterSpec {
  int k;
  int pre_k;
  int mode;
  int n_group;
  int topk_group;
  float tau;
  const float* noise;  // [T, E] Gumbel samples (soft gating)
};
constexpr int kMaxGroups = 32;
// Rows a token may fan out to (k): kMaxTopK for the top-k routers, up to
// kMaxFanout (= E) for soft gating.
constexpr int kMaxFanout = 16;

inline int ceil_div(int a, int b) { return (a + b - 1) / b; }
inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------------- route.cu
// Gate GEMM + softmax + top-k, fused. `dtype` 0 = fp32, 1 = bf16. `err`
// (nullable) receives kErrTimeout from the tensor-core gate.
cudaError_t launch_route(int dtype, const void* x, const void* Wg, const float* bias, int T,
                         int d, int E, RouterSpec rs, int32_t* topk_idx,
                         float* topk_w, float* logits, uint32_t* err, cudaStream_t s);

// ---------------------------------------------------------------- gate_tc.cu
// Tensor-core gate (bf16, E a multiple of 8 up to 256, 16-byte aligned x, W_g).
bool gate_tc_supported(int dtype, int E, const void* Wg, const void* x);
cudaError_t launch_gate_tc(const void* x, const void* Wg, const float* bias, int T, int d, int E,
                           RouterSpec rs, int32_t* topk_idx, float* topk_w,
                           float* logits, uint32_t* err, cudaStream_t s);

// ---------------------------------------------------------------- dispatch.cu
// Zero counts[E] and offsets[E+1] (empty batch).
cudaError_t launch_dispatch_empty(int E, int32_t* counts, int32_t* offsets, cudaStream_t s);
// Per-chunk histograms -> hist[e * nchunk + c]; also zeroes `nzero` words
// at `zero` (the GEMM tile counters) when non-null.
cudaError_t launch_dispatch_count(const int32_t* topk_idx, int T, int k, int E, int nchunk,
                                  int32_t* hist, uint32_t* err, uint32_t* zero, int nzero,
                                  cudaStream_t s);
// Per-expert exclusive scan over chunks -> base[e * nchunk + c], counts[e].
cudaError_t launch_dispatch_scan(const int32_t* hist, int nchunk, int E, int32_t* base,
                                 int32_t* counts, cudaStream_t s);
// Stable ranks -> pos, src, offsets; row copy (or FP8 quantisation) -> x_perm.
// FP8 scale per row: static_scale when > 0, else the row's absmax / 448.
cudaError_t launch_dispatch_scatter(int dtype, int fp8, float static_scale, const void* x,
                                    const int32_t* topk_idx,
                                    int T, int d, int k, int E, int nchunk,
                                    const int32_t* counts, const int32_t* base,
                                    int32_t* offsets, int32_t* pos, int32_t* src, void* x_perm,
                                    float* x_scale, uint32_t* err, cudaStream_t s);
// Small batches (R <= kDispatchFusedMaxRows): count, scan and scatter in one
// kernel (each CTA counts all ids); also zeroes `nzero` words at `zero`.
constexpr long long kDispatchFusedMaxRows = 4096;
cudaError_t launch_dispatch_fused(int dtype, int fp8, float static_scale, const void* x,
                                  const int32_t* topk_idx, int T, int d, int k, int E,
                                  int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                                  void* x_perm, float* x_scale, uint32_t* err, uint32_t* zero,
                                  int nzero, cudaStream_t s);
// x_perm[pos[t k + j]] = x[t] for every token and slot (rows of d elements
// of dtype; the dispatch's layout, k <= kMaxTopK); entries with pos outside
// [0, T k) are skipped.
cudaError_t launch_scatter_rows(int dtype, const void* x, const int32_t* pos, int T, int k,
                                int d, void* x_perm, cudaStream_t s);
// Soft gating's layout (every token to every expert, token order): counts,
// offsets, pos, src; zeroes `nzero` words at `zero` when non-null.
cudaError_t launch_dense_layout(int T, int E, int32_t* counts, int32_t* offsets, int32_t* pos,
                                int32_t* src, uint32_t* zero, int nzero, cudaStream_t s);

// ---------------------------------------------------------------- combine.cu
cudaError_t launch_combine(int dtype, const float* y, const int32_t* pos, const float* w, int T,
                           int d, int k, int R, void* out, uint32_t* err, cudaStream_t s);

// ---------------------------------------------------------------- payload_out.cu
// Per-row min/max affine FP8 quantisation of the expert outputs, and the
// combine that decodes it.
cudaError_t launch_quantize_out(const float* y, int R, int d, uint8_t* yq, float* ys, float* yz,
                                cudaStream_t s);
cudaError_t launch_combine_fp8(int dtype, const uint8_t* yq, const float* ys, const float* yz,
                               const int32_t* pos, const float* w, int T, int d, int k, int R,
                               void* out, uint32_t* err, cudaStream_t s);

// ---------------------------------------------------------------- gemm_tc.cu
// Grouped GEMM over expert segments on tcgen05: out[r] = epi(A[a(r)] . W[e])
// for the rows r of expert e's segment [offsets[e], offsets[e+1]); a(r) = r,
// or r - offsets[e] when a_shared (every expert reads the same a_rows rows of
// A). A [a_rows, K] bf16, or E4M3 bytes when a_fp8 (epi 0 only: expanded to
// bf16 in shared memory, the row scale applied in the epilogue); W [E, K, N]
// bf16. epi 0: (row scale) -> SiLU -> bf16 out; epi 1: fp32 out.
// `tile_ctr` must be zero at launch. tile_n: 0 (the built-in choice of pair
// tile width), 256 or 512 (forced; the fp8 token rows always take 256).
// gather_src non-null (epi 0, bf16, not a_shared): A is x [a_rows, K] and
// routed row r reads x row gather_src[r] (no packed copy of the rows).
// zout non-null (epi 0): the pre-activation Z [R, N] (fp32, after the row
// scale: the value SiLU takes) is written too.
// Bound of the grouped GEMM epilogue's wait for a finished accumulator in
// later launches (0: the default kWaitLimitNs); a test hook.
void set_gemm_epilogue_wait_ns(uint64_t ns);
cudaError_t launch_gemm_tc(int epi, const void* A, int a_fp8, int a_rows, int a_shared, int R,
                           const void* W, int E, int K, int N, const int32_t* offsets,
                           const float* row_scale, void* out, uint32_t* err, uint32_t* tile_ctr,
                           const int32_t* gather_src, int tile_n, int num_sms, cudaStream_t s,
                           float* zout = nullptr);

// ---------------------------------------------------------------- backward.cu
// The backward pass's kernels (dtype 0 = fp32, 1 = bf16 for the tensors the
// forward takes; every gradient and intermediate is fp32).
// dY[pos(t,j)] = w[t,j] dout[t] (when dY is non-null; when dYs is, its bf16
// split [R][2d] = [hi | lo]); hs (bf16 layers, nullable): for p = pos(t,j),
// the bf16 split [R][2f] of w[t,j] h[p] (h the forward's H [R][f]);
// dw[t,j] = <dout[t], Y[pos(t,j)]>; also zeroes `nzero`
// words at `zero`, writes seg01 = {0, T} and, when segk is non-null, the
// token chunks segk[i] = min(i chunk, T), i = 0 .. nsegk (nsegk < 128).
// doutp, wr (nullable): per routed row p = pos(t, j), dout[t] (the layer's dtype,
// bit for bit) and w[t, j].
cudaError_t launch_combine_bwd(int dtype, const void* dout, const float* y, const int32_t* pos,
                               const float* w, int T, int d, int k, int R, float* dY, void* dYs,
                               const void* h, int f, void* hs, void* doutp, float* wr, float* dw,
                               uint32_t* err, uint32_t* zero, int nzero, int32_t* seg01,
                               int32_t* segk, int nsegk, int chunk, cudaStream_t s);
// dL [T, E] from dw through the router's softmax Jacobian (mode as RouterSpec),
// and, when dLs is non-null, its bf16 split [T][2E] = [hi | lo].
cudaError_t launch_router_bwd(const float* L, const int32_t* idx, const float* w, const float* dw,
                              int T, int E, int k, int mode, int pre_k, float tau, float* dL,
                              void* dLs, cudaStream_t s);
// out[r] = A[r] . W[e]^T over the segments (W [E][N][K], dtype wdtype);
// silu: out holds Z and gets acc * SiLU'(Z).
cudaError_t launch_gemm_nt(int wdtype, bool silu, const float* A, const void* W, int E, int R,
                           int K, int N, const int32_t* offsets, float* out, uint32_t* err,
                           cudaStream_t s);
// out[e] = A_e^T . B_e over each segment's rows (A [*, M] dtype adtype,
// shared rows when a_shared; B fp32 [R, N]); out [E][M][N].
// The same GEMM with the weights stored transposed: y[r] = A[r] . W_e^T,
// W bf16 [E][N][k_wrap] row-major, A bf16 [R, K] with K = k_wrap or
// 2 k_wrap (k >= k_wrap reads weight column k - k_wrap: the hi | lo operand
// split against one weight). zin null: out = y, fp32 [R, N]; else out =
// the bf16 split [R][2N] = [hi | lo] of (row_scale[r] y) * SiLU'(zin) (zin
// fp32 [R, N]; row_scale nullable: 1). a_shared: A holds a_rows rows and
// row r of expert e reads row r - offsets[e] (else a_rows = R).
cudaError_t launch_gemm_tc_wt(const void* A, int R, const void* Wt, int E, int K, int k_wrap,
                              int N, const int32_t* offsets, const float* zin, void* out,
                              uint32_t* err, uint32_t* tile_ctr, int num_sms, cudaStream_t s,
                              const float* row_scale = nullptr, int a_rows = -1,
                              int a_shared = 0);

// The experts' weight gradients on the tensor cores (wgrad_tc.cu):
// out[e] = A_e^T . (Bs_e[:, :N] + Bs_e[:, N:]) over the rows of expert e's
// segment (A row r, or r - offsets[e] with a_shared), A bf16 [a_rows, M],
// Bs bf16 [R, 2N] (the hi | lo split), out fp32 [E][M][N]; M a multiple of
// 64, N of 8.
cudaError_t launch_wgrad_tc(const void* A, int a_rows, int a_shared, const void* Bs, int R, int E,
                            int M, int N, const int32_t* offsets, float* out, uint32_t* err,
                            int num_sms, cudaStream_t s);
// The same with the split on A: out[e] = (As_e[:, :M] + As_e[:, M:])^T . B_e,
// As bf16 [R, 2M] (hi | lo), B bf16 [b_rows, N], B row r of expert e's
// segment (or r - offsets[e] with b_shared).
cudaError_t launch_wgrad_tc_split_a(const void* As, int R, const void* B, int b_rows,
                                    int b_shared, int E, int M, int N, const int32_t* offsets,
                                    float* out, uint32_t* err, int num_sms, cudaStream_t s);
cudaError_t launch_gemm_tn(int adtype, const void* A, int a_shared, const float* B, int E, int R,
                           int M, int N, const int32_t* offsets, float* out, uint32_t* err,
                           cudaStream_t s);
// part[c][e] = sum of dL[t, e] over the tokens of chunk c ([c chunk, (c+1)
// chunk), c < nchunk), in a fixed order.
cudaError_t launch_bias_bwd(const float* dL, int T, int E, int chunk, int nchunk, float* part,
                            cudaStream_t s);
// oa[i] = sum_{s < Sa} pa[s][i] (i < na) and ob likewise, s ascending; a job
// with S = 0 is skipped.
cudaError_t launch_reduce_partials(const float* pa, int Sa, size_t na, float* oa, const float* pb,
                                   int Sb, size_t nb, float* ob, cudaStream_t s);
cudaError_t launch_undispatch(const float* dxg, const float* dxp, const int32_t* pos, int T, int d,
                              int k, int R, float* dx, cudaStream_t s);

// ---------------------------------------------------------------- gemm_simt.cu
// The same grouped GEMM in fp32 FMA for fp32 layers.
// zout (epi 0, nullable): the pre-activation Z [R, N] is written too.
cudaError_t launch_gemm_simt(int epi, const float* A, int a_shared, int R, const float* W, int E,
                             int K, int N, const int32_t* offsets, float* out, uint32_t* err,
                             cudaStream_t s, float* zout = nullptr);

}  // namespace moe
