// dispatch.cu - pack the routed rows contiguously by expert id (DeepSeek-V4
// EP article, section 3.3: "one send chunk per expert"; Deepseek-MoE
// sync-tax article, section 2.1: per-destination packed buffers). On one GPU
// the all-to-all layout is a stable counting sort of the flat entries
// i = t*k + j by expert id, done in three kernels with no atomics on data:
//
//  count    one CTA per chunk of kDispatchTokensPerChunk tokens: shared-memory
//           histogram of the chunk's expert ids -> hist[e][chunk]
//  scan     one CTA per expert: exclusive scan of hist[e][.] over chunks ->
//           base[e][chunk] (rows of expert e that earlier chunks own) and
//           counts[e]
//  scatter  one CTA per chunk: offsets = exclusive scan of counts (each CTA
//           recomputes it from E <= 256 values); the stable rank of an entry
//           inside its chunk comes from warp match_any + popc of the lanes
//           below it plus the counts of earlier warps; then each warp copies
//           one token row, read once with 16-byte loads and written to its k
//           destinations (or quantised to an FP8 E4M3 payload with a
//           per-token absmax scale, or one static scale for every row,
//           sync-tax article section 3.1).
//
// Small batches (R = T*k <= kDispatchFusedMaxRows) run the scatter kernel
// alone ("fused"): every CTA counts all R expert ids itself (warp-aggregated
// shared-memory counters: the totals and the entries of earlier chunks), so
// the count and scan launches and their hist/base tables drop out.
//
// With no x_perm (the grouped GEMM then gathers each routed row from x
// through src itself) the scatter kernels write only the layout: counts,
// offsets, pos and src.
//
// Expert ids outside [0, E) are skipped and flag kErrBadIndex.
#include <cstdint>
#include <type_traits>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"

namespace moe {
namespace {

constexpr int kTPC = kDispatchTokensPerChunk;

__global__ void dispatch_empty_kernel(int E, int32_t* counts, int32_t* offsets) {
  pdl_wait();
  pdl_trigger();
  for (int e = threadIdx.x; e <= E; e += blockDim.x) {
    if (e < E) counts[e] = 0;
    offsets[e] = 0;
  }
}

__global__ void __launch_bounds__(128) dispatch_count_kernel(const int32_t* __restrict__ idx,
                                                             int T, int k, int E, int nchunk,
                                                             int32_t* __restrict__ hist,
                                                             uint32_t* __restrict__ err,
                                                             uint32_t* __restrict__ zero,
                                                             int nzero) {
  __shared__ int h[kMaxExperts];
  pdl_wait();
  pdl_trigger();
  const int c = blockIdx.x;
  if (zero != nullptr && c == 0 && static_cast<int>(threadIdx.x) < nzero) zero[threadIdx.x] = 0u;
  for (int e = threadIdx.x; e < E; e += blockDim.x) h[e] = 0;
  __syncthreads();
  const long long i0 = static_cast<long long>(c) * kTPC * k;
  const long long R = static_cast<long long>(T) * k;
  const int n = static_cast<int>(min(static_cast<long long>(kTPC * k), R - i0));
  for (int q = threadIdx.x; q < n; q += blockDim.x) {
    const int e = __ldg(idx + i0 + q);
    if (e >= 0 && e < E)
      atomicAdd(&h[e], 1);
    else
      atomicOr(err, kErrBadIndex);
  }
  __syncthreads();
  for (int e = threadIdx.x; e < E; e += blockDim.x)
    hist[static_cast<size_t>(e) * nchunk + c] = h[e];
}

// Block-wide exclusive scan of one int per thread (256 threads).
__device__ __forceinline__ int block_exclusive_scan_256(int v, int* total) {
  __shared__ int warp_sums[8];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(0xffffffffu, incl, off);
    if (lane >= off) incl += o;
  }
  if (lane == 31) warp_sums[w] = incl;
  __syncthreads();
  int wbase = 0, all = 0;
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    if (i < w) wbase += warp_sums[i];
    all += warp_sums[i];
  }
  __syncthreads();
  *total = all;
  return wbase + incl - v;
}

__global__ void __launch_bounds__(256) dispatch_scan_kernel(const int32_t* __restrict__ hist,
                                                            int nchunk, int E,
                                                            int32_t* __restrict__ base,
                                                            int32_t* __restrict__ counts) {
  pdl_wait();
  pdl_trigger();
  const int e = blockIdx.x;
  const int32_t* h = hist + static_cast<size_t>(e) * nchunk;
  int32_t* b = base + static_cast<size_t>(e) * nchunk;
  // each thread owns a contiguous run of chunks
  const int per = (nchunk + 255) / 256;
  const int c0 = threadIdx.x * per;
  const int c1 = min(c0 + per, nchunk);
  int sum = 0;
  for (int c = c0; c < c1; ++c) sum += __ldg(h + c);
  int total;
  int run = block_exclusive_scan_256(sum, &total);
  for (int c = c0; c < c1; ++c) {
    b[c] = run;
    run += __ldg(h + c);
  }
  if (threadIdx.x == 0) counts[e] = total;
}

__device__ __forceinline__ float bf16_to_f32(uint16_t u) {
  return __uint_as_float(static_cast<uint32_t>(u) << 16);
}

// Running largest magnitudes of bf16 pairs (max is exact in bf16), and the
// largest of a pair as fp32.
__device__ __forceinline__ __nv_bfloat162 absmax8(__nv_bfloat162 m, const uint4& v) {
  const __nv_bfloat162* h = reinterpret_cast<const __nv_bfloat162*>(&v);
#pragma unroll
  for (int i = 0; i < 4; ++i) m = __hmax2(m, __habs2(h[i]));
  return m;
}
__device__ __forceinline__ float pair_max(__nv_bfloat162 m) {
  return fmaxf(__bfloat162float(m.x), __bfloat162float(m.y));
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
  return v;
}

// The token's payload scale: the static one if given, else fp32(amax / 448)
// (1 for an all-zero row).
__device__ __forceinline__ float payload_scale(float amax, float static_scale) {
  return static_scale > 0.f ? static_scale : ((amax == 0.f) ? 1.f : __fdiv_rn(amax, 448.f));
}

// Rows of up to 32 * kRowRegVecs 16-byte vectors (d <= 5120 bf16) are held
// in registers by the FP8 quantiser.
constexpr int kRowRegVecs = 20;

// 8 floats -> 8 E4M3 bytes of x / s (the IEEE quotient, then round to
// nearest even, saturating), element 0 in the lowest byte. FAST: the
// quotient from y = RN(1/s) and two residual corrections (quotient_rn, the
// same bits); otherwise one IEEE division per element. CLAMP = false: the
// caller knows |x| <= 448 s.
template <bool FAST, bool CLAMP = true>
__device__ __forceinline__ uint2 quant8(const float (&v)[8], float s, float y) {
  uint32_t w[2];
#pragma unroll
  for (int h = 0; h < 2; ++h) {
    uint32_t acc = 0;
#pragma unroll
    for (int p = 0; p < 2; ++p) {
      const float x0 = v[h * 4 + p * 2], x1 = v[h * 4 + p * 2 + 1];
      const float a = FAST ? quotient_rn<CLAMP>(x0, s, y) : __fdiv_rn(x0, s);
      const float b = FAST ? quotient_rn<CLAMP>(x1, s, y) : __fdiv_rn(x1, s);
      const __nv_fp8x2_storage_t q =
          __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
      acc |= static_cast<uint32_t>(q) << (16 * p);
    }
    w[h] = acc;
  }
  return make_uint2(w[0], w[1]);
}

// Pass 2 of the FP8 payload for one token (one warp): q = E4M3(x / s) for
// the row's 16-byte vectors, written to each of its routed rows p[j] >= 0.
// The division form (scales outside [2^-64, 2^64] only) keeps one load in
// flight per lane, so that it does not raise the kernel's register count.
template <bool FAST>
__device__ __forceinline__ void quant_row(const uint4* __restrict__ xr, int nvec, int lane,
                                          float s, const int (&p)[kMaxTopK],
                                          uint2* __restrict__ dst) {
  const float y = FAST ? __frcp_rn(s) : 0.f;
  const size_t row_vecs = static_cast<size_t>(nvec);
  constexpr int UQ = FAST ? 4 : 1;
  for (int v0 = lane; v0 < nvec; v0 += 32 * UQ) {
    uint4 val[UQ];
#pragma unroll
    for (int u = 0; u < UQ; ++u)
      if (v0 + 32 * u < nvec) val[u] = __ldg(xr + v0 + 32 * u);
#pragma unroll
    for (int u = 0; u < UQ; ++u) {
      const int v = v0 + 32 * u;
      if (v >= nvec) break;
      const uint16_t* h = reinterpret_cast<const uint16_t*>(&val[u]);
      float f[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) f[i] = bf16_to_f32(h[i]);
      const uint2 q = quant8<FAST>(f, s, y);
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (p[j] >= 0) dst[static_cast<size_t>(p[j]) * row_vecs + v] = q;
    }
  }
}

// dtype 0: fp32 rows, 1: bf16 rows. FP8 only with bf16. FUSED: counts and
// the earlier chunks' rows per expert come from this CTA's own pass over all
// ids (counts is then an output, base unused; `zero` gets nzero zero words).
template <int DT, bool FP8, bool FUSED>
__global__ void __launch_bounds__(256) dispatch_scatter_kernel(
    const void* __restrict__ xv, const int32_t* __restrict__ idx, int T, int d, int k, int E,
    int nchunk, int32_t* __restrict__ counts, const int32_t* __restrict__ base,
    int32_t* __restrict__ offsets, int32_t* __restrict__ pos, int32_t* __restrict__ src,
    void* __restrict__ x_perm, float* __restrict__ x_scale, float static_scale,
    uint32_t* __restrict__ err, uint32_t* __restrict__ zero, int nzero, int bulk) {
  __shared__ int off_s[kMaxExperts + 1];
  __shared__ uint64_t rows_bar;
  __shared__ int cnt_w[2][kMaxExperts];  // per-warp expert counts (<= 64 entries, 2 warps)
  __shared__ int pos_s[kTPC * kMaxTopK];
  __shared__ int tot_s[FUSED ? kMaxExperts : 1];     // FUSED: rows per expert
  __shared__ int before_s[FUSED ? kMaxExperts : 1];  // FUSED: rows in earlier chunks
  pdl_wait();
  pdl_trigger();
  const int tid = threadIdx.x, lane = tid & 31, w = tid >> 5;
  const int c = blockIdx.x;
  const long long R = static_cast<long long>(T) * k;
  const long long i0 = static_cast<long long>(c) * kTPC * k;

  if constexpr (FUSED) {
    if (zero != nullptr && c == 0 && tid < nzero) zero[tid] = 0u;
    for (int e = tid; e < E; e += 256) {
      tot_s[e] = 0;
      before_s[e] = 0;
    }
    __syncthreads();
    // every CTA counts all R ids; a warp's equal ids are added at once
    for (long long b0 = static_cast<long long>(w) * 32; b0 < R; b0 += 256) {
      const long long i = b0 + lane;
      int e = i < R ? __ldg(idx + i) : -1;
      const bool valid = e >= 0 && e < E;
      if (i < R && !valid && c == 0) atomicOr(err, kErrBadIndex);
      if (!valid) e = -1;
      const unsigned mask = __match_any_sync(0xffffffffu, e);
      const unsigned early = __ballot_sync(0xffffffffu, i < i0);
      if (valid && lane == __ffs(mask) - 1) {
        atomicAdd(&tot_s[e], __popc(mask));
        const int nb = __popc(mask & early);
        if (nb) atomicAdd(&before_s[e], nb);
      }
    }
    __syncthreads();
  }

  // offsets = exclusive scan of counts
  {
    const int v = (tid < E) ? (FUSED ? tot_s[tid] : __ldg(counts + tid)) : 0;
    int total;
    const int ex = block_exclusive_scan_256(v, &total);
    if (tid < E) off_s[tid] = ex;
    if (tid == 0) off_s[E] = total;
    if (c == 0) {
      if (tid < E) offsets[tid] = ex;
      if (tid == 0) offsets[E] = total;
      if (FUSED && tid < E) counts[tid] = v;
    }
  }
  for (int q = tid; q < 2 * kMaxExperts; q += 256) (&cnt_w[0][0])[q] = 0;
  __syncthreads();

  // stable ranks of this chunk's entries (at most 64: warps 0 and 1)
  const int n = static_cast<int>(min(static_cast<long long>(kTPC * k), R - i0));
  int e = -2;
  unsigned mask = 0;
  if (w < 2) {
    const int q = w * 32 + lane;
    if (q < n) {
      e = __ldg(idx + i0 + q);
      if (e < 0 || e >= E) e = -1;
    }
    mask = __match_any_sync(0xffffffffu, e);
    const int leader = __ffs(mask) - 1;
    if (lane == leader && e >= 0) cnt_w[w][e] = __popc(mask);
  }
  __syncthreads();
  if (w < 2) {
    const int q = w * 32 + lane;
    if (q < n) {
      int p = -1;
      if (e >= 0) {
        const int before = (w == 1) ? cnt_w[0][e] : 0;
        const int rank = before + __popc(mask & ((1u << lane) - 1u));
        p = off_s[e] + (FUSED ? before_s[e] : __ldg(base + static_cast<size_t>(e) * nchunk + c)) +
            rank;
        src[p] = static_cast<int32_t>((i0 + q) / k);
      }
      pos[i0 + q] = p;
      pos_s[q] = p;
    }
  }
  if (x_perm == nullptr) return;  // layout only: no rows are packed
  __syncthreads();

  if constexpr (!FP8) {
    constexpr int ES = DT == 0 ? 4 : 2;
    if (bulk) {
      // rows of at most kDispatchBulkRowBytes: warp 0 pulls the chunk's rows
      // into shared memory with bulk copies (one round of latency) and sends
      // each to its k destinations with bulk stores (asynchronous, no
      // register traffic); the other warps are done
      extern __shared__ __align__(16) uint8_t rows_s[];
      if (w != 0) return;
      const int t0 = c * kTPC;
      const int ntok = min(kTPC, T - t0);
      const uint32_t rb = static_cast<uint32_t>(d) * ES;
      if (lane == 0) {
        ptx::mbar_init(&rows_bar, 1);
        ptx::fence_mbar_init();
        ptx::mbar_arrive_expect_tx(&rows_bar, rb * static_cast<uint32_t>(ntok));
        for (int q = 0; q < ntok; ++q)
          ptx::bulk_load(rows_s + q * rb,
                         static_cast<const char*>(xv) + static_cast<size_t>(t0 + q) * rb, rb,
                         &rows_bar);
      }
      __syncwarp();
      if (!__all_sync(0xffffffffu, ptx::mbar_wait(&rows_bar, 0, kWaitLimitNs))) {
        if (lane == 0) atomicOr(err, kErrTimeout);
        ptx::mbar_wait(&rows_bar, 0, kWaitLimitNs);  // the copies land before exit
        return;
      }
      for (int qj = lane; qj < ntok * k; qj += 32) {
        const int pj = pos_s[qj];
        if (pj >= 0)
          ptx::bulk_store(static_cast<char*>(x_perm) + static_cast<size_t>(pj) * rb,
                          rows_s + (qj / k) * rb, rb);
      }
      ptx::bulk_commit_group();
      ptx::bulk_wait_group0();  // the rows are written before the CTA exits
      return;
    }
    // row copy: the whole CTA strides the chunk's rows (16-byte vectors),
    // four loads in flight per thread; each row is read once and written to
    // its k destinations
    const int nvec = d * ES / 16;
    const int t0 = c * kTPC;
    const int ntok = min(kTPC, T - t0);
    const int items = ntok * nvec;
    const uint4* xr = reinterpret_cast<const uint4*>(static_cast<const char*>(xv) +
                                                     static_cast<size_t>(t0) * d * ES);
    uint4* dst = reinterpret_cast<uint4*>(x_perm);
    const size_t row_vecs = static_cast<size_t>(nvec);
    constexpr int U = 4;
    for (int base = tid; base < items; base += 256 * U) {
      uint4 val[U];
      int it[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        it[u] = base + u * 256;
        if (it[u] < items) val[u] = __ldg(xr + it[u]);
      }
#pragma unroll
      for (int u = 0; u < U; ++u) {
        if (it[u] >= items) continue;
        const int q = it[u] / nvec, v = it[u] - q * nvec;
        for (int j = 0; j < k; ++j) {
          const int pj = pos_s[q * k + j];
          if (pj >= 0) dst[static_cast<size_t>(pj) * row_vecs + v] = val[u];
        }
      }
    }
    return;
  }

  // FP8 payload: warp w quantises token t0 + w
  const int t = c * kTPC + w;
  if (t >= T) return;
  int p[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) p[j] = (j < k) ? pos_s[w * k + j] : -1;

  if constexpr (FP8) {
    const int nvec = d / 8;
    const uint4* xr =
        reinterpret_cast<const uint4*>(static_cast<const __nv_bfloat16*>(xv) +
                                       static_cast<size_t>(t) * d);
    uint2* dst = reinterpret_cast<uint2*>(x_perm);
    float s;
    if (nvec <= 32 * kRowRegVecs) {
      // one read of the row: it stays in registers (kRowRegVecs 16-byte
      // vectors per lane, all loads in flight at once) between the absmax
      // and the cast
      uint4 val[kRowRegVecs];
#pragma unroll
      for (int u = 0; u < kRowRegVecs; ++u)
        if (lane + 32 * u < nvec) val[u] = __ldg(xr + lane + 32 * u);
      float amax = 0.f;
      if (static_scale <= 0.f) {
        __nv_bfloat162 m2 = __floats2bfloat162_rn(0.f, 0.f);
#pragma unroll
        for (int u = 0; u < kRowRegVecs; ++u)
          if (lane + 32 * u < nvec) m2 = absmax8(m2, val[u]);
        amax = warp_max(pair_max(m2));
      }
      s = payload_scale(amax, static_scale);
      if (quotient_scale_ok(s)) {  // s is uniform across the warp
        const float y = __frcp_rn(s);
        const size_t row_vecs = static_cast<size_t>(nvec);
        // a per-token scale bounds every |x / s| by 448: no clamp
        auto quant_reg = [&](auto clamp) {
#pragma unroll
          for (int u = 0; u < kRowRegVecs; ++u) {
            const int v = lane + 32 * u;
            if (v >= nvec) break;
            const uint16_t* h = reinterpret_cast<const uint16_t*>(&val[u]);
            float f[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) f[i] = bf16_to_f32(h[i]);
            const uint2 q = quant8<true, decltype(clamp)::value>(f, s, y);
#pragma unroll
            for (int j = 0; j < kMaxTopK; ++j)
              if (p[j] >= 0) dst[static_cast<size_t>(p[j]) * row_vecs + v] = q;
          }
        };
        if (static_scale > 0.f)
          quant_reg(std::true_type{});
        else
          quant_reg(std::false_type{});
      } else {
        quant_row<false>(xr, nvec, lane, s, p, dst);
      }
    } else {
      // wider rows: pass 1 reads the row for its absmax (skipped with a
      // static scale), pass 2 reads it again, from L2
      constexpr int UQ = 4;  // 16-byte loads in flight per lane
      float amax = 0.f;
      for (int v0 = lane; static_scale <= 0.f && v0 < nvec; v0 += 32 * UQ) {
        uint4 val[UQ];
#pragma unroll
        for (int u = 0; u < UQ; ++u)
          if (v0 + 32 * u < nvec) val[u] = __ldg(xr + v0 + 32 * u);
#pragma unroll
        for (int u = 0; u < UQ; ++u) {
          if (v0 + 32 * u >= nvec) break;
          amax = fmaxf(amax, pair_max(absmax8(__floats2bfloat162_rn(0.f, 0.f), val[u])));
        }
      }
      amax = warp_max(amax);
      s = payload_scale(amax, static_scale);
      if (quotient_scale_ok(s))
        quant_row<true>(xr, nvec, lane, s, p, dst);
      else
        quant_row<false>(xr, nvec, lane, s, p, dst);
    }
    if (lane == 0) {
#pragma unroll
      for (int j = 0; j < kMaxTopK; ++j)
        if (p[j] >= 0) x_scale[p[j]] = s;
    }
  }
}

// Soft gating sends every token to every expert in token order: the layout
// is known without counting. counts[e] = T, offsets[e] = e T, pos[t E + e] =
// e T + t, src[e T + t] = t; also zeroes `nzero` words at `zero` (the GEMM
// tile counters).
__global__ void __launch_bounds__(256) dense_layout_kernel(int T, int E, int32_t* __restrict__ counts,
                                                           int32_t* __restrict__ offsets,
                                                           int32_t* __restrict__ pos,
                                                           int32_t* __restrict__ src,
                                                           uint32_t* __restrict__ zero, int nzero) {
  pdl_wait();
  pdl_trigger();
  const long long R = static_cast<long long>(T) * E;
  const long long i = static_cast<long long>(blockIdx.x) * 256 + threadIdx.x;
  if (i < R) {
    const int t = static_cast<int>(i / E), e = static_cast<int>(i % E);
    pos[i] = e * T + t;
    src[i] = static_cast<int32_t>(i % T);  // row i = e' T + t' holds token t'
  }
  if (blockIdx.x == 0) {
    if (threadIdx.x <= E) offsets[threadIdx.x] = threadIdx.x * T;
    if (threadIdx.x < E) counts[threadIdx.x] = T;
    if (zero != nullptr && threadIdx.x < nzero) zero[threadIdx.x] = 0u;
  }
}

// x_perm[pos[t k + j]] = x[t] for every token t and slot j < k (rows of
// `vecs` 16-byte vectors): one warp per token reads its row once, four
// vectors per lane in flight, and writes them to each of the token's k
// routed rows (reading x once per routed row instead moved k times the
// bytes). A pos outside [0, R) (the dispatch's mark of an entry it
// dropped) is skipped.
__global__ void __launch_bounds__(256) scatter_rows_kernel(const uint4* __restrict__ x,
                                                           const int32_t* __restrict__ pos, int T,
                                                           int k, long long R, int vecs,
                                                           uint4* __restrict__ x_perm) {
  pdl_wait();
  pdl_trigger();
  const long long t = static_cast<long long>(blockIdx.x) * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  const int lane = threadIdx.x & 31;
  int p[kMaxTopK];
#pragma unroll
  for (int j = 0; j < kMaxTopK; ++j) {
    p[j] = j < k ? __ldg(pos + t * k + j) : -1;
    if (p[j] >= R) p[j] = -1;
  }
  const uint4* a = x + static_cast<size_t>(t) * vecs;
  constexpr int U = 4;
  for (int v0 = lane; v0 < vecs; v0 += 32 * U) {
    uint4 val[U];
#pragma unroll
    for (int u = 0; u < U; ++u)
      if (v0 + 32 * u < vecs) val[u] = __ldg(a + v0 + 32 * u);
#pragma unroll
    for (int j = 0; j < kMaxTopK; ++j) {
      if (p[j] < 0) continue;
      uint4* b = x_perm + static_cast<size_t>(p[j]) * vecs;
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (v0 + 32 * u < vecs) b[v0 + 32 * u] = val[u];
    }
  }
}

// Rows copied by bulk copies through shared memory: plain (not FP8) rows of
// at most kDispatchBulkRowBytes (the chunk's rows take kTPC times that).
constexpr int kDispatchBulkRowBytes = 8192;
int bulk_rows(int dtype, int fp8, int d) {
  const long long rb = static_cast<long long>(d) * (dtype == 0 ? 4 : 2);
  return !fp8 && rb % 16 == 0 && rb <= kDispatchBulkRowBytes ? 1 : 0;
}

// Opt the plain-row scatter kernels into their shared memory, once.
template <typename K>
cudaError_t set_bulk_smem(K) {
  static std::once_flag once;
  static cudaError_t st = cudaSuccess;
  std::call_once(once, [] {
    const int bytes = kTPC * kDispatchBulkRowBytes;
    const auto a = cudaFuncAttributeMaxDynamicSharedMemorySize;
    st = cudaFuncSetAttribute(dispatch_scatter_kernel<0, false, false>, a, bytes);
    if (st == cudaSuccess) st = cudaFuncSetAttribute(dispatch_scatter_kernel<1, false, false>, a, bytes);
    if (st == cudaSuccess) st = cudaFuncSetAttribute(dispatch_scatter_kernel<0, false, true>, a, bytes);
    if (st == cudaSuccess) st = cudaFuncSetAttribute(dispatch_scatter_kernel<1, false, true>, a, bytes);
  });
  return st;
}

}  // namespace

cudaError_t launch_dispatch_empty(int E, int32_t* counts, int32_t* offsets, cudaStream_t s) {
  return launch_pdl(dispatch_empty_kernel, dim3(1), dim3(256), 0, s, E, counts, offsets);
}

cudaError_t launch_dispatch_count(const int32_t* topk_idx, int T, int k, int E, int nchunk,
                                  int32_t* hist, uint32_t* err, uint32_t* zero, int nzero,
                                  cudaStream_t s) {
  return launch_pdl(dispatch_count_kernel, dim3(nchunk), dim3(128), 0, s, topk_idx, T, k, E,
                    nchunk, hist, err, zero, nzero);
}

cudaError_t launch_dispatch_scan(const int32_t* hist, int nchunk, int E, int32_t* base,
                                 int32_t* counts, cudaStream_t s) {
  return launch_pdl(dispatch_scan_kernel, dim3(E), dim3(256), 0, s, hist, nchunk, E, base,
                    counts);
}

cudaError_t launch_dispatch_scatter(int dtype, int fp8, float static_scale, const void* x,
                                    const int32_t* topk_idx, int T, int d, int k, int E,
                                    int nchunk, const int32_t* counts, const int32_t* base,
                                    int32_t* offsets, int32_t* pos, int32_t* src, void* x_perm,
                                    float* x_scale, uint32_t* err, cudaStream_t s) {
  const dim3 grid(nchunk), block(256);
  auto kernel = dtype == 0 ? dispatch_scatter_kernel<0, false, false>
                : (!fp8 ? dispatch_scatter_kernel<1, false, false>
                        : dispatch_scatter_kernel<1, true, false>);
  const int bulk = x_perm != nullptr ? bulk_rows(dtype, fp8, d) : 0;
  const size_t smem = bulk ? static_cast<size_t>(kTPC) * d * (dtype == 0 ? 4 : 2) : 0;
  if (bulk) {
    const cudaError_t st = set_bulk_smem(kernel);
    if (st != cudaSuccess) return st;
  }
  return launch_pdl(kernel, grid, block, smem, s, x, topk_idx, T, d, k, E, nchunk,
                    const_cast<int32_t*>(counts), base, offsets, pos, src, x_perm, x_scale,
                    static_scale, err, static_cast<uint32_t*>(nullptr), 0, bulk);
}

cudaError_t launch_dispatch_fused(int dtype, int fp8, float static_scale, const void* x,
                                  const int32_t* topk_idx, int T, int d, int k, int E,
                                  int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                                  void* x_perm, float* x_scale, uint32_t* err, uint32_t* zero,
                                  int nzero, cudaStream_t s) {
  const int nchunk = ceil_div(T, kTPC);
  const dim3 grid(nchunk), block(256);
  auto kernel = dtype == 0 ? dispatch_scatter_kernel<0, false, true>
                : (!fp8 ? dispatch_scatter_kernel<1, false, true>
                        : dispatch_scatter_kernel<1, true, true>);
  const int bulk = x_perm != nullptr ? bulk_rows(dtype, fp8, d) : 0;
  const size_t smem = bulk ? static_cast<size_t>(kTPC) * d * (dtype == 0 ? 4 : 2) : 0;
  if (bulk) {
    const cudaError_t st = set_bulk_smem(kernel);
    if (st != cudaSuccess) return st;
  }
  return launch_pdl(kernel, grid, block, smem, s, x, topk_idx, T, d, k, E, nchunk, counts,
                    static_cast<const int32_t*>(nullptr), offsets, pos, src, x_perm, x_scale,
                    static_scale, err, zero, nzero, bulk);
}

cudaError_t launch_scatter_rows(int dtype, const void* x, const int32_t* pos, int T, int k,
                                int d, void* x_perm, cudaStream_t s) {
  if (T <= 0) return cudaSuccess;
  if (k < 1 || k > kMaxTopK) return cudaErrorInvalidValue;
  const int vecs = d * (dtype == 0 ? 4 : 2) / 16;
  return launch_pdl(scatter_rows_kernel, dim3(ceil_div(T, 8)), dim3(256), 0, s,
                    static_cast<const uint4*>(x), pos, T, k,
                    static_cast<long long>(T) * k, vecs, static_cast<uint4*>(x_perm));
}

cudaError_t launch_dense_layout(int T, int E, int32_t* counts, int32_t* offsets, int32_t* pos,
                                int32_t* src, uint32_t* zero, int nzero, cudaStream_t s) {
  const long long R = static_cast<long long>(T) * E;
  const int blocks = static_cast<int>((R + 255) / 256) > 0 ? static_cast<int>((R + 255) / 256) : 1;
  return launch_pdl(dense_layout_kernel, dim3(blocks), dim3(256), 0, s, T, E, counts, offsets,
                    pos, src, zero, nzero);
}

}  // namespace moe
