// route.cu - gate projection fused with the router (DeepSeek-V4 EP article,
// sections 2.1 and 3.2): per token, logits L = x W_g + b in fp32, then a
// warp-level partial top-pre_k by repeated warp argmax (larger logit first,
// lower expert id on ties), then the weights:
//   renorm:        w_j = exp(L_j - L_max) / sum_{i<k} exp(L_i - L_max)
//                  (= the full max-subtracted softmax of the chosen experts
//                  divided by their sum)
//   pre_k softmax: w_j = exp(L_j - L_max) / sum_{i<pre_k} exp(L_i - L_max)
//   group-limited: as renorm, over the experts of the topk_group groups with
//                  the best mean probability (DeepSeek V3/V4 parallel-
//                  strategy article, EP section: the node limit)
//   soft gating:   w_e = softmax_e((L_e + g_e) / tau) over all E experts, g
//                  the caller's Gumbel samples (sync-tax article, 3.3)
// The logits never go to HBM unless the caller asks for them.
//
// Two gate GEMM shapes:
//  * E <= 32 ("narrow"): 4 warps per token split the hidden dimension; each
//    thread accumulates its slice for all E experts, a butterfly reduces
//    inside each warp and the 4 warp partials are added in warp order.
//  * E > 32, or many tokens ("tiled"): a CTA computes a token x expert tile
//    from shared-memory staged x and W_g with a register micro-tile per
//    thread, accumulates 32-long K chunks and folds them into the totals with
//    compensated (Kahan) summation, which keeps |L - L_fp64| ~1e-7 at
//    d = 7168.
#include <cfloat>
#include <cstdint>
#include <cstddef>
#include <mutex>

#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {
namespace {

using topk::warp_select_and_weigh;

// dynamic shared memory the small-batch kernel may take
constexpr int kRouteSmemMax = 200 * 1024;

__device__ __forceinline__ float to_f32(float v) { return v; }
__device__ __forceinline__ float to_f32(__nv_bfloat16 v) { return __bfloat162float(v); }

// ---------------------------------------------------------------- small batches
// E = NE in {8, 16, 32} (bf16) or {4, 8, 16} (fp32): W_g rows of RB = 16, 32
// or 64 bytes, small enough with TPB tokens' x rows to sit in shared memory.
// A CTA of 8 warps takes TPB = 64 / NE tokens and pulls W_g and their x rows
// in with bulk copies on one mbarrier: one round of memory latency for the
// CTA, where per-thread loads of the hidden dimension took several. Thread c
// then takes x vectors c, c + 256, ... (VEC elements) of every token and the
// VEC W_g rows under them, read in a rotated order (row (j + c) % VEC first)
// so the 8 threads of a quarter-warp hit distinct banks. Partial sums: a
// reduce-scatter butterfly in each warp (lane l keeps outputs 2l, 2l + 1 of
// the 64, output q * NE + e), then the 8 warp totals added in warp order: the
// result does not depend on scheduling.
template <int N>
__device__ __forceinline__ void warp_reduce_scatter(float (&v)[N]) {
  static_assert(N % 32 == 0, "N must be a multiple of 32");
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int m = 16, len = N; m > 0; m >>= 1, len >>= 1) {
    const bool upper = (lane & m) != 0;
#pragma unroll
    for (int j = 0; j < len / 2; ++j) {
      const float send = upper ? v[j] : v[j + len / 2];
      const float keep = upper ? v[j + len / 2] : v[j];
      v[j] = keep + __shfl_xor_sync(0xffffffffu, send, m);
    }
  }
}

template <typename Tin, int NE>
__host__ __device__ constexpr int smem_tpb() { return 64 / NE; }

template <typename Tin, int NE>
size_t route_smem_bytes(int d) {
  return static_cast<size_t>(d) * NE * sizeof(Tin) +
         static_cast<size_t>(smem_tpb<Tin, NE>()) * d * sizeof(Tin) + 8 * 64 * 4 + 16;
}

template <typename Tin, int NE>
__global__ void __launch_bounds__(256) route_smem_kernel(
    const Tin* __restrict__ x, const Tin* __restrict__ Wg, const float* __restrict__ bias, int T,
    int d, int E, RouterSpec rs, int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
    float* __restrict__ logits, uint32_t* __restrict__ err) {
  constexpr int TPB = smem_tpb<Tin, NE>();
  constexpr int N = TPB * NE;  // 64 outputs
  constexpr int VEC = 16 / sizeof(Tin);
  constexpr int RB = NE * sizeof(Tin);
  constexpr int PIECES = RB / 16;
  static_assert(N == 64 && RB % 16 == 0, "shape");
  extern __shared__ __align__(16) uint8_t sm[];
  const size_t xbytes = static_cast<size_t>(d) * sizeof(Tin);
  uint8_t* sW = sm;
  uint8_t* sX = sm + static_cast<size_t>(d) * RB;
  float* part = reinterpret_cast<float*>(sX + TPB * xbytes);
  uint64_t* bar = reinterpret_cast<uint64_t*>(part + 8 * N);
  const int t0 = blockIdx.x * TPB;
  const int nt = min(TPB, T - t0);
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    ptx::mbar_init(bar, 1);
    ptx::fence_mbar_init();
  }
  __syncthreads();
  pdl_wait();
  pdl_trigger();
  if (threadIdx.x == 0) {
    const uint32_t wbytes = static_cast<uint32_t>(d) * RB;
    ptx::mbar_arrive_expect_tx(bar, wbytes + static_cast<uint32_t>(nt * xbytes));
    ptx::bulk_load(sW, Wg, wbytes, bar);
    for (int q = 0; q < nt; ++q)
      ptx::bulk_load(sX + q * xbytes, x + static_cast<size_t>(t0 + q) * d,
                     static_cast<uint32_t>(xbytes), bar);
  }
  // a timeout is a common decision of the CTA; the copies must land before
  // its shared memory is released
  if (!__syncthreads_and(ptx::mbar_wait(bar, 0, kWaitLimitNs))) {
    if (threadIdx.x == 0 && err != nullptr) atomicOr(err, kErrTimeout);
    ptx::mbar_wait(bar, 0, kWaitLimitNs);
    return;
  }

  float acc[N];
#pragma unroll
  for (int o = 0; o < N; ++o) acc[o] = 0.f;
  const int nvec = d / VEC;
  for (int v = threadIdx.x; v < nvec; v += 256) {
    float xv[TPB][VEC];
#pragma unroll
    for (int q = 0; q < TPB; ++q) {
      const uint4 u = *reinterpret_cast<const uint4*>(sX + q * xbytes + v * 16);
      const Tin* ue = reinterpret_cast<const Tin*>(&u);
#pragma unroll
      for (int jj = 0; jj < VEC; ++jj) xv[q][jj] = to_f32(ue[jj]);
    }
#pragma unroll
    for (int jj = 0; jj < VEC; ++jj) {
      const int j = (jj + threadIdx.x) & (VEC - 1);
      const uint8_t* wr = sW + (static_cast<size_t>(v) * VEC + j) * RB;
      float wv[NE];
#pragma unroll
      for (int pc = 0; pc < PIECES; ++pc) {
        const uint4 u = *reinterpret_cast<const uint4*>(wr + pc * 16);
        const Tin* ue = reinterpret_cast<const Tin*>(&u);
#pragma unroll
        for (int ee = 0; ee < 16 / static_cast<int>(sizeof(Tin)); ++ee)
          wv[pc * (16 / sizeof(Tin)) + ee] = to_f32(ue[ee]);
      }
      // x element j of the vector: a register array indexed by the rotated
      // j would go to local memory, so select it with a static loop
      float xj[TPB];
#pragma unroll
      for (int q = 0; q < TPB; ++q) {
        xj[q] = xv[q][0];
#pragma unroll
        for (int jj2 = 1; jj2 < VEC; ++jj2) xj[q] = (j == jj2) ? xv[q][jj2] : xj[q];
      }
#pragma unroll
      for (int q = 0; q < TPB; ++q)
#pragma unroll
        for (int e = 0; e < NE; ++e) acc[q * NE + e] = fmaf(xj[q], wv[e], acc[q * NE + e]);
    }
  }
  warp_reduce_scatter<N>(acc);
  part[w * N + 2 * lane] = acc[0];
  part[w * N + 2 * lane + 1] = acc[1];
  __syncthreads();

  // warp w selects for tokens t0 + w, t0 + w + 8, ...; lane e owns expert e
  for (int q = w; q < nt; q += 8) {
    const int t = t0 + q;
    float mine = -INFINITY;
    if (lane < E) {
      const int o = q * NE + lane;
      float sum = part[o];
#pragma unroll
      for (int ww = 1; ww < 8; ++ww) sum += part[ww * N + o];
      mine = sum + (bias ? __ldg(bias + lane) : 0.f);
      if (logits) logits[static_cast<size_t>(t) * E + lane] = mine;
    }
    float vv[1] = {mine};
    int id[1] = {lane < E ? lane : 0x7fffffff};
    if (rs.mode == topk::kRouterSoft) {
      topk::warp_soft_weigh<1>(vv, id, E, rs, t, topk_idx, topk_w);
    } else {
      if (rs.mode == topk::kRouterGroup) topk::warp_group_limit<1>(vv, id, E, rs);
      warp_select_and_weigh<1>(vv, id, rs, t, topk_idx, topk_w);
    }
  }
}

template <typename Tin, int NE>
cudaError_t launch_smem(const Tin* x, const Tin* Wg, const float* bias, int T, int d, int E,
                        RouterSpec rs, int32_t* topk_idx, float* topk_w, float* logits,
                        uint32_t* err, cudaStream_t s) {
  const size_t bytes = route_smem_bytes<Tin, NE>(d);
  static std::once_flag once;
  static cudaError_t st = cudaSuccess;
  std::call_once(once, [] {
    st = cudaFuncSetAttribute(route_smem_kernel<Tin, NE>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, kRouteSmemMax);
  });
  if (st != cudaSuccess) return st;
  return launch_pdl(route_smem_kernel<Tin, NE>, dim3(ceil_div(T, smem_tpb<Tin, NE>())),
                    dim3(256), bytes, s, x, Wg, bias, T, d, E, rs, topk_idx, topk_w, logits,
                    err);
}

// The small-batch kernel applies when E is one of its row widths, every x
// row and W_g start 16-byte aligned, and the tiles fit in shared memory.
// `err` may be null (the stage call has no workspace): a timeout is then
// not recorded.
template <typename Tin>
bool try_launch_smem(const Tin* x, const Tin* Wg, const float* bias, int T, int d, int E,
                     RouterSpec rs, int32_t* topk_idx, float* topk_w, float* logits,
                     uint32_t* err, cudaStream_t s, cudaError_t* out) {
  if (reinterpret_cast<uintptr_t>(Wg) % 16 != 0 ||
      reinterpret_cast<uintptr_t>(x) % 16 != 0 || (static_cast<size_t>(d) * sizeof(Tin)) % 16 != 0)
    return false;
  constexpr int E1 = 16 / sizeof(Tin);  // 16-byte rows
#define MOE_SMEM(NE)                                                                         \
  if (E == NE && route_smem_bytes<Tin, NE>(d) <= static_cast<size_t>(kRouteSmemMax)) {      \
    *out = launch_smem<Tin, NE>(x, Wg, bias, T, d, E, rs, topk_idx, topk_w, logits, err, s); \
    return true;                                                                             \
  }
  MOE_SMEM(E1)
  MOE_SMEM(2 * E1)
  MOE_SMEM(4 * E1)
#undef MOE_SMEM
  return false;
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
    int d, int E, RouterSpec rs, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, float* __restrict__ logits) {
  constexpr int VEC = 16 / sizeof(Tin);  // elements per 16-byte load
  __shared__ float part[4][TPB][NE];
  pdl_wait();
  pdl_trigger();
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int t0 = blockIdx.x * TPB;

  float acc[TPB][NE];
#pragma unroll
  for (int q = 0; q < TPB; ++q)
#pragma unroll
    for (int e = 0; e < NE; ++e) acc[q][e] = 0.f;

  const int nvec = d / VEC;
  // unrolled so that several chunks' loads are in flight per thread (the
  // kernel is bound by load latency, not bandwidth)
#pragma unroll 4
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
    if (rs.mode == topk::kRouterSoft) {
      topk::warp_soft_weigh<1>(v, id, E, rs, t, topk_idx, topk_w);
      continue;
    }
    if (rs.mode == topk::kRouterGroup) topk::warp_group_limit<1>(v, id, E, rs);
    warp_select_and_weigh<1>(v, id, rs, t, topk_idx, topk_w);
  }
}

// ---------------------------------------------------------------- tiled
// A CTA of 256 threads computes a tile of NTT*TM tokens x NTE*TE experts
// (NTT*NTE = 256 threads). Thread (ty, tx) owns tokens ty*TM .. ty*TM+TM-1
// and experts g*(NTE*V) + tx*V + v (g < TE/V, v < V, V = min(TE, 4)), so
// each k step is one vector load of x (broadcast in the warp) plus TE/V
// vector loads of W_g (consecutive lanes read consecutive addresses). x and
// W_g stream through shared memory (fp32) in 32-long K chunks, the next
// chunk's global loads (16-byte vectors) issued before this chunk's math;
// each chunk's sums are folded into the totals with Kahan summation.
constexpr int kTileBK = 32;

template <typename Tin, int TM, int TE, int NTT, int KG, bool VW>
__global__ void __launch_bounds__(256) route_tiled_kernel(
    const Tin* __restrict__ x, const Tin* __restrict__ Wg, const float* __restrict__ bias, int T,
    int d, int E, RouterSpec rs, int32_t* __restrict__ topk_idx,
    float* __restrict__ topk_w, float* __restrict__ logits) {
  constexpr int NG = 256 / KG;     // threads per K group
  constexpr int NTE = NG / NTT;
  constexpr int BT = NTT * TM;     // tokens per tile
  constexpr int EP = NTE * TE;     // experts per tile (>= E, padded)
  constexpr int V = TE < 4 ? TE : 4;
  constexpr int G = TE / V;
  constexpr int EVEC = 16 / sizeof(Tin);               // elements per 16-byte load
  constexpr int NXV = BT * kTileBK / EVEC;              // x vectors per chunk
  constexpr int XLD = (NXV + NG - 1) / NG;               // ... per thread
  constexpr int WLD = (kTileBK * EP + NG * EVEC - 1) / (NG * EVEC);
  static_assert((BT * kTileBK) % EVEC == 0 && EP % EVEC == 0, "tile must split into vectors");
  extern __shared__ __align__(16) float tsm[];
  pdl_wait();
  pdl_trigger();
  const int kg = threadIdx.x / NG;          // this thread's K group
  const int tid = threadIdx.x % NG;         // index inside the group
  float* xs = tsm + kg * kTileBK * (BT + EP);   // [kTileBK][BT] of this group
  float* ws = xs + kTileBK * BT;                // [kTileBK][EP] of this group
  float* Ls = tsm;                              // [BT][EP] after the K loop (aliases)

  const int tx = tid % NTE, ty = tid / NTE;
  const int t0 = blockIdx.x * BT;

  float tot[TM][TE], comp[TM][TE];
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) tot[i][j] = comp[i][j] = 0.f;

  uint4 xr[XLD], wr[WLD];
  auto load_chunk = [&](int k0) {
#pragma unroll
    for (int u = 0; u < XLD; ++u) {
      const int q = tid + u * NG;                 // vector index in the tile
      const int r = q / (kTileBK / EVEC), cv = q % (kTileBK / EVEC);
      const int t = t0 + r;
      xr[u] = (q < NXV && t < T)
                  ? __ldg(reinterpret_cast<const uint4*>(x + static_cast<size_t>(t) * d + k0) + cv)
                  : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int u = 0; u < WLD; ++u) {
      const int q = tid + u * NG;
      const int r = q / (EP / EVEC), cv = q % (EP / EVEC);
      const int e0 = cv * EVEC;
      if (VW && r < kTileBK && e0 + EVEC <= E) {   // rows 16-byte aligned (checked by the launcher)
        wr[u] = __ldg(reinterpret_cast<const uint4*>(Wg + static_cast<size_t>(k0 + r) * E + e0));
      } else if (r < kTileBK && e0 < E) {          // element loads
        Tin tmp[EVEC];
#pragma unroll
        for (int i = 0; i < EVEC; ++i)
          tmp[i] = (e0 + i < E) ? Wg[static_cast<size_t>(k0 + r) * E + e0 + i] : Tin(0.f);
        wr[u] = *reinterpret_cast<const uint4*>(tmp);
      } else {
        wr[u] = make_uint4(0, 0, 0, 0);
      }
    }
  };
  auto store_chunk = [&]() {
#pragma unroll
    for (int u = 0; u < XLD; ++u) {
      const int q = tid + u * NG;
      if (q >= NXV) continue;
      const int r = q / (kTileBK / EVEC), c0 = (q % (kTileBK / EVEC)) * EVEC;
      const Tin* v = reinterpret_cast<const Tin*>(&xr[u]);
#pragma unroll
      for (int i = 0; i < EVEC; ++i) xs[(c0 + i) * BT + r] = to_f32(v[i]);
    }
#pragma unroll
    for (int u = 0; u < WLD; ++u) {
      const int q = tid + u * NG;
      const int r = q / (EP / EVEC), e0 = (q % (EP / EVEC)) * EVEC;
      if (r < kTileBK) {
        const Tin* v = reinterpret_cast<const Tin*>(&wr[u]);
#pragma unroll
        for (int i = 0; i < EVEC; ++i) ws[r * EP + e0 + i] = to_f32(v[i]);
      }
    }
  };

  // group kg takes chunks kg, kg + KG, ... (all groups run the same number of
  // iterations so that the CTA barriers line up; a group past the end idles)
  const int nchunk = d / kTileBK;
  const int iters = (nchunk + KG - 1) / KG;
  if (kg < nchunk) load_chunk(kg * kTileBK);
  for (int it = 0; it < iters; ++it) {
    const int c = it * KG + kg;
    const int k0 = c * kTileBK;
    __syncthreads();          // previous chunk's math is done with xs / ws
    if (c < nchunk) store_chunk();
    __syncthreads();
    if (c >= nchunk) continue;
    if (c + KG < nchunk) load_chunk(k0 + KG * kTileBK);
    float acc[TM][TE];
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TE; ++j) acc[i][j] = 0.f;
#pragma unroll 4
    for (int kk = 0; kk < kTileBK; ++kk) {
      float a[TM], b[TE];
      const float* xp = xs + kk * BT + ty * TM;
      if constexpr (TM == 4) {
        const float4 v = *reinterpret_cast<const float4*>(xp);
        a[0] = v.x; a[1] = v.y; a[2] = v.z; a[3] = v.w;
      } else if constexpr (TM == 2) {
        const float2 v = *reinterpret_cast<const float2*>(xp);
        a[0] = v.x; a[1] = v.y;
      } else {
#pragma unroll
        for (int i = 0; i < TM; ++i) a[i] = xp[i];
      }
#pragma unroll
      for (int g = 0; g < G; ++g) {
        const float* wp = ws + kk * EP + g * (NTE * V) + tx * V;
        if constexpr (V == 4) {
          const float4 v = *reinterpret_cast<const float4*>(wp);
          b[g * 4 + 0] = v.x; b[g * 4 + 1] = v.y; b[g * 4 + 2] = v.z; b[g * 4 + 3] = v.w;
        } else if constexpr (V == 2) {
          const float2 v = *reinterpret_cast<const float2*>(wp);
          b[g * 2 + 0] = v.x; b[g * 2 + 1] = v.y;
        } else {
          b[g] = wp[0];
        }
      }
#pragma unroll
      for (int i = 0; i < TM; ++i)
#pragma unroll
        for (int j = 0; j < TE; ++j) acc[i][j] = fmaf(a[i], b[j], acc[i][j]);
    }
#pragma unroll
    for (int i = 0; i < TM; ++i)
#pragma unroll
      for (int j = 0; j < TE; ++j) {
        const float y = acc[i][j] - comp[i][j];
        const float s2 = tot[i][j] + y;
        comp[i][j] = (s2 - tot[i][j]) - y;
        tot[i][j] = s2;
      }
  }
  __syncthreads();

  // K-group totals -> shared [KG][BT][EP], added in group order, then the
  // logits tile [BT][EP]
  float* part = tsm;
#pragma unroll
  for (int i = 0; i < TM; ++i)
#pragma unroll
    for (int j = 0; j < TE; ++j) {
      const int e = (j / V) * (NTE * V) + tx * V + (j % V);
      const int r = ty * TM + i;
      part[(kg * BT + r) * EP + e] = tot[i][j];
    }
  __syncthreads();
  for (int q = threadIdx.x; q < BT * EP; q += 256) {
    const int r = q / EP, e = q % EP;
    float sum = part[q];
#pragma unroll
    for (int g = 1; g < KG; ++g) sum += part[g * BT * EP + q];
    float val = -INFINITY;
    if (e < E) val = sum + (bias ? __ldg(bias + e) : 0.f);
    if (logits && e < E && t0 + r < T) logits[static_cast<size_t>(t0 + r) * E + e] = val;
    part[q] = val;   // each q is read and rewritten by the same thread
  }
  __syncthreads();

  // 8 warps select and weigh BT/8 tokens each; lane holds experts lane + 32*j
  constexpr int NJ = (EP + 31) / 32;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
#pragma unroll 1
  for (int r = warp; r < BT; r += 8) {
    const int t = t0 + r;
    if (t >= T) break;
    float v[NJ];
    int id[NJ];
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
      const int e = lane + 32 * j;
      v[j] = (e < EP) ? Ls[r * EP + e] : -INFINITY;
      id[j] = (e < E) ? e : 0x7fffffff;
    }
    if (rs.mode == topk::kRouterSoft) {
      topk::warp_soft_weigh<NJ>(v, id, E, rs, t, topk_idx, topk_w);
      continue;
    }
    if (rs.mode == topk::kRouterGroup) topk::warp_group_limit<NJ>(v, id, E, rs);
    warp_select_and_weigh<NJ>(v, id, rs, t, topk_idx, topk_w);
  }
}

template <typename Tin, int TM, int TE, int NTT, int KG, bool VW>
cudaError_t launch_tiled_v(const Tin* x, const Tin* Wg, const float* bias, int T, int d, int E,
                           RouterSpec rs, int32_t* topk_idx, float* topk_w,
                           float* logits, cudaStream_t s) {
  constexpr int NTE = 256 / KG / NTT;
  constexpr int BT = NTT * TM, EP = NTE * TE;
  constexpr size_t smem_k = static_cast<size_t>(KG) * kTileBK * (BT + EP) * sizeof(float);
  constexpr size_t smem_l = static_cast<size_t>(KG) * BT * EP * sizeof(float);
  constexpr size_t smem = smem_k > smem_l ? smem_k : smem_l;
  static bool attr_set = false;
  if (!attr_set) {
    const cudaError_t e = cudaFuncSetAttribute(route_tiled_kernel<Tin, TM, TE, NTT, KG, VW>,
                                               cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    attr_set = true;
  }
  return launch_pdl(route_tiled_kernel<Tin, TM, TE, NTT, KG, VW>, dim3(ceil_div(T, BT)), dim3(256),
                    smem, s, x, Wg, bias, T, d, E, rs, topk_idx, topk_w, logits);
}

// W_g rows are read as 16-byte vectors only when every row starts 16-byte
// aligned (aligned base and E * sizeof(Tin) a multiple of 16).
template <typename Tin, int TM, int TE, int NTT, int KG = 1>
cudaError_t launch_tiled(const Tin* x, const Tin* Wg, const float* bias, int T, int d, int E,
                         RouterSpec rs, int32_t* topk_idx, float* topk_w,
                         float* logits, cudaStream_t s) {
  const bool vw = (reinterpret_cast<uintptr_t>(Wg) % 16 == 0) &&
                  ((static_cast<size_t>(E) * sizeof(Tin)) % 16 == 0);
  if (vw)
    return launch_tiled_v<Tin, TM, TE, NTT, KG, true>(x, Wg, bias, T, d, E, rs,
                                                      topk_idx, topk_w, logits, s);
  return launch_tiled_v<Tin, TM, TE, NTT, KG, false>(x, Wg, bias, T, d, E, rs,
                                                     topk_idx, topk_w, logits, s);
}

template <typename Tin>
cudaError_t launch_route_t(const Tin* x, const Tin* Wg, const float* bias, int T, int d, int E,
                           RouterSpec rs, int32_t* topk_idx, float* topk_w,
                           float* logits, uint32_t* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  // d >= 1024: the load rounds of the per-thread kernel dominate (on a
  // d = 128 layer the bulk-copy kernel measured slower)
  if (E <= 32 && T < 4096 && d >= 1024) {
    cudaError_t st = cudaSuccess;
    if (try_launch_smem<Tin>(x, Wg, bias, T, d, E, rs, topk_idx, topk_w, logits, err, s, &st))
      return st;
  }
  if (E <= 32 && T >= 4096) {
    // 64 tokens per CTA, K split over 4 groups of 64 threads
    if (E <= 16)
      return launch_tiled<Tin, 4, 4, 16, 4>(x, Wg, bias, T, d, E, rs, topk_idx,
                                            topk_w, logits, s);   // 64 tokens x 16 experts
    return launch_tiled<Tin, 4, 4, 16, 2>(x, Wg, bias, T, d, E, rs, topk_idx,
                                          topk_w, logits, s);     // 64 tokens x 32 experts
  }
  if (E <= 32) {
    const bool vw = (reinterpret_cast<uintptr_t>(Wg) % 16 == 0) &&
                    ((E * static_cast<int>(sizeof(Tin))) % 16 == 0);
    // two tokens per CTA: each W_g row read serves both (measured faster
    // than one token per CTA at T = 1024, d = 4096, E = 8 on GB300)
    const dim3 block(128);
#define MOE_NARROW(NE, TPB, VW)                                                          \
  return launch_pdl(route_narrow_kernel<Tin, NE, TPB, VW>, dim3(ceil_div(T, TPB)), block, 0, s, \
                    x, Wg, bias, T, d, E, rs, topk_idx, topk_w, logits)
#define MOE_NARROW_E(TPB, VW) \
  do {                        \
    if (E <= 8)               \
      MOE_NARROW(8, TPB, VW); \
    else if (E <= 16)         \
      MOE_NARROW(16, TPB, VW);\
    else                      \
      MOE_NARROW(32, TPB, VW);\
  } while (0)
    if (vw)
      MOE_NARROW_E(2, true);
    else
      MOE_NARROW_E(2, false);
#undef MOE_NARROW_E
#undef MOE_NARROW
  } else if (E <= 64) {
    return launch_tiled<Tin, 4, 2, 8>(x, Wg, bias, T, d, E, rs, topk_idx, topk_w,
                                      logits, s);   // 32 tokens x 64 experts
  } else if (E <= 128) {
    return launch_tiled<Tin, 4, 4, 8>(x, Wg, bias, T, d, E, rs, topk_idx, topk_w,
                                      logits, s);   // 32 tokens x 128 experts
  } else {
    return launch_tiled<Tin, 4, 8, 8>(x, Wg, bias, T, d, E, rs, topk_idx, topk_w,
                                      logits, s);   // 32 tokens x 256 experts
  }
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_route(int dtype, const void* x, const void* Wg, const float* bias, int T,
                         int d, int E, RouterSpec rs, int32_t* topk_idx,
                         float* topk_w, float* logits, uint32_t* err, cudaStream_t s) {
  // tensor-core gate: always for E a multiple of 64; for narrower gates only
  // with enough 128-token CTAs to fill the GPU (the SIMT kernels win on small
  // batches, e.g. T = 1024)
  if (T > 0 && gate_tc_supported(dtype, E, Wg, x) && (E % 64 == 0 || T >= 4096))
    return launch_gate_tc(x, Wg, bias, T, d, E, rs, topk_idx, topk_w, logits, err,
                          s);
  if (dtype == 0)
    return launch_route_t<float>(static_cast<const float*>(x), static_cast<const float*>(Wg),
                                 bias, T, d, E, rs, topk_idx, topk_w, logits, err, s);
  return launch_route_t<__nv_bfloat16>(static_cast<const __nv_bfloat16*>(x),
                                       static_cast<const __nv_bfloat16*>(Wg), bias, T, d, E, rs,
                                       topk_idx, topk_w, logits, err, s);
}

}  // namespace moe
