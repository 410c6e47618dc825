// gate_tc.cu - gate projection and router on the tensor cores, for bf16
// layers with E a multiple of 8 up to 256 (DeepSeek-V4 EP article, sections
// 2.1 and 3.2): L = x W_g + b, then the same warp top-k and weights as
// route.cu. The weight tile is Ep = E rounded up to 64 experts wide; TMA
// zero-fills the columns past E and the padded logits are never read.
//
// The gate is a GEMM of T x d by d x E (60 GFLOP for 16384 tokens, d = 7168,
// E = 256), too much for fp32 FMA, but fp32 accumulation inside tcgen05 over
// K = 7168 drifts up to 4e-5 from fp64 (measured on GB300), past the 1e-5
// logit / 1e-6 weight bounds. So the MMA accumulator restarts every 128 K
// (two 64-wide k-blocks) and the CUDA cores add each 128-long partial into
// fp32 totals: measured error then 1.7e-6 max, 1.8e-7 RMS at K = 7168.
//
// CTA = 128 tokens x Ep experts (tcgen05.mma.cta_group::1 M128 N=Ep K16), one
// CTA per 128 tokens:
//   warp 0     TMA producer: x [128 tokens][64 k] (K-major) and W_g
//              [64 k][E] as E/64 boxes of 64 experts (MN-major), 128-byte
//              swizzle, a 192 KB ring of 4 (E = 256) to 8 (E = 64) stages
//   warp 1     TMEM allocation + MMA issue; commits a chunk to one of
//              min(8, 512 / E) E-column accumulators
//   warps 2-9  epilogue: warp (half, q) adds TMEM lanes 32q..32q+31, columns
//              of its half, into register totals after every chunk
// then all warps meet, write logits (+ bias) to shared memory over the ring,
// and one thread per token selects and weighs it. Every wait is bounded.
#include <cfloat>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "topk.cuh"

namespace moe {

namespace {

using namespace ptx;

constexpr int BM = 128, BK = 64, CHUNK_KB = 2;
constexpr int X_BYTES = BM * BK * 2;     // 16 KB
constexpr int BOX_BYTES = BK * 64 * 2;   // 8 KB: [64 k][64 experts]
constexpr int MAX_E = 256;
// The stage ring is 192 KB: 4 stages of 48 KB at E = 256, up to 8 stages
// of 24 KB at E = 64 (a stage is x [128][64] plus E/64 weight boxes).
constexpr int RING_BYTES = 4 * (X_BYTES + (MAX_E / 64) * BOX_BYTES);
constexpr int MAX_STAGES = 8;
constexpr int NUM_EPI_WARPS = 8;
constexpr int NUM_THREADS = 64 + 32 * NUM_EPI_WARPS;
constexpr int OFF_BAR = RING_BYTES;
constexpr int MAX_ACC = 8;                    // TMEM accumulators (512 / E of them)
constexpr int NUM_BARS = 2 * MAX_STAGES + 2 * MAX_ACC + 1;  // full, empty, tfull, tempty, drain
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;
// The logits tile is [BM][E + 1] (padded: row-strided writes hit distinct banks).
static_assert(BM * (MAX_E + 1) * 4 <= OFF_BAR, "logits tile must fit over the stage ring");

// EMAX (64, 128 or 256) bounds E: the epilogue keeps EMAX/2 totals per
// thread.
template <int EMAX>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    gate_tc_kernel(const __grid_constant__ CUtensorMap tmX, const __grid_constant__ CUtensorMap tmW,
                   const float* __restrict__ bias, int T, int d, int E, RouterSpec rs,
                   int32_t* __restrict__ topk_idx, float* __restrict__ topk_w,
                   float* __restrict__ logits, uint32_t* __restrict__ err, int ksplit) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + OFF_BAR);
  uint64_t* empty = full + MAX_STAGES;
  uint64_t* tfull = empty + MAX_STAGES;
  uint64_t* tempty = tfull + MAX_ACC;
  uint64_t* drain = tempty + MAX_ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  float* Ls = reinterpret_cast<float*>(smem);  // [BM][E + 1] after the main loop

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  // ksplit = 2: a cluster of two CTAs shares the 128-token tile, CTA `part`
  // accumulating k-blocks [part * KB/2, ...) of d; the partial logits are
  // added through distributed shared memory and each CTA routes 64 tokens
  const int part = ksplit == 2 ? static_cast<int>(cluster_ctarank()) : 0;
  const int t0 = (blockIdx.x / ksplit) * BM;
  // the weight tile is Ep = E rounded up to 64 experts wide: TMA zero-fills
  // the boxes past E, and the padded columns are never read back
  const int Ep = (E + 63) & ~63;
  const int nwbox = Ep / 64;
  const uint32_t stage_bytes = static_cast<uint32_t>(X_BYTES + nwbox * BOX_BYTES);
  const int nst = min(MAX_STAGES, RING_BYTES / static_cast<int>(stage_bytes));
  const int KB_all = d / BK;
  const int kb0 = part == 0 ? 0 : KB_all / 2;
  const int KB = (ksplit == 2 && part == 0) ? KB_all / 2 : KB_all - kb0;  // this CTA's k-blocks
  const int nchunk = (KB + CHUNK_KB - 1) / CHUNK_KB;
  // TMEM: 512 columns (one CTA per SM) as 512 / E accumulators of E columns,
  // so the MMA runs up to that many 128-K chunks ahead of the epilogue
  constexpr int HALF = EMAX / 2;
  const uint32_t tmem_cols = 512u;
  const int nacc = min(MAX_ACC, 512 / Ep);

  if (warp == 0 && lane == 0) {
    for (int i = 0; i < MAX_STAGES; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    for (int i = 0; i < MAX_ACC; ++i) {
      mbar_init(&tfull[i], 1);
      mbar_init(&tempty[i], NUM_EPI_WARPS);
    }
    mbar_init(drain, 1);
    fence_mbar_init();
  } else if (warp == 1) {
    tmem_alloc(tmem_slot, tmem_cols);
    tmem_relinquish();
  }
  __syncthreads();
  tc_fence_after();
  // barriers and tensor memory are set up: from here on global memory
  pdl_wait();
  pdl_trigger();
  const uint32_t tmem_base = *tmem_slot;
  bool timed_out = false;

  float tot[HALF];
#pragma unroll
  for (int j = 0; j < HALF; ++j) tot[j] = 0.f;

  if (warp == 0) {
    if (lane == 0) {
      prefetch_tmap(&tmX);
      prefetch_tmap(&tmW);
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      for (int kb = 0; kb < KB; ++kb) {
        if (!mbar_wait_spin(&empty[s], ph ^ 1u, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        uint8_t* st = smem + s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], stage_bytes);
        tma_load_2d(st, &tmX, &full[s], (kb0 + kb) * BK, t0);
        for (int c = 0; c < nwbox; ++c)
          tma_load_2d(st + X_BYTES + c * BOX_BYTES, &tmW, &full[s], c * 64, (kb0 + kb) * BK);
        armed |= 1u << s;
        armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
        if (++s == nst) {
          s = 0;
          ph ^= 1u;
        }
      }
      for (int i = 0; i < nst; ++i)
        if ((armed >> i) & 1u)
          if (!mbar_wait(&full[i], (armed_ph >> i) & 1u, kWaitLimitNs)) timed_out = true;
    }
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = make_idesc_bf16_f32(BM, Ep, /*A MN*/ false, /*B MN*/ true);
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool issued = false;
      for (int c = 0; c < nchunk && !timed_out; ++c) {
        if (!mbar_wait_spin(&tempty[acc], aph ^ 1u, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * Ep);
        const int kb_end = min(KB, (c + 1) * CHUNK_KB);
        for (int kb = c * CHUNK_KB; kb < kb_end; ++kb) {
          if (!mbar_wait_spin(&full[s], ph, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          tc_fence_after();
          const uint32_t a_base = smem_u32(smem + s * stage_bytes);
          const uint32_t b_base = a_base + X_BYTES;
#pragma unroll
          for (int kk = 0; kk < BK / 16; ++kk)
            tc_mma_f16(d_tmem, make_sdesc_sw128(a_base + kk * 32, 16, 1024),
                       make_sdesc_sw128(b_base + kk * 2048, BOX_BYTES, 1024), idesc,
                       (kb != c * CHUNK_KB || kk != 0) ? 1u : 0u);
          issued = true;
          tc_commit(&empty[s]);
          if (++s == nst) {
            s = 0;
            ph ^= 1u;
          }
        }
        if (timed_out) break;
        tc_commit(&tfull[acc]);
        if (++acc == nacc) {
          acc = 0;
          aph ^= 1u;
        }
      }
      if (timed_out && issued) {  // MMAs in flight finish before TMEM is freed
        tc_commit(drain);
        mbar_wait(drain, 0, kWaitLimitNs);
      }
    }
  } else {
    // epilogue: columns [half * Ep/2, half * Ep/2 + Ep/2) of lanes 32q..32q+31
    const int q = warp & 3;
    const int half = (warp - 2) >> 2;
    const int ncol = Ep / 2;
    int acc = 0;
    uint32_t aph = 0;
    for (int c = 0; c < nchunk; ++c) {
      const bool ok = mbar_wait(&tfull[acc], aph, kWaitLimitNs);
      if (!__all_sync(0xffffffffu, ok)) {
        timed_out = true;
        break;
      }
      tc_fence_after();
      const uint32_t tb = tmem_base + static_cast<uint32_t>(acc * Ep + half * ncol) +
                          (static_cast<uint32_t>(q * 32) << 16);
#pragma unroll
      for (int cc = 0; cc < HALF / 32; ++cc) {
        if (cc * 32 < ncol) {
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + cc * 32, v);
          tmem_ld_wait();
#pragma unroll
          for (int j = 0; j < 32; ++j) tot[cc * 32 + j] += __uint_as_float(v[j]);
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&tempty[acc]);
      if (++acc == nacc) {
        acc = 0;
        aph ^= 1u;
      }
    }
  }

  if (timed_out && err != nullptr) atomicOr(err, kErrTimeout);
  __syncthreads();  // the ring is idle: reuse it for the logits tile
  // ksplit = 2: CTA `part` finishes rows [64 part, 64 part + 64); its partial
  // sums of the other half go straight into the peer's tile at row r ^ 64
  // (the rows the peer does not finish itself) with remote stores
  const uint32_t peer_ls =
      ksplit == 2 ? mapa_shared(smem_u32(Ls), static_cast<uint32_t>(part ^ 1)) : 0u;
  if (warp >= 2) {
    const int q = warp & 3, half = (warp - 2) >> 2, ncol = Ep / 2;
    const int r = q * 32 + lane;
    const bool own_row = (r / (BM / 2)) == part;
#pragma unroll
    for (int j = 0; j < HALF; ++j) {
      if (j < ncol && half * ncol + j < E) {
        const int e = half * ncol + j;
        if (ksplit == 2) {
          if (own_row)
            Ls[r * (E + 1) + e] = tot[j];  // this CTA's partial sum
          else
            st_shared_cluster_s32(peer_ls + static_cast<uint32_t>(((r ^ (BM / 2)) * (E + 1) + e) * 4),
                                  __float_as_int(tot[j]));
        } else {
          const float val = tot[j] + (bias ? __ldg(bias + e) : 0.f);
          Ls[r * (E + 1) + e] = val;
          if (logits && t0 + r < T) logits[static_cast<size_t>(t0 + r) * E + e] = val;
        }
      }
    }
  }
  if (ksplit == 2) {
    // the barrier makes the peer's remote stores visible (and none is in
    // flight past it); rows [64 part, 64 part + 64) then add the two
    // partials (P0 + P1 is the same sum either way round) and the bias from
    // local shared memory
    cluster_sync();
    for (int i = threadIdx.x; i < (BM / 2) * E; i += NUM_THREADS) {
      const int r = (BM / 2) * part + i / E, e = i - (i / E) * E;
      const int o = r * (E + 1) + e;
      const float val = (Ls[o] + Ls[(r ^ (BM / 2)) * (E + 1) + e]) + (bias ? __ldg(bias + e) : 0.f);
      Ls[o] = val;
      if (logits && t0 + r < T) logits[static_cast<size_t>(t0 + r) * E + e] = val;
    }
    __syncthreads();
  } else {
    __syncthreads();
  }
  // selection and weights from the logits rows in shared memory (stride
  // E + 1): hard top-k with two threads per token, four with the K split
  // (each a share of the experts, lists merged: the serial insertion scan
  // over E was ~40 % of the kernel at E = 64, measured); group-limited and
  // soft routers one thread per token
  const int r_lo = ksplit == 2 ? (BM / 2) * part : 0;
  const int nrows = BM / ksplit;
  if (rs.mode == topk::kRouterRenorm || rs.mode == topk::kRouterPrek) {
    // 256 threads: two per token for 128 rows, four for the 64 of a split
    if (threadIdx.x < 256) {
      if (ksplit == 2) {
        const int r = r_lo + (threadIdx.x >> 2);
        topk::group_select_and_weigh<4>(Ls + r * (E + 1), E, rs, t0 + r, threadIdx.x & 3,
                                        t0 + r < T, topk_idx, topk_w);
      } else {
        const int r = r_lo + (threadIdx.x >> 1);
        topk::group_select_and_weigh<2>(Ls + r * (E + 1), E, rs, t0 + r, threadIdx.x & 1,
                                        t0 + r < T, topk_idx, topk_w);
      }
    }
  } else if (threadIdx.x < nrows) {
    const int r = r_lo + threadIdx.x;
    if (t0 + r < T) {
      if (rs.mode == topk::kRouterSoft)
        topk::thread_soft_weigh(Ls + r * (E + 1), E, rs, t0 + r, topk_idx, topk_w);
      else
        topk::thread_select_and_weigh(Ls + r * (E + 1), E, rs, t0 + r, topk_idx, topk_w);
    }
  }
  __syncthreads();
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem_base, tmem_cols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 g_enc = nullptr;
std::once_flag g_enc_once;

bool map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
            uint32_t box_rows) {
  std::call_once(g_enc_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_enc = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  if (!g_enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  return g_enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides,
               box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// K is split across a CTA pair when two CTAs per 128-token tile still fit in
// one wave and each half has at least two k-blocks (GB300, T = 8192, d =
// 2048, E = 64: 64 CTAs left 88 SMs idle).
int gate_ksplit(int T, int d) {
  static int sms = 0;
  if (sms == 0) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      sms = 1;
  }
  return (2 * ceil_div(T, BM) <= sms && d / BK >= 4) ? 2 : 1;
}

template <int EMAX>
cudaError_t launch_emax(const CUtensorMap& mx, const CUtensorMap& mw, const float* bias, int T,
                        int d, int E, RouterSpec rs, int32_t* idx, float* w,
                        float* logits, uint32_t* err, cudaStream_t s) {
  static std::once_flag once;
  static cudaError_t st = cudaSuccess;
  std::call_once(once, [] {
    st = cudaFuncSetAttribute(gate_tc_kernel<EMAX>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                              SMEM_BYTES);
  });
  if (st != cudaSuccess) return st;
  const int ksplit = gate_ksplit(T, d);
  cudaLaunchConfig_t lc = {};
  lc.gridDim = dim3(ceil_div(T, BM) * ksplit);
  lc.blockDim = dim3(NUM_THREADS);
  lc.dynamicSmemBytes = SMEM_BYTES;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = static_cast<unsigned>(ksplit);
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  return cudaLaunchKernelEx(&lc, gate_tc_kernel<EMAX>, mx, mw, bias, T, d, E, rs, idx, w, logits,
                            err, ksplit);
}

}  // namespace

bool gate_tc_supported(int dtype, int E, const void* Wg, const void* x) {
  // E % 8 == 0: a W_g row is a whole number of 16-byte units (TMA stride)
  return dtype == 1 && E >= 8 && E <= MAX_E && E % 8 == 0 &&
         reinterpret_cast<uintptr_t>(Wg) % 16 == 0 && reinterpret_cast<uintptr_t>(x) % 16 == 0;
}

cudaError_t launch_gate_tc(const void* x, const void* Wg, const float* bias, int T, int d, int E,
                           RouterSpec rs, int32_t* topk_idx, float* topk_w,
                           float* logits, uint32_t* err, cudaStream_t s) {
  if (T == 0) return cudaSuccess;
  CUtensorMap mx, mw;
  std::memset(&mx, 0, sizeof(mx));
  std::memset(&mw, 0, sizeof(mw));
  if (!map_2d(&mx, x, static_cast<uint64_t>(T), static_cast<uint64_t>(d), 64, BM))
    return cudaErrorInvalidValue;
  if (!map_2d(&mw, Wg, static_cast<uint64_t>(d), static_cast<uint64_t>(E), 64, BK))
    return cudaErrorInvalidValue;
  if (E <= 64)
    return launch_emax<64>(mx, mw, bias, T, d, E, rs, topk_idx, topk_w, logits,
                           err, s);
  if (E <= 128)
    return launch_emax<128>(mx, mw, bias, T, d, E, rs, topk_idx, topk_w, logits,
                            err, s);
  return launch_emax<256>(mx, mw, bias, T, d, E, rs, topk_idx, topk_w, logits,
                          err, s);
}

}  // namespace moe
