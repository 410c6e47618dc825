// wgrad_tc.cu - the experts' weight gradients on the sm_103a tensor cores
// (tcgen05 + TMEM, 2-SM pair mode, fed by TMA). In backpropagation the
// gradient reaches only the activated experts (DeepSeek-V4 EP article,
// section 2.1), so each expert's weight gradient is a sum over the rows
// routed to it:
//
//   dW[e][m][n] = sum over r in [offsets[e], offsets[e+1]) of A[a(r)][m] * dB[r][n]
//
// with A the rows' bf16 activations (the dispatched tokens for dW1, the
// layer input for the gate's dW_g; a(r) = r, or r - offsets[e] when every
// expert reads the same rows) and dB their fp32 output gradient, held as
// two bf16 parts dB = hi + lo ([R][2N]: columns [0, N) hi, [N, 2N) lo; hi +
// lo carries dB to ~2^-17 relative). Or the other way round (split A): for
// dW2 = sum_r (w_r H_r)^T dout_r the fp32 operand is A' = w H, split into
// [R][2M], and B the bf16 dout rows (per routed row; or dout itself, b(r) =
// r - offsets[e], when every expert reads the same rows). Both parts go
// through the tensor cores into one fp32 accumulator, so the result has the
// accuracy of an fp32 operand. Output fp32 [E][M][N]; an expert with no rows
// gets zeros.
//
// Tiles: 256 output rows (m) x 256 output columns (n) of one expert, computed
// by a cluster of two CTAs (one per SM of an SM pair) with one
// tcgen05.mma.cta_group::2 M256 N256 K16 per k-step and operand part, issued
// by the even CTA. CTA r stages only rows m0 + 128 r .. +127 of A and
// columns n0 + 128 r .. +127 of B, each operand's split one twice (hi and
// lo), and its tensor memory receives
// its 128 output rows; per SM this is half the shared-memory traffic per flop
// of a one-CTA 128 x 128 tile (measured bound by that traffic). The
// contraction runs over the expert's rows in blocks of 64 (ragged: the last
// block holds n_e mod 64 rows). Both operands are read MN-major straight
// from their row-major storage: a TMA box [64 rows][64 columns] (128-byte
// swizzle) is 64 contraction rows of 64 consecutive m (or n), so the
// transposes cost nothing. Per block and CTA: A 16 KB, hi 16 KB, lo 16 KB.
//
// A block whose valid rows are a whole number of 16-row k-steps (every block
// but an expert's last, and that one when its row count is a multiple of
// 16) needs nothing done to it: both CTAs' loads complete directly on the
// even CTA's full barrier (the pair form of the TMA load), which the even
// CTA's producer arms for both CTAs' bytes. In an expert's last block
// otherwise, rows of its last k-step past the expert's end are whatever
// follows in memory (the next expert's rows, or the TMA's zero fill past
// the matrix): each CTA's loads then land on its own barrier, a forwarder
// warp overwrites those rows with zeros in the staged tiles (row j of a box
// is its 128-byte line j; the swizzle permutes within the line) and
// releases the stage to the MMA: the even CTA's by an arrive on the full
// barrier, the odd CTA's by a 16-byte bulk copy into the even CTA whose
// completion is counted on that barrier (a cluster-scope release arrive per
// stage measured far slower in the FP8 prologue of the forward GEMM).
// k-steps wholly past the end are skipped.
//
// Schedule: a persistent grid of as many clusters as fit at once walks the
// tiles (expert, m block, n block) with a stride of the cluster count; every
// expert has the same tile count and the tiles of one expert are adjacent,
// so the clusters running side by side share its operand rows through L2.
// Warp roles: warp 0 TMA producer (4-stage ring of 48 KB), warp 1 TMEM
// allocation (both CTAs) and MMA issue (even CTA), warp 2 forwarder, warps
// 3-6 epilogue (tcgen05.ld of their TMEM lane quadrant, 32 x 32 fp32 blocks
// staged in shared memory, two buffers a warp, written by TMA stores clipped
// at the matrix edge). Two 256-column accumulators let a tile's epilogue
// overlap the next tile's main loop. Every wait is bounded; a timeout sets
// kErrTimeout, drains the copies and MMAs in flight, frees TMEM and exits.
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cuda_bf16.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

using namespace ptx;

namespace wg {
constexpr int BM = 256, BN = 256, BK = 64;  // pair tile; a CTA holds half of M and of N
constexpr int BOX_BYTES = BK * 64 * 2;      // [64 rows][64 columns] bf16
constexpr int HALF_BYTES = 2 * BOX_BYTES;   // this CTA's 128 m (or n) x 64 rows
constexpr int STAGES = 4;
constexpr int STAGE_BYTES = 3 * HALF_BYTES;  // A, hi, lo
constexpr int NUM_ACC = 2;
constexpr int ACC_COLS = BN;
constexpr int TMEM_COLS = NUM_ACC * ACC_COLS;
constexpr int NUM_EPI = 4;
constexpr int EPI_WARP0 = 3;
constexpr int THREADS = 32 * (EPI_WARP0 + NUM_EPI);
constexpr int STG_BYTES = 32 * 32 * 4;  // one 32 x 32 fp32 block; two per epilogue warp
constexpr int OFF_STG = STAGES * STAGE_BYTES;
constexpr int OFF_BAR = OFF_STG + NUM_EPI * 2 * STG_BYTES;
// lfull, full, empty, tfull, tempty, drain
constexpr int NUM_BARS = 3 * STAGES + 2 * NUM_ACC + 1;
constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
constexpr int OFF_SINK = (OFF_MISC + 16 + 15) & ~15;  // 16 bytes the odd CTA's releases copy
constexpr int OFF_SEG = OFF_SINK + 16;
constexpr int SMEM_BYTES = OFF_SEG + (kMaxExperts + 1) * 4 + 1024;
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
// M256 N256 (pair), A and B both MN-major
constexpr uint32_t IDESC = make_idesc_bf16_f32(BM, BN, true, true);

struct Params {
  const int32_t* offsets;
  uint32_t* err;
  int E, M, N, R;
  int a_shared;
  int b_shared;  // B row of routed row r: r - offsets[e] (split A only)
  int tiles_m, tiles_n, total;
};

struct Tile {
  int e, m0, n0;
};

__device__ __forceinline__ Tile decode(int t, const Params& p) {
  const int per = p.tiles_m * p.tiles_n;
  Tile r;
  r.e = t / per;
  const int l = t - r.e * per;
  const int mb = l / p.tiles_n;
  r.m0 = mb * BM;
  r.n0 = (l - mb * p.tiles_n) * BN;
  return r;
}

// A block that goes through the forwarder: its last k-step holds rows past
// the expert's end.
__device__ __forceinline__ bool needs_zeroing(int n, int kb) {
  return (min(BK, n - kb * BK) & 15) != 0;
}

// Ring position over the k-blocks of a CTA's tiles (every role walks the
// same sequence).
struct Ring {
  int s = 0;
  uint32_t ph = 0;
  __device__ __forceinline__ void next() {
    if (++s == STAGES) {
      s = 0;
      ph ^= 1u;
    }
  }
};
}  // namespace wg

// SPLIT_A: A is the split operand ([R][2M]) and B single ([rows][N]);
// otherwise A single ([rows][M]) and B split ([R][2N])
template <bool SPLIT_A>
__global__ void __launch_bounds__(wg::THREADS, 1)
    wgrad_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                      const __grid_constant__ CUtensorMap tmB,
                      const __grid_constant__ CUtensorMap tmY, const wg::Params p) {
  using namespace wg;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint64_t* lfull = reinterpret_cast<uint64_t*>(smem + OFF_BAR);  // this CTA's loads landed
  uint64_t* full = lfull + STAGES;     // even CTA: both CTAs' stages released
  uint64_t* empty = full + STAGES;     // both CTAs, from one multicast commit
  uint64_t* tfull = empty + STAGES;    // both CTAs, multicast commit
  uint64_t* tempty = tfull + NUM_ACC;  // even CTA: every epilogue warp of both CTAs
  uint64_t* drain = tempty + NUM_ACC;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + OFF_MISC);
  int* s_ok = reinterpret_cast<int*>(smem + OFF_MISC + 4);
  int* seg = reinterpret_cast<int*>(smem + OFF_SEG);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int cl = static_cast<int>(blockIdx.x >> 1), ncl = static_cast<int>(gridDim.x >> 1);
  const int E = p.E;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    for (int e = lane; e <= E; e += 32) seg[e] = __ldg(p.offsets + e);
    __syncwarp();
    bool bad = false;
    for (int e = lane; e < E; e += 32) {
      const int lo = seg[e], hi = seg[e + 1];
      bad |= lo < 0 || hi < lo || hi > p.R;
    }
    bad = __any_sync(0xffffffffu, bad);
    if (lane == 0) {
      // segments out of range: every expert is taken as empty (zeros out)
      *s_ok = bad ? 0 : 1;
      if (bad && blockIdx.x == 0) atomicOr(p.err, kErrBadIndex);
      for (int i = 0; i < STAGES; ++i) {
        mbar_init(&lfull[i], 1);
        mbar_init(&full[i], 1);
        mbar_init(&empty[i], 1);
      }
      for (int i = 0; i < NUM_ACC; ++i) {
        mbar_init(&tfull[i], 1);
        mbar_init(&tempty[i], 2 * NUM_EPI);
      }
      mbar_init(drain, 1);
      fence_mbar_init();
    }
  } else if (warp == 1) {
    tmem_alloc_pair(tmem_slot, TMEM_COLS);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const bool seg_ok = *s_ok != 0;
  auto rows_of = [&](int e) { return seg_ok ? seg[e + 1] - seg[e] : 0; };
  bool timed_out = false;

  if (warp == 0) {
    // -------------------------------------------------------------- TMA producer (both CTAs)
    if (lane == 0) {
      prefetch_tmap(&tmA);
      prefetch_tmap(&tmB);
      Ring rg;
      const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
      // lfull[s] completes once per forwarded block in stage s: its phase
      // parity per stage, and the parity of the last such use to drain
      uint32_t lph = 0, larmed = 0, larmed_ph = 0;
      // 64-wide boxes of CTA r's halves that start inside the matrix (M a
      // multiple of 64); the MMA's rows / columns from a skipped box, or
      // from a box's part past N, are never stored
      auto boxes_a = [&](const Tile& tl, int r) {
        const int mh = tl.m0 + r * 128;
        return mh < p.M ? min(2, (p.M - mh) / 64) : 0;
      };
      auto boxes_b = [&](const Tile& tl, int r) {
        const int nh = tl.n0 + r * 128;
        return nh < p.N ? min(2, (p.N - nh + 63) / 64) : 0;
      };
      for (int t = cl; t < p.total && !timed_out; t += ncl) {
        const Tile tl = decode(t, p);
        const int n = rows_of(tl.e);
        if (n == 0) continue;
        const int lo = seg[tl.e];
        const int a0 = p.a_shared ? 0 : lo;
        const int b0 = p.b_shared ? 0 : lo;
        const int mh = tl.m0 + static_cast<int>(rank) * 128;
        const int nh = tl.n0 + static_cast<int>(rank) * 128;
        const int na = boxes_a(tl, static_cast<int>(rank));
        const int nb = boxes_b(tl, static_cast<int>(rank));
        // the split operand's boxes count twice
        auto cta_bytes = [&](int a, int b) {
          return static_cast<uint32_t>((SPLIT_A ? 2 * a + b : a + 2 * b) * BOX_BYTES);
        };
        const uint32_t bytes = cta_bytes(na, nb);
        // both CTAs' bytes, counted on the even CTA's full barrier
        const uint32_t pair_bytes =
            cta_bytes(boxes_a(tl, 0), boxes_b(tl, 0)) + cta_bytes(boxes_a(tl, 1), boxes_b(tl, 1));
        // stage slots: A (or A hi) | B (or B hi) | the split operand's lo
        auto load_stage = [&](uint8_t* st, int kb, auto load) {
          for (int c = 0; c < na; ++c) load(st + c * BOX_BYTES, &tmA, mh + c * 64, a0 + kb * BK);
          for (int c = 0; c < nb; ++c)
            load(st + HALF_BYTES + c * BOX_BYTES, &tmB, nh + c * 64, b0 + kb * BK);
          if constexpr (SPLIT_A) {
            for (int c = 0; c < na; ++c)
              load(st + 2 * HALF_BYTES + c * BOX_BYTES, &tmA, p.M + mh + c * 64, a0 + kb * BK);
          } else {
            for (int c = 0; c < nb; ++c)
              load(st + 2 * HALF_BYTES + c * BOX_BYTES, &tmB, p.N + nh + c * 64, b0 + kb * BK);
          }
        };
        const int nkb = (n + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          if (!mbar_wait_spin(&empty[rg.s], rg.ph ^ 1u, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          uint8_t* st = smem + rg.s * STAGE_BYTES;
          if (needs_zeroing(n, kb)) {
            uint64_t* bar = &lfull[rg.s];
            mbar_arrive_expect_tx(bar, bytes);
            load_stage(st, kb, [&](uint8_t* dst, const CUtensorMap* m, int c0, int c1) {
              tma_load_2d(dst, m, bar, c0, c1);
            });
            larmed |= 1u << rg.s;
            larmed_ph = (larmed_ph & ~(1u << rg.s)) | (lph & (1u << rg.s));
            lph ^= 1u << rg.s;
          } else {
            if (rank == 0) mbar_arrive_expect_tx(&full[rg.s], pair_bytes);
            const uint32_t bar = leader_full + static_cast<uint32_t>(rg.s * 8);
            load_stage(st, kb, [&](uint8_t* dst, const CUtensorMap* m, int c0, int c1) {
              tma_load_2d_pair(dst, m, bar, c0, c1);
            });
          }
          rg.next();
        }
      }
      // no copy may still be landing when the CTA exits (the direct ones are
      // counted on the even CTA's full barriers, which its forwarder drains)
      for (int i = 0; i < STAGES; ++i)
        if ((larmed >> i) & 1u)
          if (!mbar_wait_spin(&lfull[i], (larmed_ph >> i) & 1u, kWaitLimitNs)) timed_out = true;
    }
  } else if (warp == 1) {
    if (rank == 0) {
      // ------------------------------------------------------------ MMA issue (even CTA, whole warp waits)
      Ring rg;
      int acc = 0;
      uint32_t aph = 0;
      bool issued = false;
      for (int t = cl; t < p.total; t += ncl) {
        const Tile tl = decode(t, p);
        const int n = rows_of(tl.e);
        if (n == 0) continue;
        if (!__all_sync(0xffffffffu, mbar_wait_spin(&tempty[acc], aph ^ 1u, kWaitLimitNs))) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * ACC_COLS);
        const int nkb = (n + BK - 1) / BK;
        for (int kb = 0; kb < nkb; ++kb) {
          // both CTAs' bytes landed (direct), or released by both CTAs'
          // forwarders (the odd one's bytes at cluster scope)
          if (!__all_sync(0xffffffffu,
                          mbar_wait_spin_cluster(&full[rg.s], rg.ph, kWaitLimitNs))) {
            timed_out = true;
            break;
          }
          if (lane == 0) {
            tc_fence_after();
            const int ksteps = (min(BK, n - kb * BK) + 15) / 16;
            const uint32_t a_base = smem_u32(smem + rg.s * STAGE_BYTES);
            const uint32_t b_base = a_base + HALF_BYTES, l_base = a_base + 2 * HALF_BYTES;
            for (int kk = 0; kk < ksteps; ++kk) {
              const uint64_t ad = make_sdesc_sw128(a_base + kk * 2048, BOX_BYTES, 1024);
              const uint64_t bd = make_sdesc_sw128(b_base + kk * 2048, BOX_BYTES, 1024);
              const uint64_t ld = make_sdesc_sw128(l_base + kk * 2048, BOX_BYTES, 1024);
              // (A hi or A) x (B or B hi), then the lo part against the other
              tc_mma_f16_pair(d_tmem, ad, bd, IDESC, (kb | kk) != 0 ? 1u : 0u);
              if constexpr (SPLIT_A)
                tc_mma_f16_pair(d_tmem, ld, bd, IDESC, 1u);
              else
                tc_mma_f16_pair(d_tmem, ad, ld, IDESC, 1u);
            }
            tc_commit_pair_mc(&empty[rg.s], 0x3);
          }
          __syncwarp();
          issued = true;
          rg.next();
        }
        if (timed_out) break;
        if (lane == 0) tc_commit_pair_mc(&tfull[acc], 0x3);
        __syncwarp();
        if (++acc == NUM_ACC) {
          acc = 0;
          aph ^= 1u;
        }
      }
      if (timed_out && issued) {
        // the MMAs in flight finish before TMEM is freed
        if (lane == 0) tc_commit_pair_mc(drain, 0x1);
        __syncwarp();
        mbar_wait_spin(drain, 0, kWaitLimitNs);
      }
    }
  } else if (warp == 2) {
    // -------------------------------------------------------------- forwarder (both CTAs)
    const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
    const uint32_t leader_sink = mapa_shared(smem_u32(smem + OFF_SINK), 0);
    const uint32_t my_sink = smem_u32(smem + OFF_SINK);
    Ring rg;
    uint32_t armed = 0, armed_ph = 0;
    uint32_t lph = 0;  // lfull's phase parity per stage (forwarded blocks only)
    for (int t = cl; t < p.total && !timed_out; t += ncl) {
      const Tile tl = decode(t, p);
      const int n = rows_of(tl.e);
      if (n == 0) continue;
      const int nkb = (n + BK - 1) / BK;
      for (int kb = 0; kb < nkb; ++kb) {
        armed |= 1u << rg.s;
        armed_ph = (armed_ph & ~(1u << rg.s)) | (rg.ph << rg.s);
        if (!needs_zeroing(n, kb)) {  // loaded straight onto the even CTA's full barrier
          rg.next();
          continue;
        }
        const uint32_t want = (lph >> rg.s) & 1u;
        lph ^= 1u << rg.s;
        if (!__all_sync(0xffffffffu, mbar_wait_spin(&lfull[rg.s], want, kWaitLimitNs))) {
          timed_out = true;
          break;
        }
        const int valid = min(BK, n - kb * BK);
        const int ksteps = (valid + 15) / 16;
        if (valid & 15) {
          // rows [valid, 16 ksteps) of the last k-step belong to no row of
          // this expert: zeros in this CTA's six boxes
          uint8_t* st = smem + rg.s * STAGE_BYTES;
          const int z0 = valid * 128, per_box = (ksteps * 16 - valid) * 8;
          for (int i = lane; i < 6 * per_box; i += 32) {
            const int b = i / per_box, j = i - b * per_box;
            *reinterpret_cast<uint4*>(st + b * BOX_BYTES + z0 + j * 16) = make_uint4(0, 0, 0, 0);
          }
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive_expect_tx(&full[rg.s], 16u);  // + the odd CTA's 16 bytes
          else
            bulk_copy_s2cluster(leader_sink, my_sink, 16u,
                                leader_full + static_cast<uint32_t>(rg.s * 8));
        }
        rg.next();
      }
    }
    // even CTA: every stage's bytes (both CTAs' direct loads, the odd CTA's
    // release copies) have landed before either CTA exits
    if (rank == 0)
      for (int i = 0; i < STAGES; ++i)
        if ((armed >> i) & 1u)
          if (!mbar_wait_spin_cluster(&full[i], (armed_ph >> i) & 1u, kWaitLimitNs))
            timed_out = true;
  } else {
    // -------------------------------------------------------------- epilogue (both CTAs)
    // warp w reads TMEM lanes 32 (w % 4) .. +31 = this CTA's output rows
    // m0 + 128 rank + 32 (w % 4) + lane; columns = the tile's 256 n
    const int q = warp & 3;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);
    uint8_t* stg0 = smem + OFF_STG + (warp - EPI_WARP0) * 2 * STG_BYTES;
    int acc = 0;
    uint32_t aph = 0;
    bool stg_zero = false;  // buffer 0 holds zeros
    int last = -1;          // buffer of the most recent store group
    // before buffer b is rewritten, its last store has read it out
    auto claim = [&](int b) {
      if (lane == 0) {
        if (last == b)
          bulk_wait_group_read0();
        else
          bulk_wait_group_read1();
      }
      __syncwarp();
    };
    for (int t = cl; t < p.total; t += ncl) {
      const Tile tl = decode(t, p);
      const int n = rows_of(tl.e);
      const int mrow = tl.m0 + static_cast<int>(rank) * 128 + q * 32;
      const bool rows_in = mrow < p.M;
      const int out_row = tl.e * p.M + mrow;
      if (n == 0) {
        // an expert with no rows: store zeros from a zeroed staging block
        if (rows_in) {
          if (!stg_zero) {
            claim(0);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(stg0 + lane * 128 + i * 16) = make_uint4(0, 0, 0, 0);
            fence_proxy_async_shared();
            __syncwarp();
            stg_zero = true;
          }
          if (lane == 0) {
            for (int c = 0; c < BN / 32; ++c)
              if (tl.n0 + c * 32 < p.N) tma_store_2d(&tmY, smem_u32(stg0), tl.n0 + c * 32, out_row);
            bulk_commit_group();
          }
          last = 0;
        }
        continue;
      }
      if (!__all_sync(0xffffffffu, mbar_wait_spin(&tfull[acc], aph, kWaitLimitNs))) {
        timed_out = true;
        break;
      }
      tc_fence_after();
      const uint32_t tb =
          tmem_base + static_cast<uint32_t>(acc * ACC_COLS) + (static_cast<uint32_t>(q * 32) << 16);
      if (rows_in) {
#pragma unroll 1
        for (int c = 0; c < BN / 32; ++c) {
          const int col = tl.n0 + c * 32;
          if (col >= p.N) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tb + c * 32, v);
          tmem_ld_wait();
          const int b = c & 1;
          claim(b);
          uint8_t* stg = stg0 + b * STG_BYTES;
          uint8_t* row_p = stg + lane * 128;
#pragma unroll
          for (int i = 0; i < 8; ++i)
            *reinterpret_cast<uint4*>(row_p + ((i ^ (lane & 7)) << 4)) =
                make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
          fence_proxy_async_shared();
          __syncwarp();
          if (lane == 0) {
            tma_store_2d(&tmY, smem_u32(stg), col, out_row);
            bulk_commit_group();
          }
          last = b;
          if (b == 0) stg_zero = false;
        }
      }
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&tempty[acc]);
        else
          mbar_arrive_remote(leader_tempty + static_cast<uint32_t>(acc * 8));
      }
      if (++acc == NUM_ACC) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group0();  // this warp's stores are done
  }

  if (timed_out) atomicOr(p.err, kErrTimeout);
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, TMEM_COLS);
  }
}

cudaError_t set_wgrad_smem_attr() {
  static std::once_flag once;
  static cudaError_t st = cudaSuccess;
  std::call_once(once, [] {
    st = cudaFuncSetAttribute(wgrad_pair_kernel<false>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, wg::SMEM_BYTES);
    if (st == cudaSuccess)
      st = cudaFuncSetAttribute(wgrad_pair_kernel<true>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, wg::SMEM_BYTES);
  });
  return st;
}

// Clusters of two that can be resident at once (cached per device): a
// persistent grid must fit at once (a pair needs two free SMs of one GPC).
int resident_clusters(const cudaLaunchConfig_t& lc_in, int num_sms) {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cache[dev] > 0) return cache[dev];
  cudaLaunchConfig_t lc = lc_in;
  lc.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)));
  int n = 0;
  // (both forms: the same threads, registers within the launch bound and shared memory)
  if (cudaOccupancyMaxActiveClusters(&n, wgrad_pair_kernel<false>, &lc) != cudaSuccess || n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  cache[dev] = n;
  return n;
}

}  // namespace

namespace {
// Either form: A [a_rows][M] single and B [R][2N] split, or (split_a) A
// [R][2M] split and B [b_rows][N] single.
cudaError_t launch_wgrad(const void* A, int a_rows, int a_shared, const void* B, int b_rows,
                         int b_shared, int split_a, int R, int E, int M, int N,
                         const int32_t* offsets, float* out, uint32_t* err, int num_sms,
                         cudaStream_t s) {
  if (E <= 0) return cudaSuccess;
  if (M <= 0 || N <= 0 || M % 64 != 0 || N % 8 != 0 || num_sms < 2 || E > kMaxExperts)
    return cudaErrorInvalidValue;
  if (R <= 0 || a_rows <= 0 || b_rows <= 0)  // no rows anywhere: every gradient is zero
    return cudaMemsetAsync(out, 0, static_cast<size_t>(E) * M * N * 4, s);
  CUtensorMap mA, mB, mY;
  std::memset(&mA, 0, sizeof(mA));
  std::memset(&mB, 0, sizeof(mB));
  std::memset(&mY, 0, sizeof(mY));
  const uint64_t a_cols = static_cast<uint64_t>(M) * (split_a ? 2 : 1);
  const uint64_t b_cols = static_cast<uint64_t>(N) * (split_a ? 1 : 2);
  if (!make_map_2d(&mA, A, static_cast<uint64_t>(a_rows), a_cols, 64, wg::BK) ||
      !make_map_2d(&mB, B, static_cast<uint64_t>(b_rows), b_cols, 64, wg::BK) ||
      !make_map_2d_out(&mY, out, static_cast<uint64_t>(E) * M, static_cast<uint64_t>(N), true))
    return cudaErrorInvalidValue;
  wg::Params prm;
  prm.offsets = offsets;
  prm.err = err;
  prm.E = E;
  prm.M = M;
  prm.N = N;
  prm.R = R;
  prm.a_shared = a_shared;
  prm.b_shared = b_shared;
  prm.tiles_m = ceil_div(M, wg::BM);
  prm.tiles_n = ceil_div(N, wg::BN);
  prm.total = E * prm.tiles_m * prm.tiles_n;
  cudaError_t st = set_wgrad_smem_attr();
  if (st != cudaSuccess) return st;
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(wg::THREADS);
  lc.dynamicSmemBytes = wg::SMEM_BYTES;
  lc.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // see pdl_wait
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  lc.attrs = attr;
  lc.numAttrs = 2;
  const int resident = resident_clusters(lc, num_sms);
  const int clusters = prm.total < resident ? prm.total : resident;
  lc.gridDim = dim3(static_cast<unsigned>(2 * clusters));
  return split_a ? cudaLaunchKernelEx(&lc, wgrad_pair_kernel<true>, mA, mB, mY, prm)
                 : cudaLaunchKernelEx(&lc, wgrad_pair_kernel<false>, mA, mB, mY, prm);
}
}  // namespace

cudaError_t launch_wgrad_tc(const void* A, int a_rows, int a_shared, const void* Bs, int R, int E,
                            int M, int N, const int32_t* offsets, float* out, uint32_t* err,
                            int num_sms, cudaStream_t s) {
  return launch_wgrad(A, a_rows, a_shared, Bs, R, 0, 0, R, E, M, N, offsets, out, err, num_sms, s);
}

cudaError_t launch_wgrad_tc_split_a(const void* As, int R, const void* B, int b_rows,
                                    int b_shared, int E, int M, int N, const int32_t* offsets,
                                    float* out, uint32_t* err, int num_sms, cudaStream_t s) {
  return launch_wgrad(As, R, 0, B, b_rows, b_shared, 1, R, E, M, N, offsets, out, err, num_sms,
                      s);
}

}  // namespace moe
