// gemm_tc.cu - grouped expert GEMM on the sm_103a tensor cores (tcgen05 +
// TMEM, 2-SM pair mode), fed by TMA, over the variable-length expert segments
// the dispatch produced. One kernel serves both projections of the expert
// FFN ("L1 + Act + L2", DeepSeek V3/V4 parallel-strategy article, Waved-EP
// section):
//   W1 pass: H[r] = SiLU(s_r * A[r] . W1[e])  -> bf16   (epi 0)
//   W2 pass: Y[r] = H[r] . W2[e]              -> fp32   (epi 1)
// for the rows r of each expert's segment [offsets[e], offsets[e+1]); the
// backward's dgrad uses it too (fp32 out, or epi 2: dZ[r] = (A[r] . W[e]) *
// SiLU'(Z[r]) written as its bf16 split [hi | lo], the operand of the next
// GEMMs).
//
// Work split. A cluster of two CTAs (one per SM of an SM pair) computes a
// pair tile of 256 token rows x 256 output features with one
// tcgen05.mma.cta_group::2 M256 N256 K16 per k-step, issued by the even CTA.
// Each CTA stages only its own 128 token rows (A, K-major) and its own
// 128-feature half of the weight tile (B, the row-major weight read
// MN-major), and each CTA's tensor memory receives the accumulator rows of
// its own tokens. Per SM this is 2/3 of the shared-memory traffic of a
// one-CTA M128 N256 tile (TMA fills plus tensor-core operand reads), which is
// what bounds the one-CTA form. An expert's rows are covered by full
// 256-row tiles plus, for the remainder, one swapped tile (weights as the
// MMA's M side, the remaining tokens as its N, any multiple of 16), so a
// short tail costs a fraction of a full tile. Tiles run expert by expert,
// weight tile by weight tile, with the token tiles of one weight tile
// adjacent, so pairs running side by side share the weight tile through
// L2; an expert with no rows has no tiles and its weights are never read
// (the contiguous per-expert weight layout of the DeepSeek-V4 EP article,
// section 5.2, makes every weight tile one strided TMA box).
//
// Shared memory per CTA: a 6-stage ring of 32 KB (16 KB token rows, 16 KB
// weight half, 128-byte swizzle) for 256-feature tiles, or 4 stages of 48 KB
// for 512-feature tiles (two MMAs per k-step sharing the token operand, used
// for long-K SiLU passes with many tiles). Warp roles: warp 0 TMA producer
// (one thread, both CTAs); warp 1 TMEM allocation (both CTAs) and MMA issue
// (even CTA); warps 2.. epilogue, 8 for the SiLU pass (two per TMEM lane
// quadrant, each half the columns) and 4 for the fp32 pass (tcgen05.ld 32
// columns at a time, FP8 row scale and SiLU, then a 32 x 32 block staged in
// shared memory and written by one TMA store; rows of a swapped or merged
// remainder are stored by the threads, rows past the segment masked). Every
// wait is bounded; a timeout sets kErrTimeout and the kernel drains its
// copies and MMAs, frees TMEM and exits.
//
// FP8 token rows (the dispatch's E4M3 payload, W1 pass): the producer loads
// each CTA's 128 rows x 64 E4M3 bytes into the first half of the stage's
// token slot; 8 converter warps (two groups of 4 on alternate stages) expand
// them in place to the bf16 layout the MMA reads (exact) and release the
// stage: the even CTA's warps by an arrive, the odd CTA's by 16-byte bulk
// copies whose bytes complete the even CTA's full barrier. The per-row
// payload scale is applied in the epilogue. This is the GEMM's dequantising
// prologue; no bf16 copy of the payload is written to memory.
//
// Gathered token rows (GA, the W1 pass of the single-GPU form of the
// Waved-EP fusion, DeepSeek V3/V4 parallel-strategy article: the dispatch
// and the first expert GEMM in one pass): the packed rows are never written.
// Row r of expert e's segment is row src[r] of x; 4 gather warps copy each
// stage's rows from x into the swizzled token slot with 16-byte cp.async
// copies (whole 128-byte row pieces per 8 lanes), wait for their own copies,
// and release the stage like the FP8 converters do. TMA keeps the weight
// boxes.
#include <atomic>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "ptx.cuh"
#include "tmap.cuh"

namespace moe {
namespace {

using namespace ptx;

struct TcParams {
  const int32_t* gsrc;  // GA: token of each routed row (the dispatch's src)
  const void* gx;       // GA: x [gx_rows, K] bf16, the rows gathered
  int gx_rows;
  const int32_t* offsets;
  const float* row_scale;
  const float* zin;    // epi 2: the pre-activation Z [R, N] (fp32)
  float* zout;         // epi 0, nullable: also write the pre-activation Z [R, N]
                       // (fp32, the value SiLU takes), for a backward pass
  void* out;
  uint32_t* err;
  uint32_t* tile_ctr;  // next tile to hand out; zero before the launch
  int E, K, N, R, n_tiles;
  int n_tiles_m;       // feature blocks of a merged tile (ceil(N / 224))
  int group;           // token tiles of one expert that run over all its
                       // feature blocks before the next ones (>= 1)
  int a_rows;          // rows of A
  int a_shared;        // 1: output row r of expert e reads A row r - offsets[e]
  int k_wrap;          // BT: columns of the stored weight; k-block kb reads
                       // columns (64 kb) mod k_wrap (K = 2 k_wrap stacks it twice)
  uint64_t epi_wait_ns;  // bound of the epilogue's wait for a finished accumulator
};

// SiLU'(z) = s (1 + z (1 - s)), s = sigmoid(z), with the approximate exp
// and divide (relative error under 1e-5 over the range where s is not
// flushed, far below the 2e-3 bound on bf16 layers' gradients; for z < -87
// the denominator passes 2^126, s flushes to 0 and so does SiLU'(z))
__device__ __forceinline__ float silu_grad(float z) {
  const float sg = __fdividef(1.f, 1.f + __expf(-z));
  return sg * (1.f + z * (1.f - sg));
}
// v = hi + lo, hi = bf16(v), lo = bf16(v - hi), two values packed per word
__device__ __forceinline__ void split2(float a, float b, uint32_t* hi, uint32_t* lo) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
  const float2 hf = __bfloat1622float2(h);
  const __nv_bfloat162 l = __floats2bfloat162_rn(a - hf.x, b - hf.y);
  *hi = *reinterpret_cast<const uint32_t*>(&h);
  *lo = *reinterpret_cast<const uint32_t*>(&l);
}
__device__ __forceinline__ void split1(float v, __nv_bfloat16* hi, __nv_bfloat16* lo) {
  *hi = __float2bfloat16_rn(v);
  *lo = __float2bfloat16_rn(v - __bfloat162float(*hi));
}

// z * sigmoid(z) with the approximate divide: the result is rounded to bf16,
// far coarser than the few-ulp error of __expf / __fdividef. For z < -87 the
// denominator passes 2^126 and the quotient flushes to 0 (|silu| < 1e-36).
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.f + __expf(-z)); }

// ---------------------------------------------------------------- pair kernel
// Synchronisation across the pair:
//   full[s]   (even CTA) the TMA bytes of both CTAs: each CTA loads into its
//             own shared memory and counts the bytes on the even CTA's
//             barrier (the cta_group::2 form of the tensor copy);
//   empty[s]  both CTAs, from one multicast tcgen05.commit;
//   tfull     both CTAs, multicast commit after a tile's last MMA;
//   tempty    (even CTA) one arrive per epilogue warp of either CTA;
//   tq_full   both CTAs: the even CTA's producer claims the next tile with a
//             global atomic and posts its index to a slot of both CTAs' tile
//             queues (local store + st.shared::cluster, then arrive);
//   tq_empty  (even CTA) every reader of a queue slot: the even CTA's MMA
//             thread and epilogue warps, the odd CTA's producer and
//             epilogue warps.
// Tiles are claimed in index order as pairs become free (dynamic
// scheduling): a fixed round-robin split left some pairs with every full
// tile and others with every short tail.
namespace pairk {
constexpr int BM = 256, BK = 64;
constexpr int A_BYTES = 128 * BK * 2;       // 16 KB: this CTA's 128 rows
constexpr int BOX_BYTES = BK * 64 * 2;      // 8 KB: [64 k][64 n]
constexpr int HALF_B_BYTES = 2 * BOX_BYTES; // 16 KB: this CTA's 128 features of one MMA
constexpr int TMEM_COLS = 512;
// Epilogue warps: 8 for the SiLU pass (two per TMEM lane quadrant, each half
// the columns: the exp/divide work is issue-bound at one warp per SM
// sub-partition), 4 for the fp32 passes (plain stores; more warps only add
// store bursts against the operand loads, measured slower on GB300).
template <int EPI, int NB>
__host__ __device__ constexpr int num_epi_warps() { return EPI == 0 ? 8 : 4; }
// FP8 token rows (A8): 8 more warps expand the staged E4M3 tiles to bf16,
// two groups of 4 taking alternate stages (one group's chain per stage, ~720
// cycles measured, is longer than the MMA's k-block).
constexpr int CONV_GROUP = 4;
template <bool A8>
__host__ __device__ constexpr int num_conv_warps() { return A8 ? 2 * CONV_GROUP : 0; }
// Gathered token rows (GA): 4 more warps copy each stage's rows from x.
constexpr int GATHER_WARPS = 4;
template <bool GA>
__host__ __device__ constexpr int num_gather_warps() { return GA ? GATHER_WARPS : 0; }
template <int EPI, int NB, bool A8 = false, bool GA = false>
__host__ __device__ constexpr int num_threads() {
  return 64 + 32 * (num_epi_warps<EPI, NB>() + num_conv_warps<A8>() + num_gather_warps<GA>());
}

// Merged tiles (256-feature shape only). An expert whose rows end in a short
// remainder (1..TAIL_MAX rows after at least one full 256-row tile) covers
// its last full tile and the remainder together: 224 features per tile, the
// odd CTA's weight half shifted to start at n0 + 112 so that the pair MMA
// M256 N224 sees 224 contiguous features, plus one swapped MMA M256 (the
// same staged weights, features n0 .. n0 + 239 with 16 seen twice) x
// N = remainder padded to 16, accumulating at TMEM column 224. The whole tile
// still fits one 256-column accumulator, and the remainder costs neither a
// second read of the weight tile nor a tile of its own.
constexpr int MT_W = 224, MT_HALF = 112, TAIL_MAX = 32;
constexpr int TAIL_SLOT = (TAIL_MAX / 2) * BK * 2;  // 2 KB: this CTA's half of the remainder

// NB = 1: 256-feature pair tiles, two TMEM accumulators (the epilogue of one
// tile overlaps the next tile's main loop), 6 stages of 32 KB.
// NB = 2: 512-feature pair tiles, two M256 N256 MMAs per k-step sharing the
// token operand, one accumulator filling TMEM, 4 stages of 48 KB: a third
// fewer operand bytes per flop through L2 and shared memory, the epilogue
// exposed once per tile.
template <int NB>
struct Shape {
  static constexpr int BN = 256 * NB;
  static constexpr bool MERGE = NB == 1;  // merged remainder tiles
  static constexpr int STAGES = NB == 1 ? 6 : 4;
  static constexpr int B_BYTES = NB * HALF_B_BYTES;
  static constexpr int T_BYTES = MERGE ? TAIL_SLOT : 0;
  static constexpr int STAGE_BYTES = A_BYTES + B_BYTES + T_BYTES;
  static constexpr int NUM_ACC = 2 / NB;
  static constexpr int ACC_COLS = TMEM_COLS / NUM_ACC;
  static constexpr int OFF_A = 0;
  static constexpr int OFF_B = STAGES * A_BYTES;
  static constexpr int OFF_T = OFF_B + STAGES * B_BYTES;
  static constexpr int OFF_BAR = STAGES * STAGE_BYTES;
  static constexpr int TQ = 8;  // tile queue slots
  // full, empty, tfull, tempty, drain, tq_full, tq_empty, a8_full
  static constexpr int NUM_BARS = 3 * STAGES + 2 * NUM_ACC + 1 + 2 * TQ;
  static constexpr int OFF_MISC = OFF_BAR + NUM_BARS * 8;
  static constexpr int OFF_TQ = OFF_MISC + 16;
  static constexpr int OFF_SEG = OFF_TQ + TQ * 4;
  static constexpr int OFF_TSTART = OFF_SEG + (kMaxExperts + 1) * 4;
  // 16 bytes that the odd CTA's FP8 converters copy to the even CTA (A8)
  static constexpr int OFF_SINK = (OFF_TSTART + (kMaxExperts + 1) * 4 + 15) & ~15;
  static constexpr int SMEM_USED = OFF_SINK + 16;
  static constexpr int SMEM_BYTES = SMEM_USED + 1024;
  static_assert(SMEM_BYTES <= 227 * 1024, "shared memory");
};

// Output staging: each epilogue warp puts a block of its 32 rows x 32
// columns in shared memory past the ring (fp32: 128-byte rows, 128-byte
// swizzle; bf16: 64-byte rows, 64-byte swizzle; 1024-byte aligned) and
// writes it with one TMA store: whole row segments instead of 16-byte pieces
// of 32 different rows per store instruction. (A build whose fp32 warps
// exchanged 16-byte pieces by shuffles so that each plain store wrote four
// whole 128-byte row segments, with no staging, measured 1 % slower on the
// 256-expert layer's W2 pass.)
template <int EPI>
__host__ __device__ constexpr int stg_bytes() { return EPI == 0 ? 32 * 32 * 2 : 32 * 32 * 4; }
template <int NB>
__host__ __device__ constexpr int off_stg() {
  return (Shape<NB>::SMEM_USED + 1023) & ~1023;
}
template <int EPI, int NB>
__host__ __device__ constexpr int smem_bytes() {
  return off_stg<NB>() + num_epi_warps<EPI, NB>() * stg_bytes<EPI>() + 1024;
}
static_assert(smem_bytes<0, 1>() <= 227 * 1024 && smem_bytes<0, 2>() <= 227 * 1024 &&
                  smem_bytes<1, 1>() <= 227 * 1024 && smem_bytes<1, 2>() <= 227 * 1024 &&
                  smem_bytes<2, 1>() <= 227 * 1024,
              "shared memory");

// Descriptor of this CTA's staged weights at k-step kk: MN-major (two
// [64 k][64 n] boxes, 8 KB apart; a k-step is 16 rows of 128 bytes) or, for
// transposed weights, K-major ([128 n][64 k], a k-step is 32 bytes along the
// swizzled row).
template <bool BT>
__device__ __forceinline__ uint64_t wdesc(uint32_t base, int kk) {
  return BT ? make_sdesc_sw128(base + kk * 32, 16, 1024)
            : make_sdesc_sw128(base + kk * 2048, BOX_BYTES, 1024);
}

struct PTile {
  int e, row0, ntok, n0;  // token rows [row0, row0 + ntok), features from n0
  bool swap;              // tail tile: weights are the MMA's M side, tokens its N
  int width;              // features (bn, or MT_W for a merged tile)
  int tail;               // merged tile: remainder rows at row0 + BM (else 0)
};

__device__ __forceinline__ bool merges(int rows, bool merge) {
  const int full = rows / BM, rem = rows - full * BM;
  return merge && full > 0 && rem > 0 && rem <= TAIL_MAX;
}

// Tiles of one expert with `rows` rows.
__device__ __forceinline__ int expert_tiles(int rows, int n_tiles, int n_tiles_m, bool merge) {
  const int full = rows / BM, rem = rows - full * BM;
  if (merges(rows, merge)) return (full - 1) * n_tiles + n_tiles_m;
  return (full + (rem > 0 ? 1 : 0)) * n_tiles;
}

// An expert's rows are covered by full 256-row pair tiles and, for the
// remainder (1..255 rows), one swapped tile whose MMA N is the remainder
// rounded up to 16, so a short tail costs a fraction of a full tile; or, for
// a remainder of at most TAIL_MAX rows, merged tiles (see MT_W) in place of
// the last full tile and the swapped one.
// Order: the expert's token tiles go in groups of `group`; a group runs over
// every weight tile (feature block), weight tile by weight tile, before the
// next group starts, and the group's token tiles of one weight tile are
// adjacent. Pairs running side by side then share each weight tile, and a
// group's token rows stay in L2 while its weight tiles stream past: with
// one group per expert (the plain weight-tile-major order) a heavy
// expert's token rows left L2 between its weight tiles and were read again
// from DRAM for each of them.
__device__ __forceinline__ void order(int local, int mt, int n_tiles, int group, int& nt, int& m) {
  const int g = local / (group * n_tiles);
  const int base = g * group;
  const int gm = min(group, mt - base);  // token tiles in this group
  const int idx = local - base * n_tiles;
  nt = idx / gm;
  m = base + (idx - nt * gm);
}

__device__ __forceinline__ PTile decode(int tile, const int* tstart, const int* seg, int E,
                                        int n_tiles, int bn, int n_tiles_m, bool merge,
                                        int group) {
  int lo = 0, hi = E;
  while (hi - lo > 1) {
    const int mid = (lo + hi) >> 1;
    if (tstart[mid] <= tile)
      lo = mid;
    else
      hi = mid;
  }
  PTile t;
  t.e = lo;
  const int local = tile - tstart[lo];
  const int rows = seg[lo + 1] - seg[lo];
  const int full = rows / BM, rem = rows - full * BM;
  t.width = bn;
  t.tail = 0;
  if (merges(rows, merge)) {
    const int plain = (full - 1) * n_tiles;
    if (local >= plain) {
      t.row0 = seg[lo] + (full - 1) * BM;
      t.swap = false;
      t.ntok = BM;
      t.n0 = (local - plain) * MT_W;
      t.width = MT_W;
      t.tail = rem;
      return t;
    }
    int nt, m;
    order(local, full - 1, n_tiles, group, nt, m);
    t.row0 = seg[lo] + m * BM;
    t.swap = false;
    t.ntok = BM;
    t.n0 = nt * bn;
    return t;
  }
  const int mt = full + (rem > 0 ? 1 : 0);
  int nt, m;
  order(local, mt, n_tiles, group, nt, m);
  t.row0 = seg[lo] + m * BM;
  t.swap = m == full;
  t.ntok = t.swap ? rem : BM;
  t.n0 = nt * bn;
  return t;
}
}  // namespace pairk

// BT: the weights are stored transposed, [E][N][k_wrap] row-major (the
// layer's own W2 for dH = dY W2^T, W1 for dX = dZ W1^T), and are read
// K-major: one [128 features][64 k] box per CTA and k-block, with no
// transposed copy in memory.
template <int EPI, int NB, bool A8, bool BT = false, bool GA = false>
__global__ void __launch_bounds__(pairk::num_threads<EPI, NB, A8, GA>(), 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA,
                     const __grid_constant__ CUtensorMap tmA8,
                     const __grid_constant__ CUtensorMap tmB,
                     const __grid_constant__ CUtensorMap tmY, const TcParams p) {
  using S = pairk::Shape<NB>;
  constexpr int NEW = pairk::num_epi_warps<EPI, NB>();
  constexpr int NH = NEW / 4;  // warps per TMEM lane quadrant
  constexpr int NCV = pairk::num_conv_warps<A8>();
  constexpr int NGW = pairk::num_gather_warps<GA>();
  static_assert(!GA || (!A8 && !BT), "gathered rows: bf16 rows, weights read MN-major");
  // FP8 token rows come without merged remainder tiles (a remainder is a
  // swapped tile, its rows expanded like any other)
  constexpr bool MERGE = S::MERGE && !A8;
  static_assert(!BT || (NB == 1 && !A8), "transposed weights: 256-feature tiles, bf16 rows");
  // instruction descriptors (A or B K-major / MN-major per the weight layout)
  constexpr uint32_t IDESC_N = make_idesc_bf16_f32(pairk::BM, 256, false, !BT);
  constexpr uint32_t IDESC_M = make_idesc_bf16_f32(pairk::BM, pairk::MT_W, false, !BT);
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>(
      (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + S::OFF_A;
  uint8_t* sB = smem + S::OFF_B;
  uint8_t* sT = smem + S::OFF_T;  // merged tiles' remainder rows (MERGE)
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S::OFF_BAR);
  uint64_t* empty = full + S::STAGES;
  uint64_t* tfull = empty + S::STAGES;
  uint64_t* tempty = tfull + S::NUM_ACC;
  uint64_t* drain = tempty + S::NUM_ACC;
  uint64_t* tq_full = drain + 1;
  uint64_t* tq_empty = tq_full + S::TQ;
  uint64_t* a8_full = tq_empty + S::TQ;  // A8: this CTA's E4M3 tile has landed
  int* tq = reinterpret_cast<int*>(smem + S::OFF_TQ);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + S::OFF_MISC);
  int* s_total = reinterpret_cast<int*>(smem + S::OFF_MISC + 4);
  int* seg = reinterpret_cast<int*>(smem + S::OFF_SEG);
  int* tstart = reinterpret_cast<int*>(smem + S::OFF_TSTART);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int E = p.E;
  pdl_wait();
  pdl_trigger();

  if (warp == 0) {
    for (int e = lane; e <= E; e += 32) seg[e] = __ldg(p.offsets + e);
    __syncwarp();
    bool ok = true;
    int running = 0;
    for (int b = 0; b < E; b += 32) {
      const int e = b + lane;
      int tiles = 0;
      bool bad = false;
      if (e < E) {
        const int lo = seg[e], hi = seg[e + 1];
        bad = lo < 0 || hi < lo || hi > p.R;
        tiles = bad ? 0 : pairk::expert_tiles(hi - lo, p.n_tiles, p.n_tiles_m, MERGE);
      }
      if (__any_sync(0xffffffffu, bad)) ok = false;
      int incl = tiles;
#pragma unroll
      for (int off = 1; off < 32; off <<= 1) {
        const int o = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += o;
      }
      if (e < E) tstart[e] = running + incl - tiles;
      running += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      tstart[E] = running;
      *s_total = ok ? running : 0;
      if (!ok && blockIdx.x == 0) atomicOr(p.err, kErrBadIndex);
      for (int i = 0; i < S::STAGES; ++i) {
        // A8: the producer's arrive and one arrive per warp of the even
        // CTA's converter group for this stage; the odd CTA's converters
        // signal through bytes (see the converters)
        mbar_init(&full[i], A8 ? 1 + pairk::CONV_GROUP : (GA ? 1 + NGW : 1));
        mbar_init(&empty[i], 1);
        mbar_init(&a8_full[i], 1);
      }
      for (int i = 0; i < S::NUM_ACC; ++i) {
        mbar_init(&tfull[i], 1);
        mbar_init(&tempty[i], 2 * NEW);  // epilogue warps of both CTAs
      }
      mbar_init(drain, 1);
      for (int i = 0; i < S::TQ; ++i) {
        mbar_init(&tq_full[i], 1);
        mbar_init(&tq_empty[i], 2 + 2 * NEW + 2 * NCV + 2 * NGW);
      }
      fence_mbar_init();
    }
  } else if (warp == 1) {
    tmem_alloc_pair(tmem_slot, pairk::TMEM_COLS);
    tmem_relinquish_pair();
  }
  __syncthreads();
  cluster_sync();  // the peer's barriers exist before anyone signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int total = *s_total;
  const int KB = p.K / pairk::BK;
  bool timed_out = false;

  // Tile queue. Readers take slots in order; `next_tile` waits for the slot
  // (cluster-scope acquire: the odd CTA's copy is written remotely), reads
  // the index and releases the slot on the even CTA's tq_empty.
  int q_slot = 0;
  uint32_t q_ph = 0;
  const uint32_t leader_tq_empty = mapa_shared(smem_u32(tq_empty), 0);
  auto next_tile = [&](bool whole_warp) -> int {
    const bool ok = mbar_wait_cluster(&tq_full[q_slot], q_ph, kWaitLimitNs);
    const bool all_ok = whole_warp ? __all_sync(0xffffffffu, ok) : ok;
    int t = total;  // a timeout reads as the end of the work
    if (all_ok) {
      t = tq[q_slot];
      if (!whole_warp || lane == 0) {
        if (rank == 0)
          mbar_arrive(&tq_empty[q_slot]);
        else
          mbar_arrive_remote(leader_tq_empty + static_cast<uint32_t>(q_slot * 8));
      }
    } else {
      timed_out = true;
    }
    if (++q_slot == S::TQ) {
      q_slot = 0;
      q_ph ^= 1u;
    }
    return t;
  };

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      if (!GA) prefetch_tmap(&tmA);
      if (!A8 && !GA) prefetch_tmap(&tmA8);
      prefetch_tmap(&tmB);
      int s = 0;
      uint32_t ph = 0, armed = 0, armed_ph = 0;
      // both CTAs' bytes of a stage are counted on the even CTA's full[s]
      const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
      // even CTA: claim tiles (one claim ahead) and post them; odd CTA: read
      // them from its queue copy
      const uint32_t peer_tq = mapa_shared(smem_u32(tq), 1);
      const uint32_t peer_tq_full = mapa_shared(smem_u32(tq_full), 1);
      // unsigned: any counter value maps to a valid tile or to the end
      uint32_t claimed = rank == 0 ? atomicAdd(p.tile_ctr, 1u) : 0u;
      // GA: the even CTA posts each tile one ahead of the one it loads, so
      // the gather warps can fetch the next tile's row tokens while they
      // copy the current one (the post: both CTAs' queue copies, then the
      // end marker once the tiles run out; a timeout posts the end)
      auto post = [&](int tile) -> int {
        if (!mbar_wait_cluster(&tq_empty[q_slot], q_ph ^ 1u, kWaitLimitNs)) {
          timed_out = true;
          tile = total;
        }
        tq[q_slot] = tile;
        st_shared_cluster_s32(peer_tq + static_cast<uint32_t>(q_slot * 4), tile);
        mbar_arrive(&tq_full[q_slot]);
        mbar_arrive_remote(peer_tq_full + static_cast<uint32_t>(q_slot * 8));
        if (++q_slot == S::TQ) {
          q_slot = 0;
          q_ph ^= 1u;
        }
        return tile;
      };
      auto claim = [&]() -> int {
        const uint32_t c = atomicAdd(p.tile_ctr, 1u);
        return c < static_cast<uint32_t>(total) ? static_cast<int>(c) : total;
      };
      int ahead = -1;  // GA: the tile posted but not yet loaded
      for (;;) {
        int tile;
        if (GA && rank == 0) {
          if (ahead < 0)
            ahead = post(claimed < static_cast<uint32_t>(total) ? static_cast<int>(claimed) : total);
          tile = ahead;
          if (tile < total && !timed_out) ahead = post(claim());
        } else if (rank == 0) {
          tile = claimed < static_cast<uint32_t>(total) ? static_cast<int>(claimed) : total;
          if (!mbar_wait_cluster(&tq_empty[q_slot], q_ph ^ 1u, kWaitLimitNs)) {
            timed_out = true;
            tile = total;
          }
          tq[q_slot] = tile;
          st_shared_cluster_s32(peer_tq + static_cast<uint32_t>(q_slot * 4), tile);
          mbar_arrive(&tq_full[q_slot]);
          mbar_arrive_remote(peer_tq_full + static_cast<uint32_t>(q_slot * 8));
          if (++q_slot == S::TQ) {
            q_slot = 0;
            q_ph ^= 1u;
          }
          if (tile < total) claimed = atomicAdd(p.tile_ctr, 1u);
        } else {
          tile = next_tile(false);
        }
        if (tile >= total || timed_out) break;
        const pairk::PTile t = pairk::decode(tile, tstart, seg, E, p.n_tiles, S::BN, p.n_tiles_m, MERGE, p.group);
        // normal tile: this CTA's 128 rows; swapped tile: its half of the N tokens
        const int half_rows = t.swap ? ((t.ntok + 15) & ~15) / 2 : 128;
        const int a_base = p.a_shared ? seg[t.e] : 0;
        const int my_row = min(t.row0 - a_base + static_cast<int>(rank) * half_rows, p.a_rows - 1);
        // MMA j covers features n0 + 256 j + [0, 256); this CTA holds the
        // 128 at n0 + 256 j + half_w rank (half_w = 128, or 112 in a merged
        // tile); a box is issued when it starts below N (one that runs past
        // N is zero-filled, its bytes still counted)
        const int half_w = t.tail > 0 ? pairk::MT_HALF : 128;
        // (BT: one [128][64] box, counted as two 8 KB boxes)
        auto boxes = [&](int n) {
          if (BT) return n < p.N ? 2 : 0;
          return n < p.N ? min(2, (p.N - n + 63) / 64) : 0;
        };
        int nbox[NB];
        // A8: the token rows land on this CTA's a8_full, not on full; the
        // odd CTA's converter warps each send 16 bytes to full instead. GA:
        // the gather warps copy the rows; the odd CTA's send 16 bytes each
        uint32_t bytes = A8   ? static_cast<uint32_t>(16 * pairk::CONV_GROUP)
                         : GA ? static_cast<uint32_t>(16 * NGW)
                              : 2u * pairk::A_BYTES;
#pragma unroll
        for (int j = 0; j < NB; ++j) {
          nbox[j] = boxes(t.n0 + j * 256 + static_cast<int>(rank) * half_w);
          bytes += static_cast<uint32_t>((boxes(t.n0 + j * 256) + boxes(t.n0 + j * 256 + half_w)) *
                                         pairk::BOX_BYTES);
        }
        // merged tile: this CTA's half of the remainder rows (8 or 16) in
        // 8-row boxes
        const int tail_half = ((t.tail + 15) & ~15) / 2;
        const int tail_row = t.row0 - a_base + pairk::BM + static_cast<int>(rank) * tail_half;
        if (!GA) bytes += static_cast<uint32_t>(2 * tail_half * pairk::BK * 2);
        const int brow = t.e * p.K;
        for (int kb = 0; kb < KB; ++kb) {
          if (!mbar_wait_spin(&empty[s], ph ^ 1u, kWaitLimitNs)) {
            timed_out = true;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(&full[s], bytes);
          const uint32_t bar = leader_full + static_cast<uint32_t>(s * 8);
          if constexpr (A8) {
            // 128 rows x 64 E4M3 bytes (64-byte swizzle) into the first half
            // of the stage's token slot; the converters expand them in place
            mbar_arrive_expect_tx(&a8_full[s], static_cast<uint32_t>(pairk::A_BYTES / 2));
            tma_load_2d(sA + s * pairk::A_BYTES, &tmA, &a8_full[s], kb * pairk::BK, my_row);
          } else if constexpr (GA) {
            // (the gather warps fill the token slot)
          } else {
            tma_load_2d_pair(sA + s * pairk::A_BYTES, &tmA, bar, kb * pairk::BK, my_row);
          }
          if constexpr (BT) {
            // rows e N + n0 + half_w rank .. +127 of the stored [E N][k_wrap]
            if (nbox[0] > 0)
              tma_load_2d_pair(sB + s * S::B_BYTES, &tmB, bar, (kb * pairk::BK) % p.k_wrap,
                               t.e * p.N + t.n0 + static_cast<int>(rank) * half_w);
          } else {
#pragma unroll
            for (int j = 0; j < NB; ++j)
              for (int c = 0; c < nbox[j]; ++c)
                tma_load_2d_pair(
                    sB + s * S::B_BYTES + j * pairk::HALF_B_BYTES + c * pairk::BOX_BYTES, &tmB,
                    bar, t.n0 + j * 256 + static_cast<int>(rank) * half_w + c * 64,
                    brow + kb * pairk::BK);
          }
          if constexpr (MERGE && !GA) {
            for (int r = 0; r < tail_half; r += 8)
              tma_load_2d_pair(sT + s * S::T_BYTES + r * pairk::BK * 2, &tmA8, bar,
                               kb * pairk::BK, min(tail_row + r, p.a_rows - 1));
          }
          armed |= 1u << s;
          armed_ph = (armed_ph & ~(1u << s)) | (ph << s);
          if (++s == S::STAGES) {
            s = 0;
            ph ^= 1u;
          }
        }
      }
      // drain (even CTA: its full[s] also counts the odd CTA's bytes; A8:
      // each CTA's own E4M3 copies)
      if (rank == 0)
        for (int i = 0; i < S::STAGES; ++i)
          if ((armed >> i) & 1u)
            if (!mbar_wait_spin(&full[i], (armed_ph >> i) & 1u, kWaitLimitNs)) timed_out = true;
      if (A8)
        for (int i = 0; i < S::STAGES; ++i)
          if ((armed >> i) & 1u)
            if (!mbar_wait_spin(&a8_full[i], (armed_ph >> i) & 1u, kWaitLimitNs)) timed_out = true;
    }
  } else if (warp == 1) {
    if (lane == 0 && rank == 0) {
      // -------------------------------------------------------- MMA issuer (even CTA)
      int s = 0, acc = 0;
      uint32_t ph = 0, aph = 0;
      bool issued = false;
      for (;;) {
        const int tile = next_tile(false);
        if (tile >= total || timed_out) break;
        if (!mbar_wait_spin(&tempty[acc], aph ^ 1u, kWaitLimitNs)) {
          timed_out = true;
          break;
        }
        tc_fence_after();
        const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * S::ACC_COLS);
        const pairk::PTile t = pairk::decode(tile, tstart, seg, E, p.n_tiles, S::BN, p.n_tiles_m, MERGE, p.group);
        // MMAs with any feature below N (the rest of a last tile is skipped)
        const int nmma = min(NB, (p.N - t.n0 + 255) / 256);
        // swapped tile: A = weights (the B slot), B = tokens (K-major, the A slot)
        const uint32_t idesc =
            t.swap ? make_idesc_bf16_f32(pairk::BM, (t.ntok + 15) & ~15, !BT, false) : IDESC_N;
        bool merged = false;
        if constexpr (MERGE) merged = t.tail > 0;
        if (merged) {
          // merged tile: per k-block the four M256 N224 MMAs, then the
          // remainder's four swapped MMAs into columns 224.. (its own loop:
          // the extra MMA inside the plain loop slowed every tile's issue)
          const uint32_t idesc_tail =
              make_idesc_bf16_f32(pairk::BM, (t.tail + 15) & ~15, !BT, false);
          for (int kb = 0; kb < KB; ++kb) {
            if (!(GA ? mbar_wait_spin_cluster(&full[s], ph, kWaitLimitNs)
                     : mbar_wait_spin(&full[s], ph, kWaitLimitNs))) {
              timed_out = true;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + s * pairk::A_BYTES);
            const uint32_t b_base = smem_u32(sB + s * S::B_BYTES);
            const uint32_t t_base = smem_u32(sT + s * S::T_BYTES);
#pragma unroll
            for (int kk = 0; kk < pairk::BK / 16; ++kk)
              tc_mma_f16_pair(d_tmem, make_sdesc_sw128(a_base + kk * 32, 16, 1024),
                              pairk::wdesc<BT>(b_base, kk), IDESC_M, (kb | kk) != 0 ? 1u : 0u);
#pragma unroll
            for (int kk = 0; kk < pairk::BK / 16; ++kk)
              tc_mma_f16_pair(d_tmem + pairk::MT_W, pairk::wdesc<BT>(b_base, kk),
                              make_sdesc_sw128(t_base + kk * 32, 16, 1024), idesc_tail,
                              (kb | kk) != 0 ? 1u : 0u);
            issued = true;
            tc_commit_pair_mc(&empty[s], 0x3);
            if (++s == S::STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        } else {
          for (int kb = 0; kb < KB; ++kb) {
            // A8: the odd CTA's converters released their rows with a
            // cluster-scope arrive; acquire at cluster scope
            if (!((A8 || GA) ? mbar_wait_spin_cluster(&full[s], ph, kWaitLimitNs)
                             : mbar_wait_spin(&full[s], ph, kWaitLimitNs))) {
              timed_out = true;
              break;
            }
            tc_fence_after();
            const uint32_t a_base = smem_u32(sA + s * pairk::A_BYTES);
            const uint32_t b_base = smem_u32(sB + s * S::B_BYTES);
#pragma unroll
            for (int kk = 0; kk < pairk::BK / 16; ++kk) {
              const uint64_t tok = make_sdesc_sw128(a_base + kk * 32, 16, 1024);
#pragma unroll
              for (int j = 0; j < NB; ++j) {
                if (j >= nmma) break;
                const uint64_t wt = pairk::wdesc<BT>(b_base + j * pairk::HALF_B_BYTES, kk);
                tc_mma_f16_pair(d_tmem + j * 256, t.swap ? wt : tok, t.swap ? tok : wt, idesc,
                                (kb | kk) != 0 ? 1u : 0u);
              }
            }
            issued = true;
            tc_commit_pair_mc(&empty[s], 0x3);
            if (++s == S::STAGES) {
              s = 0;
              ph ^= 1u;
            }
          }
        }
        if (timed_out) break;
        tc_commit_pair_mc(&tfull[acc], 0x3);
        if (++acc == S::NUM_ACC) {
          acc = 0;
          aph ^= 1u;
        }
      }
      if (timed_out && issued) {
        tc_commit_pair_mc(drain, 0x1);
        mbar_wait_spin(drain, 0, kWaitLimitNs);
      }
    }
  } else if (warp < 2 + NEW) {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // warp w reads TMEM lanes 32 (w % 4) .. +31; with 8 warps, warps 2-5
    // take the first half of the accumulator columns, warps 6-9 the second
    const int q = warp & 3;
    const int hh = (warp - 2) >> 2;
    const uint32_t leader_tempty = mapa_shared(smem_u32(tempty), 0);
    uint8_t* stg = smem + pairk::off_stg<NB>() + (warp - 2) * pairk::stg_bytes<EPI>();
    int acc = 0;
    uint32_t aph = 0;
    for (;;) {
      const int tile = next_tile(true);
      if (tile >= total || timed_out) break;
      const pairk::PTile t = pairk::decode(tile, tstart, seg, E, p.n_tiles, S::BN, p.n_tiles_m, MERGE, p.group);
      // (a bound a test may shorten: once the epilogue gives up, the MMA and
      // the producers stop within their own bounds with no copy armed on one
      // CTA of the pair alone, and every drain below keeps the full bound)
      const bool ok = mbar_wait_spin(&tfull[acc], aph, p.epi_wait_ns);
      if (!__all_sync(0xffffffffu, ok)) {
        timed_out = true;
        break;
      }
      tc_fence_after();
      const uint32_t tbase = tmem_base + static_cast<uint32_t>(acc * S::ACC_COLS) +
                             (static_cast<uint32_t>(q * 32) << 16);
      if (!t.swap) {
        // lane = token row of this CTA, columns = the tile's features (MMA j
        // at TMEM columns 256 j)
        const int r = static_cast<int>(rank) * 128 + q * 32 + lane;
        const bool valid = r < t.ntok && t.row0 + r < p.R;
        const size_t grow = static_cast<size_t>(t.row0) + r;
        // a warp whose 32 rows all belong to the tile (always, in a full or
        // merged tile) stores through its staging block
        const bool tma_rows = __all_sync(0xffffffffu, valid);
        const int wrow0 = t.row0 + static_cast<int>(rank) * 128 + q * 32;
        float scale = 1.f;
        if ((EPI == 0 || EPI == 2) && p.row_scale != nullptr && valid)
          scale = __ldg(p.row_scale + grow);
        const int nch = t.width / 32, per = (nch + NH - 1) / NH;
        const int c_end = min(nch, (hh + 1) * per);
#pragma unroll 1
        for (int c = hh * per; c < c_end; ++c) {
          const int col = t.n0 + c * 32;
          if (col >= p.N) break;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + c * 32, v);
          tmem_ld_wait();
          if constexpr (EPI == 2) {
            // dZ = dH * SiLU'(Z) for this row's 32 columns, split hi | lo
            if (!valid) continue;  // (tma_rows: every lane valid)
            uint32_t hi[16], lo[16];
            const float4* zr = reinterpret_cast<const float4*>(p.zin + grow * p.N + col);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float4 z = __ldg(zr + i);
              split2(__uint_as_float(v[4 * i]) * scale * silu_grad(z.x),
                     __uint_as_float(v[4 * i + 1]) * scale * silu_grad(z.y), &hi[2 * i],
                     &lo[2 * i]);
              split2(__uint_as_float(v[4 * i + 2]) * scale * silu_grad(z.z),
                     __uint_as_float(v[4 * i + 3]) * scale * silu_grad(z.w), &hi[2 * i + 1],
                     &lo[2 * i + 1]);
            }
            if (tma_rows) {
              // two bf16 32 x 32 blocks (64-byte rows, 64-byte swizzle):
              // hi at column col, lo at N + col of the [R, 2N] output
              if (lane == 0) bulk_wait_group_read0();
              __syncwarp();
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const int o = lane * 64 + ((i ^ ((lane >> 1) & 3)) << 4);
                *reinterpret_cast<uint4*>(stg + o) =
                    make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
                *reinterpret_cast<uint4*>(stg + 2048 + o) =
                    make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
              }
              fence_proxy_async_shared();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmY, smem_u32(stg), col, wrow0);
                tma_store_2d(&tmY, smem_u32(stg + 2048), p.N + col, wrow0);
                bulk_commit_group();
              }
              continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                  grow * 2 * p.N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              dst[i] = make_uint4(hi[4 * i], hi[4 * i + 1], hi[4 * i + 2], hi[4 * i + 3]);
              dst[i + p.N / 8] = make_uint4(lo[4 * i], lo[4 * i + 1], lo[4 * i + 2], lo[4 * i + 3]);
            }
            continue;
          }
          if (EPI == 1 && tma_rows) {
            // the previous store of this block has read it out
            if (lane == 0) bulk_wait_group_read0();
            __syncwarp();
            uint8_t* row_p = stg + lane * 128;
#pragma unroll
            for (int i = 0; i < 8; ++i)
              *reinterpret_cast<uint4*>(row_p + ((i ^ (lane & 7)) << 4)) =
                  make_uint4(v[4 * i], v[4 * i + 1], v[4 * i + 2], v[4 * i + 3]);
            fence_proxy_async_shared();
            __syncwarp();
            if (lane == 0) {
              tma_store_2d(&tmY, smem_u32(stg), col, wrow0);
              bulk_commit_group();
            }
            continue;
          }
          if (!valid) continue;
          if constexpr (EPI == 0) {
            if (!A8 && p.zout != nullptr) {  // (no backward for FP8 rows)
              float4* zd = reinterpret_cast<float4*>(p.zout + grow * p.N + col);
#pragma unroll
              for (int i = 0; i < 8; ++i)
                zd[i] = make_float4(__uint_as_float(v[4 * i]) * scale,
                                    __uint_as_float(v[4 * i + 1]) * scale,
                                    __uint_as_float(v[4 * i + 2]) * scale,
                                    __uint_as_float(v[4 * i + 3]) * scale);
            }
            uint32_t packed[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) {
              const float a = silu(__uint_as_float(v[2 * i]) * scale);
              const float b = silu(__uint_as_float(v[2 * i + 1]) * scale);
              const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
              packed[i] = *reinterpret_cast<const uint32_t*>(&h);
            }
            if (tma_rows) {
              if (lane == 0) bulk_wait_group_read0();
              __syncwarp();
              uint8_t* row_p = stg + lane * 64;
#pragma unroll
              for (int i = 0; i < 4; ++i)
                *reinterpret_cast<uint4*>(row_p + ((i ^ ((lane >> 1) & 3)) << 4)) =
                    make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                               packed[4 * i + 3]);
              fence_proxy_async_shared();
              __syncwarp();
              if (lane == 0) {
                tma_store_2d(&tmY, smem_u32(stg), col, wrow0);
                bulk_commit_group();
              }
              continue;
            }
            uint4* dst = reinterpret_cast<uint4*>(static_cast<__nv_bfloat16*>(p.out) +
                                                  grow * p.N + col);
#pragma unroll
            for (int i = 0; i < 4; ++i)
              dst[i] = make_uint4(packed[4 * i], packed[4 * i + 1], packed[4 * i + 2],
                                  packed[4 * i + 3]);
          } else {
            float4* dst =
                reinterpret_cast<float4*>(static_cast<float*>(p.out) + grow * p.N + col);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                   __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
          }
        }
        if constexpr (MERGE) {
          if (t.tail > 0 && hh == NH - 1) {
            // merged tile's remainder: lane = feature (this CTA's M row of
            // the swapped MMA: n0 + 112 rank + 32 q + lane, the first 112 of
            // each CTA distinct), columns = the remainder's tokens
            const int l = q * 32 + lane;
            const int f = t.n0 + static_cast<int>(rank) * pairk::MT_HALF + l;
            const bool f_ok = l < pairk::MT_HALF && f < p.N;
            uint32_t v[32];
            tmem_ld_32x32b_x32(tbase + pairk::MT_W, v);
            tmem_ld_wait();
            const int trow = t.row0 + pairk::BM;
            float my_scale = 1.f;
            if ((EPI == 0 || EPI == 2) && p.row_scale != nullptr && lane < t.tail)
              my_scale = __ldg(p.row_scale + trow + lane);
            const size_t base = static_cast<size_t>(trow) * p.N + f;
            if constexpr (EPI == 0) {
              __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + base;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const float sj = __shfl_sync(0xffffffffu, my_scale, jj);
                if (jj < t.tail && f_ok) {
                  const float z = __uint_as_float(v[jj]) * sj;
                  if (!A8 && p.zout != nullptr) p.zout[base + static_cast<size_t>(jj) * p.N] = z;
                  out[static_cast<size_t>(jj) * p.N] = __float2bfloat16_rn(silu(z));
                }
              }
            } else if constexpr (EPI == 2) {
              __nv_bfloat16* out =
                  static_cast<__nv_bfloat16*>(p.out) + static_cast<size_t>(trow) * 2 * p.N + f;
              // every Z load issued before the first store
              float z[32];
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                z[jj] = jj < t.tail && f_ok
                            ? __ldg(p.zin + static_cast<size_t>(trow + jj) * p.N + f)
                            : 0.f;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj) {
                const float sj = __shfl_sync(0xffffffffu, my_scale, jj);
                if (jj < t.tail && f_ok) {
                  __nv_bfloat16* o = out + static_cast<size_t>(jj) * 2 * p.N;
                  split1(__uint_as_float(v[jj]) * sj * silu_grad(z[jj]), o, o + p.N);
                }
              }
            } else {
              float* out = static_cast<float*>(p.out) + base;
#pragma unroll
              for (int jj = 0; jj < 32; ++jj)
                if (jj < t.tail && f_ok) out[static_cast<size_t>(jj) * p.N] = __uint_as_float(v[jj]);
            }
          }
        }
      } else {
        // lane = output feature (MMA j's M row 128 rank + 32 q + lane),
        // columns = the tail's tokens; the (MMA, 32-token chunk) pieces are
        // dealt round-robin to the warps of a lane quadrant
        const int nch = (t.ntok + 31) / 32;
#pragma unroll 1
        for (int i = hh; i < NB * nch; i += NH) {
          const int j = i / nch, c = i - j * nch;
          const int f = t.n0 + j * 256 + static_cast<int>(rank) * 128 + q * 32 + lane;
          const bool f_ok = f < p.N;
          uint32_t v[32];
          tmem_ld_32x32b_x32(tbase + j * 256 + c * 32, v);
          tmem_ld_wait();
          const int tok0 = c * 32;
          const int nt = min(32, t.ntok - tok0);
          float my_scale = 1.f;
          if ((EPI == 0 || EPI == 2) && p.row_scale != nullptr && lane < nt)
            my_scale = __ldg(p.row_scale + t.row0 + tok0 + lane);
          const size_t base = (static_cast<size_t>(t.row0) + tok0) * p.N + f;
          if constexpr (EPI == 0) {
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + base;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const float sj = __shfl_sync(0xffffffffu, my_scale, jj);
              if (jj < nt && f_ok) {
                const float z = __uint_as_float(v[jj]) * sj;
                if (!A8 && p.zout != nullptr) p.zout[base + static_cast<size_t>(jj) * p.N] = z;
                out[static_cast<size_t>(jj) * p.N] = __float2bfloat16_rn(silu(z));
              }
            }
          } else if constexpr (EPI == 2) {
            const size_t r0 = static_cast<size_t>(t.row0) + tok0;
            __nv_bfloat16* out = static_cast<__nv_bfloat16*>(p.out) + r0 * 2 * p.N + f;
            // every Z load issued before the first store
            float z[32];
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              z[jj] = jj < nt && f_ok ? __ldg(p.zin + (r0 + jj) * p.N + f) : 0.f;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj) {
              const float sj = __shfl_sync(0xffffffffu, my_scale, jj);
              if (jj < nt && f_ok) {
                __nv_bfloat16* o = out + static_cast<size_t>(jj) * 2 * p.N;
                split1(__uint_as_float(v[jj]) * sj * silu_grad(z[jj]), o, o + p.N);
              }
            }
          } else {
            float* out = static_cast<float*>(p.out) + base;
#pragma unroll
            for (int jj = 0; jj < 32; ++jj)
              if (jj < nt && f_ok) out[static_cast<size_t>(jj) * p.N] = __uint_as_float(v[jj]);
          }
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
      if (++acc == S::NUM_ACC) {
        acc = 0;
        aph ^= 1u;
      }
    }
    if (lane == 0) bulk_wait_group0();  // this warp's TMA stores are done
  } else if constexpr (GA) {
    // ------------------------------------------------------------ row gather (GA, both CTAs)
    // Thread g copies chunk g % 8 (16 bytes) of rows g / 8 + 16 j, j = 0..7,
    // of each stage's k-block: 8 lanes read one row's 128 contiguous bytes.
    // After issuing a stage, a thread with STAGES - 1 stages in flight waits
    // for the oldest (its own copies: cp.async.wait_group), makes its writes
    // visible to the tensor cores (proxy fence) and releases it to the MMA:
    // an arrive on full (even CTA), or a 16-byte bulk copy whose bytes
    // complete the even CTA's full barrier (odd CTA). The oldest stage is
    // then released one k-block before the MMA needs it; releasing only
    // with all STAGES in flight put the release behind the MMA's freeing of
    // the next slot, a stall at every k-block (measured 1.7-2.1x slower).
    const int gidx = static_cast<int>(threadIdx.x) - 32 * (2 + NEW);
    const int ch = gidx & 7;
    const int rg = gidx >> 3;
    const uint32_t swz = static_cast<uint32_t>((ch ^ (rg & 7)) << 4);
    const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
    const uint32_t leader_sink = mapa_shared(smem_u32(smem + S::OFF_SINK), 0);
    const uint32_t my_sink = smem_u32(smem + S::OFF_SINK);
    const uint4* xv = static_cast<const uint4*>(p.gx);
    // offset (in 16-byte units) of this thread's piece of a routed row's
    // token row (the tokens are loaded together first); a bad token is
    // flagged and read as token 0
    auto token_piece = [&](int tok) -> uint32_t {
      if (tok < 0 || tok >= p.gx_rows) {
        atomicOr(p.err, kErrBadIndex);
        tok = 0;
      }
      return static_cast<uint32_t>(tok) * static_cast<uint32_t>(p.K / 8) + static_cast<uint32_t>(ch);
    };
    int s = 0, so = 0, inflight = 0;
    uint32_t ph = 0;
    bool ok = true;
    auto release_oldest = [&]() {
      fence_proxy_async_shared();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(&full[so]);
        else
          bulk_copy_s2cluster(leader_sink, my_sink, 16u,
                              leader_full + static_cast<uint32_t>(so * 8));
      }
      if (++so == S::STAGES) so = 0;
      --inflight;
    };
    // this CTA's rows of a tile: 128 of a full tile, its half of a swapped
    // tile's tokens (rounded to 16); rows past the segment read a valid row
    // and feed only outputs the epilogue does not store; a merged tile adds
    // this CTA's half of the remainder rows (8 or 16)
    auto tile_rows = [&](const pairk::PTile& t, int& half_rows, int& tail_half) {
      half_rows = t.swap ? ((t.ntok + 15) & ~15) / 2 : 128;
      tail_half = MERGE ? ((t.tail + 15) & ~15) / 2 : 0;
    };
    // the tokens of this thread's rows (rows rg + 16 j, and remainder row rg)
    auto load_tokens = [&](const pairk::PTile& t, int (&tk)[9]) {
      int half_rows, tail_half;
      tile_rows(t, half_rows, tail_half);
      const int r0 = t.row0 + static_cast<int>(rank) * half_rows;
#pragma unroll
      for (int j = 0; j < 8; ++j)
        tk[j] = rg + 16 * j < half_rows ? __ldg(p.gsrc + min(r0 + rg + 16 * j, p.R - 1)) : 0;
      tk[8] = rg < tail_half
                  ? __ldg(p.gsrc + min(t.row0 + pairk::BM + static_cast<int>(rank) * tail_half + rg,
                                       p.R - 1))
                  : 0;
    };
    int next_known = -1;  // the next tile, read ahead from the queue
    int next_tok[9];
    for (;;) {
      const int tile = next_tile(true);
      if (tile >= total || timed_out) break;
      const pairk::PTile t = pairk::decode(tile, tstart, seg, E, p.n_tiles, S::BN, p.n_tiles_m, MERGE, p.group);
      int half_rows, tail_half;
      tile_rows(t, half_rows, tail_half);
      int tok[9];
      if (tile == next_known) {
#pragma unroll
        for (int j = 0; j < 9; ++j) tok[j] = next_tok[j];
      } else {
        load_tokens(t, tok);
      }
      next_known = -1;
      // row pieces: rows rg + 16 j (j < nj: the rows this CTA stages) and,
      // in a merged tile, remainder row rg
      uint32_t off[8];
      const int nj = min(8, max(0, (half_rows - rg + 15) / 16));
#pragma unroll
      for (int j = 0; j < 8; ++j) off[j] = j < nj ? token_piece(tok[j]) : 0u;
      const bool has_tail = rg < tail_half;
      const uint32_t toff = has_tail ? token_piece(tok[8]) : 0u;
      constexpr uint32_t KSTEP = pairk::BK / 8;  // a k-block in 16-byte units
      for (int kb = 0; kb < KB; ++kb) {
        bool got = true;
        if (lane == 0) got = mbar_wait_spin(&empty[s], ph ^ 1u, kWaitLimitNs);
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          ok = false;
          break;
        }
        const uint32_t dst = smem_u32(sA + s * pairk::A_BYTES) + swz;
#pragma unroll
        for (int j = 0; j < 8; ++j)
          if (j < nj)
            cp_async16(dst + static_cast<uint32_t>((rg + 16 * j) * 128), xv + off[j] + kb * KSTEP);
        if constexpr (MERGE) {
          if (has_tail)
            cp_async16(smem_u32(sT + s * S::T_BYTES) + static_cast<uint32_t>(rg * 128) + swz,
                       xv + toff + kb * KSTEP);
        }
        cp_async_commit();
        ++inflight;
        if (++s == S::STAGES) {
          s = 0;
          ph ^= 1u;
        }
        if (inflight == S::STAGES - 1) {
          cp_async_wait<S::STAGES - 2>();
          release_oldest();
        }
        if (kb == 0) {
          // the next tile is already in the queue (posted one ahead): fetch
          // its row tokens now, while this tile's rows are copied
          // (every lane acquires the slot, as next_tile does)
          const bool got_next = mbar_wait_cluster(&tq_full[q_slot], q_ph, kWaitLimitNs);
          if (__all_sync(0xffffffffu, got_next)) {
            const int nt = tq[q_slot];
            if (nt < total) {
              load_tokens(pairk::decode(nt, tstart, seg, E, p.n_tiles, S::BN, p.n_tiles_m, MERGE, p.group),
                          next_tok);
              next_known = nt;
            }
          }
        }
      }
      if (!ok) break;
    }
    // every copy lands before the CTA can leave; stages still held go to the MMA
    cp_async_wait<0>();
    while (inflight > 0) release_oldest();
    if (!ok) timed_out = true;
  } else {
    // ------------------------------------------------------------ FP8 converters (A8, both CTAs)
    // Thread ct expands row ct of each staged tile: 64 E4M3 bytes (64-byte
    // swizzle, first half of the token slot) -> 64 bf16 (128-byte swizzle,
    // the whole slot, the layout the MMA reads). E4M3 -> f16 -> fp32 -> bf16
    // is exact. Every row is read before any is overwritten (one barrier of
    // the group's warps, which also makes a timeout a common decision). Each
    // warp then releases its rows to the MMA: an arrive on full (even CTA),
    // or (odd CTA) a 16-byte bulk copy to the even CTA whose completion is
    // counted on its full barrier, like the odd CTA's weight bytes. Issuing
    // the copy does not wait; a cluster-scope release arrive from each warp
    // cost ~0.7 us per stage (measured) and paced the whole GEMM.
    // group g = 0, 1 takes the stages s with s % 2 == g (STAGES is even, so
    // fills alternate between the groups); named barrier 1 + g
    const int cidx = static_cast<int>(threadIdx.x) - 32 * (2 + NEW);
    const int g = cidx / (32 * pairk::CONV_GROUP);
    const int ct = cidx - g * 32 * pairk::CONV_GROUP;
    const uint32_t gbar = 1u + static_cast<uint32_t>(g);
    const uint32_t leader_full = mapa_shared(smem_u32(full), 0);
    const uint32_t leader_sink = mapa_shared(smem_u32(smem + S::OFF_SINK), 0);
    const uint32_t my_sink = smem_u32(smem + S::OFF_SINK);
    constexpr uint32_t GTHREADS = 32 * pairk::CONV_GROUP;
    static_assert(S::STAGES % 2 == 0, "converter groups alternate stages");
    int s = 0;
    uint32_t ph = 0;
    for (;;) {
      const int tile = next_tile(true);
      if (!bar_and(gbar, GTHREADS, tile < total && !timed_out)) break;
      bool ok = true;
      for (int kb = 0; kb < KB; ++kb) {
        if ((s & 1) != g) {
          if (++s == S::STAGES) {
            s = 0;
            ph ^= 1u;
          }
          continue;
        }
        ok = mbar_wait_spin(&a8_full[s], ph, kWaitLimitNs);
        uint8_t* slot = sA + s * pairk::A_BYTES;
        uint4 raw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i)
          raw[i] = *reinterpret_cast<const uint4*>(slot + ct * 64 + ((i ^ ((ct >> 1) & 3)) << 4));
        if (!bar_and(gbar, GTHREADS, ok)) {
          ok = false;
          break;
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const uint8_t* b = reinterpret_cast<const uint8_t*>(&raw[i]);
          uint32_t o[8];
#pragma unroll
          for (int pp = 0; pp < 8; ++pp) {
            const __nv_fp8x2_storage_t pair = static_cast<__nv_fp8x2_storage_t>(
                b[2 * pp] | (static_cast<uint16_t>(b[2 * pp + 1]) << 8));
            const __half2_raw hr = __nv_cvt_fp8x2_to_halfraw2(pair, __NV_E4M3);
            const float2 f2 = __half22float2(*reinterpret_cast<const __half2*>(&hr));
            const __nv_bfloat162 bb = __floats2bfloat162_rn(f2.x, f2.y);
            o[pp] = *reinterpret_cast<const uint32_t*>(&bb);
          }
          *reinterpret_cast<uint4*>(slot + ct * 128 + (((2 * i) ^ (ct & 7)) << 4)) =
              make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(slot + ct * 128 + (((2 * i + 1) ^ (ct & 7)) << 4)) =
              make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_shared();
        __syncwarp();
        if (lane == 0) {
          if (rank == 0)
            mbar_arrive(&full[s]);
          else
            bulk_copy_s2cluster(leader_sink, my_sink, 16u,
                                leader_full + static_cast<uint32_t>(s * 8));
        }
        if (++s == S::STAGES) {
          s = 0;
          ph ^= 1u;
        }
      }
      if (!ok) {
        timed_out = true;
        break;
      }
    }
  }

  if (timed_out) atomicOr(p.err, kErrTimeout);
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still signal or read it
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc_pair(tmem_base, pairk::TMEM_COLS);
  }
}

}  // namespace

// ---------------------------------------------------------------- host side
// Tensor maps (declared in tmap.cuh; the weight-gradient GEMM uses them too).
namespace {
std::atomic<uint64_t> g_epi_wait_ns{kWaitLimitNs};
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

PFN_cuTensorMapEncodeTiled_v12000 get_encode() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}
}  // namespace

// 2-D bf16 map over a row-major [rows, cols] matrix, box [box_rows][box_cols]
// (box_cols * 2 bytes = 128, the swizzle span).
bool make_map_2d(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols, uint32_t box_cols,
                 uint32_t box_rows) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * 2};
  const cuuint32_t box[2] = {box_cols, box_rows};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over the row-major [rows, cols] output, box [32 rows][32 cols]:
// fp32 (128-byte rows, 128-byte swizzle) for the fp32 pass, bf16 (64-byte
// rows, 64-byte swizzle) for the SiLU pass, matching the staging blocks.
bool make_map_2d_out(CUtensorMap* m, void* base, uint64_t rows, uint64_t cols, bool f32) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols * (f32 ? 4 : 2)};
  const cuuint32_t box[2] = {32, 32};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                         2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         f32 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_64B,
                         CU_TENSOR_MAP_L2_PROMOTION_NONE, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// 2-D map over row-major E4M3 token rows [rows, cols] (bytes), box
// [128 rows][64 bytes] with the 64-byte swizzle the converters read.
bool make_map_2d_e4m3(CUtensorMap* m, const void* base, uint64_t rows, uint64_t cols) {
  auto enc = get_encode();
  if (!enc) return false;
  const cuuint64_t dims[2] = {cols, rows};
  const cuuint64_t strides[1] = {cols};
  const cuuint32_t box[2] = {64, 128};
  const cuuint32_t estr[2] = {1, 1};
  const CUresult r = enc(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void*>(base), dims,
                         strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                         CU_TENSOR_MAP_SWIZZLE_64B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                         CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

namespace {

template <int EPI, int NB, bool A8, bool BT, bool GA>
cudaError_t set_pair_smem_attr() {
  static std::once_flag once;
  static cudaError_t st = cudaSuccess;
  std::call_once(once, [] {
    st = cudaFuncSetAttribute(gemm_pair_kernel<EPI, NB, A8, BT, GA>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize,
                              pairk::smem_bytes<EPI, NB>());
  });
  return st;
}

// Clusters of two that can be resident at once (cached per device and kernel).
template <int EPI, int NB, bool A8, bool BT, bool GA>
int resident_pairs(const cudaLaunchConfig_t& lc_in, int num_sms) {
  static int cache[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return num_sms / 2;
  if (cache[dev] > 0) return cache[dev];
  cudaLaunchConfig_t lc = lc_in;
  lc.gridDim = dim3(static_cast<unsigned>(2 * (num_sms / 2)));
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<EPI, NB, A8, BT, GA>, &lc) != cudaSuccess ||
      n <= 0) {
    cudaGetLastError();
    n = num_sms / 2;
  }
  cache[dev] = n;
  return n;
}

template <int EPI, int NB, bool A8, bool BT = false, bool GA = false>
cudaError_t launch_pair(const CUtensorMap& mA, const CUtensorMap& mA8, const CUtensorMap& mB,
                        const CUtensorMap& mY, TcParams prm, int num_sms,
                        cudaStream_t s) {
  using S = pairk::Shape<NB>;
  prm.n_tiles = ceil_div(prm.N, S::BN);
  prm.n_tiles_m = ceil_div(prm.N, pairk::MT_W);
  const long long max_pt =
      static_cast<long long>(ceil_div(prm.R, pairk::BM) + prm.E) *
      static_cast<long long>(prm.n_tiles > prm.n_tiles_m ? prm.n_tiles : prm.n_tiles_m);
  cudaLaunchConfig_t lc = {};
  lc.blockDim = dim3(pairk::num_threads<EPI, NB, A8, GA>());
  lc.dynamicSmemBytes = pairk::smem_bytes<EPI, NB>();
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
  cudaError_t st = set_pair_smem_attr<EPI, NB, A8, BT, GA>();
  if (st != cudaSuccess) return st;
  // a persistent grid must fit at once: as many pairs as can be resident
  // together (a pair needs two free SMs of one GPC), not num_sms / 2
  const int resident = resident_pairs<EPI, NB, A8, BT, GA>(lc, num_sms);
  const int pairs = static_cast<int>(max_pt < resident ? max_pt : resident);
  // token tiles per group: as many as keep the group's token rows (256 rows
  // of K bf16 each) within ~48 MB of the 126 MB L2 while its weight tiles
  // stream past (an expert with fewer token tiles runs in one group, the
  // plain weight-tile-major order)
  const long long tile_bytes = static_cast<long long>(pairk::BM) * prm.K * 2;
  const long long g = (48LL << 20) / (tile_bytes > 0 ? tile_bytes : 1);
  prm.group = g < 1 ? 1 : (g > (1 << 20) ? (1 << 20) : static_cast<int>(g));
  lc.gridDim = dim3(2 * pairs);
  return cudaLaunchKernelEx(&lc, gemm_pair_kernel<EPI, NB, A8, BT, GA>, mA, mA8, mB, mY, prm);
}

// 512-feature tiles (one accumulator, epilogue exposed) pay off only for the
// SiLU pass with a long main loop and many tiles per pair (measured on
// GB300: the 16384-token d = 7168 E = 256 layer's W1 pass 8 % faster; every
// shorter or fp32-output pass slower).
int pick_nb(int epi, int R, int E, int K, int N, int num_sms) {
  if (epi != 0 || K < 4096 || N < 512) return 1;
  const long long tiles = static_cast<long long>(ceil_div(R, pairk::BM) + E) * ceil_div(N, 512);
  return tiles >= 8LL * (num_sms / 2) ? 2 : 1;
}

}  // namespace

void set_gemm_epilogue_wait_ns(uint64_t ns) { g_epi_wait_ns.store(ns == 0 ? kWaitLimitNs : ns); }

cudaError_t launch_gemm_tc(int epi, const void* A, int a_fp8, int a_rows, int a_shared, int R,
                           const void* W, int E, int K, int N, const int32_t* offsets,
                           const float* row_scale, void* out, uint32_t* err, uint32_t* tile_ctr,
                           const int32_t* gather_src, int tile_n, int num_sms, cudaStream_t s,
                           float* zout) {
  if (R == 0) return cudaSuccess;
  if (num_sms < 2 || (a_fp8 && epi != 0)) return cudaErrorInvalidValue;
  if (tile_n != 0 && tile_n != 256 && tile_n != 512) return cudaErrorInvalidValue;
  // gathered rows: bf16 token rows of x read through src, W1 pass only
  if (gather_src != nullptr && (a_fp8 || a_shared || epi != 0)) return cudaErrorInvalidValue;
  CUtensorMap mA, mA8, mB, mY;
  std::memset(&mY, 0, sizeof(mY));
  std::memset(&mA, 0, sizeof(mA));
  std::memset(&mA8, 0, sizeof(mA8));
  std::memset(&mB, 0, sizeof(mB));
  // A: token rows in [128 rows][64 k] boxes, and [8 rows][64 k] boxes for
  // merged tiles' remainders (none when the rows are gathered)
  if (a_rows <= 0) return cudaErrorInvalidValue;
  if (a_fp8) {
    // E4M3 token rows, expanded to bf16 in shared memory (no merged tiles)
    if (!make_map_2d_e4m3(&mA, A, static_cast<uint64_t>(a_rows), static_cast<uint64_t>(K)))
      return cudaErrorInvalidValue;
  } else if (gather_src == nullptr &&
             (!make_map_2d(&mA, A, static_cast<uint64_t>(a_rows), static_cast<uint64_t>(K), 64,
                           128) ||
              !make_map_2d(&mA8, A, static_cast<uint64_t>(a_rows), static_cast<uint64_t>(K), 64,
                           8))) {
    return cudaErrorInvalidValue;
  }
  // B: the weights as [E*K rows, N], [64 k][64 n] boxes
  if (!make_map_2d(&mB, W, static_cast<uint64_t>(E) * K, static_cast<uint64_t>(N), 64,
                   pairk::BK))
    return cudaErrorInvalidValue;
  // both passes write their full tiles' output rows through TMA stores
  if (!make_map_2d_out(&mY, out, static_cast<uint64_t>(R), static_cast<uint64_t>(N), epi == 1))
    return cudaErrorInvalidValue;
  TcParams prm;
  prm.gsrc = gather_src;
  prm.gx = gather_src != nullptr ? A : nullptr;
  prm.gx_rows = a_rows;
  prm.offsets = offsets;
  prm.row_scale = row_scale;
  prm.zin = nullptr;
  prm.zout = epi == 0 ? zout : nullptr;
  prm.out = out;
  prm.err = err;
  prm.tile_ctr = tile_ctr;
  prm.E = E;
  prm.K = K;
  prm.N = N;
  prm.R = R;
  prm.n_tiles = 0;
  prm.a_rows = a_rows;
  prm.a_shared = a_shared;
  prm.k_wrap = K;
  prm.epi_wait_ns = g_epi_wait_ns.load();
  // tile_n 256 or 512 forces the pair-tile width; 0 takes the built-in choice
  const int nb = tile_n == 0 ? pick_nb(epi, R, E, K, N, num_sms) : tile_n / 256;
  if (a_fp8) return launch_pair<0, 1, true>(mA, mA8, mB, mY, prm, num_sms, s);
  if (gather_src != nullptr)
    return nb == 2 ? launch_pair<0, 2, false, false, true>(mA, mA8, mB, mY, prm, num_sms, s)
                   : launch_pair<0, 1, false, false, true>(mA, mA8, mB, mY, prm, num_sms, s);
  if (epi == 0)
    return nb == 2 ? launch_pair<0, 2, false>(mA, mA8, mB, mY, prm, num_sms, s)
                   : launch_pair<0, 1, false>(mA, mA8, mB, mY, prm, num_sms, s);
  return nb == 2 ? launch_pair<1, 2, false>(mA, mA8, mB, mY, prm, num_sms, s)
                 : launch_pair<1, 1, false>(mA, mA8, mB, mY, prm, num_sms, s);
}

cudaError_t launch_gemm_tc_wt(const void* A, int R, const void* Wt, int E, int K, int k_wrap,
                              int N, const int32_t* offsets, const float* zin, void* out,
                              uint32_t* err, uint32_t* tile_ctr, int num_sms, cudaStream_t s,
                              const float* row_scale, int a_rows, int a_shared) {
  if (R == 0) return cudaSuccess;
  if (a_rows < 0) a_rows = R;
  if (a_rows == 0) return cudaErrorInvalidValue;
  if (num_sms < 2 || k_wrap <= 0 || k_wrap % 64 != 0 || K % k_wrap != 0 || N % 8 != 0)
    return cudaErrorInvalidValue;
  CUtensorMap mA, mA8, mB, mY;
  std::memset(&mA, 0, sizeof(mA));
  std::memset(&mA8, 0, sizeof(mA8));
  std::memset(&mB, 0, sizeof(mB));
  std::memset(&mY, 0, sizeof(mY));
  // A: [R, K] rows in [128][64] boxes (and [8][64] for merged remainders);
  // weights: the stored [E N, k_wrap] matrix in [128 features][64 k] boxes
  if (!make_map_2d(&mA, A, static_cast<uint64_t>(a_rows), static_cast<uint64_t>(K), 64, 128) ||
      !make_map_2d(&mA8, A, static_cast<uint64_t>(a_rows), static_cast<uint64_t>(K), 64, 8) ||
      !make_map_2d(&mB, Wt, static_cast<uint64_t>(E) * N, static_cast<uint64_t>(k_wrap), 64, 128) ||
      !make_map_2d_out(&mY, out, static_cast<uint64_t>(R),
                       static_cast<uint64_t>(zin ? 2 * N : N), zin == nullptr))
    return cudaErrorInvalidValue;
  TcParams prm;
  prm.gsrc = nullptr;
  prm.gx = nullptr;
  prm.gx_rows = 0;
  prm.offsets = offsets;
  prm.row_scale = zin ? row_scale : nullptr;
  prm.zin = zin;
  prm.zout = nullptr;
  prm.out = out;
  prm.err = err;
  prm.tile_ctr = tile_ctr;
  prm.E = E;
  prm.K = K;
  prm.N = N;
  prm.R = R;
  prm.n_tiles = 0;
  prm.a_rows = a_rows;
  prm.a_shared = a_shared;
  prm.k_wrap = k_wrap;
  prm.epi_wait_ns = g_epi_wait_ns.load();
  return zin ? launch_pair<2, 1, false, true>(mA, mA8, mB, mY, prm, num_sms, s)
             : launch_pair<1, 1, false, true>(mA, mA8, mB, mY, prm, num_sms, s);
}

}  // namespace moe
