// moe_abi.cu - the exported C ABI (include/moe.h): host-side validation,
// workspace layout, and the launch sequence of each stage. No entry point
// allocates, frees or synchronises (except moe_get_device_error).
#include <cfloat>
#include <climits>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "common.cuh"
#include "moe.h"

namespace moe {
namespace {

constexpr size_t kAlign = 256;

bool aligned(const void* p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

int check_cfg(const moe_config_t* c) {
  if (c == nullptr) return MOE_ERR_INVALID_ARG;
  if (c->T < 0 || c->d <= 0 || c->f <= 0 || c->E < 1 || c->k < 1) return MOE_ERR_INVALID_ARG;
  if (c->d % 64 != 0 || c->f % 64 != 0) return MOE_ERR_INVALID_ARG;
  if (c->E > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (c->dtype != MOE_DTYPE_F32 && c->dtype != MOE_DTYPE_BF16) return MOE_ERR_INVALID_ARG;
  if (c->router < MOE_ROUTER_RENORM || c->router > MOE_ROUTER_SOFT_GUMBEL)
    return MOE_ERR_INVALID_ARG;
  if (c->router == MOE_ROUTER_GROUP_LIMITED) {
    if (c->n_group < 1 || c->n_group > kMaxGroups || c->E % c->n_group != 0)
      return MOE_ERR_INVALID_ARG;
    if (c->topk_group < 1 || c->topk_group > c->n_group) return MOE_ERR_INVALID_ARG;
    if (c->k > c->topk_group * (c->E / c->n_group)) return MOE_ERR_INVALID_ARG;
  }
  if (c->payload_fp8 < 0 || c->payload_fp8 > 2) return MOE_ERR_INVALID_ARG;
  if (c->output_fp8 != 0 && c->output_fp8 != 1) return MOE_ERR_INVALID_ARG;
  if (c->payload_fp8 == 2 && !(c->payload_scale > 0.f && c->payload_scale <= FLT_MAX))
    return MOE_ERR_INVALID_ARG;
  const int max_pre = c->E < kMaxTopK ? c->E : kMaxTopK;
  if (c->pre_k < 1 || c->pre_k > max_pre) return MOE_ERR_INVALID_ARG;
  if (c->router == MOE_ROUTER_SOFT_GUMBEL) {
    // every expert weighted: k = E rows per token, up to kMaxFanout
    if (c->k != c->E || c->E > kMaxFanout) return MOE_ERR_INVALID_ARG;
    if (!(c->tau > 0.f && c->tau <= FLT_MAX)) return MOE_ERR_INVALID_ARG;
    if (c->payload_fp8) return MOE_ERR_UNSUPPORTED;  // the GEMM reads x itself
  } else if (c->k > c->pre_k) {
    return MOE_ERR_INVALID_ARG;
  }
  if (c->payload_fp8 && c->dtype != MOE_DTYPE_BF16) return MOE_ERR_UNSUPPORTED;
  if (c->d > 65536 || c->f > 65536) return MOE_ERR_UNSUPPORTED;
  if (static_cast<long long>(c->T) * c->k > INT_MAX) return MOE_ERR_UNSUPPORTED;
  if (c->gemm_tile_n != 0 && c->gemm_tile_n != 256 && c->gemm_tile_n != 512)
    return MOE_ERR_INVALID_ARG;
  if (c->x_perm_mode < MOE_XPERM_AUTO || c->x_perm_mode > MOE_XPERM_GATHERED)
    return MOE_ERR_INVALID_ARG;
  if (c->keep_z != 0 && c->keep_z != 1) return MOE_ERR_INVALID_ARG;
  // Z is kept for the backward, which the FP8 payloads do not have
  if (c->keep_z && (c->payload_fp8 || c->output_fp8)) return MOE_ERR_UNSUPPORTED;
  // gathered rows: bf16 rows of x, no FP8 payload, not soft gating (which
  // reads x itself already)
  if (c->x_perm_mode == MOE_XPERM_GATHERED &&
      (c->dtype != MOE_DTYPE_BF16 || c->payload_fp8 || c->router == MOE_ROUTER_SOFT_GUMBEL))
    return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

size_t elem_size(int dtype) { return dtype == MOE_DTYPE_F32 ? 4 : 2; }

bool soft(const moe_config_t& c) { return c.router == MOE_ROUTER_SOFT_GUMBEL; }

// moe_forward's W1 GEMM gathers the routed rows from x through src (the
// packed rows x_perm are not written): asked for, or the library's choice
// for bf16 layers without an FP8 payload or soft gating whose packed rows
// would not stay in L2. Packing costs a write of R d bf16 values and their
// read back from wherever they sit; gathering costs the W1 GEMM some speed
// (its copies are issued by threads). Measured on GB300: the 256-expert
// top-8 layer (1.9 GB of packed rows) forwards in 6.86 ms gathered against
// 7.02 ms packed; layers whose 16-67 MB of packed rows stay in L2 were 4-7 %
// slower gathered.
constexpr size_t kGatherMinPackedBytes = size_t(256) << 20;
bool gathers(const moe_config_t& c) {
  if (c.dtype != MOE_DTYPE_BF16 || c.payload_fp8 || soft(c)) return false;
  const size_t packed = static_cast<size_t>(c.T) * c.k * c.d * 2;
  return c.x_perm_mode == MOE_XPERM_GATHERED ||
         (c.x_perm_mode == MOE_XPERM_AUTO && packed >= kGatherMinPackedBytes);
}

struct Layout {
  size_t err, hist, base, scratch_end;
  size_t topk_idx, topk_w, counts, offsets, pos, src, x_perm, x_scale, h, y, y_q, y_scale,
      y_zero, z, total;
  int nchunk;
};

Layout layout_of(const moe_config_t& c) {
  Layout L;
  const size_t R = static_cast<size_t>(c.T) * c.k;
  const size_t es = elem_size(c.dtype);
  L.nchunk = ceil_div(c.T, kDispatchTokensPerChunk);
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kAlign);
    return at;
  };
  L.err = take(kAlign);
  L.hist = take(static_cast<size_t>(c.E) * L.nchunk * 4);
  L.base = take(static_cast<size_t>(c.E) * L.nchunk * 4);
  L.scratch_end = o;
  L.topk_idx = take(R * 4);
  L.topk_w = take(R * 4);
  L.counts = take(static_cast<size_t>(c.E) * 4);
  L.offsets = take(static_cast<size_t>(c.E + 1) * 4);
  L.pos = take(R * 4);
  L.src = take(R * 4);
  // soft gating: every expert reads x itself, nothing is packed; gathered
  // rows: the W1 GEMM reads x through src
  L.x_perm = take(soft(c) || gathers(c) ? 0 : R * c.d * (c.payload_fp8 ? 1 : es));
  L.x_scale = take(c.payload_fp8 ? R * 4 : 0);
  L.h = take(R * c.f * es);
  L.y = take(R * c.d * 4);
  L.y_q = take(c.output_fp8 ? R * c.d : 0);
  L.y_scale = take(c.output_fp8 ? R * 4 : 0);
  L.y_zero = take(c.output_fp8 ? R * 4 : 0);
  L.z = take(c.keep_z ? R * c.f * 4 : 0);  // the pre-activation, for a backward
  L.total = o;
  return L;
}

template <typename T>
T* at(void* ws, size_t off) {
  return reinterpret_cast<T*>(static_cast<char*>(ws) + off);
}

int num_sms() {
  static int cache[64] = {0};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64 && cache[dev] > 0) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

int status_of(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_LAUNCH; }

cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

uint32_t* gemm_counters(void* ws) { return at<uint32_t>(ws, kGemmCounterOffset); }

void record(void* const* ev, int i, cudaStream_t s) {
  if (ev != nullptr && ev[i] != nullptr) cudaEventRecord(static_cast<cudaEvent_t>(ev[i]), s);
}

// ---------------------------------------------------------------- stages
int run_route(const moe_config_t& c, const void* x, const void* Wg, const float* bias,
              const float* noise, int32_t* idx, float* w, float* logits, uint32_t* err,
              cudaStream_t s) {
  const RouterSpec rs{c.k, c.pre_k, c.router, c.n_group, c.topk_group, c.tau, noise};
  return status_of(launch_route(c.dtype, x, Wg, bias, c.T, c.d, c.E, rs, idx, w, logits, err, s));
}

int run_dispatch(const moe_config_t& c, const Layout& L, void* ws, const void* x,
                 const int32_t* idx, int32_t* counts, int32_t* offsets, int32_t* pos,
                 int32_t* src, void* x_perm, float* x_scale, cudaStream_t s) {
  if (c.T == 0) return status_of(launch_dispatch_empty(c.E, counts, offsets, s));
  if (soft(c))  // every token to every expert: the layout needs no counting
    return status_of(launch_dense_layout(c.T, c.E, counts, offsets, pos, src, gemm_counters(ws),
                                         kNumGemmCounters, s));
  uint32_t* err = at<uint32_t>(ws, L.err);
  if (static_cast<long long>(c.T) * c.k <= kDispatchFusedMaxRows)
    return status_of(launch_dispatch_fused(
        c.dtype, c.payload_fp8 != 0, c.payload_fp8 == 2 ? c.payload_scale : 0.f, x, idx, c.T, c.d,
        c.k, c.E, counts, offsets, pos, src, x_perm, x_scale, err, gemm_counters(ws),
        kNumGemmCounters, s));
  int32_t* hist = at<int32_t>(ws, L.hist);
  int32_t* base = at<int32_t>(ws, L.base);
  // the count kernel also zeroes the GEMM tile counters for the layer
  cudaError_t e = launch_dispatch_count(idx, c.T, c.k, c.E, L.nchunk, hist, err,
                                        gemm_counters(ws), kNumGemmCounters, s);
  if (e == cudaSuccess) e = launch_dispatch_scan(hist, L.nchunk, c.E, base, counts, s);
  if (e == cudaSuccess)
    e = launch_dispatch_scatter(c.dtype, c.payload_fp8 != 0,
                                c.payload_fp8 == 2 ? c.payload_scale : 0.f, x, idx, c.T, c.d,
                                c.k, c.E, L.nchunk, counts, base, offsets, pos, src, x_perm,
                                x_scale, err, s);
  return status_of(e);
}

// which 1: the W1 pass, reading x_perm, or (gather_src non-null) x itself
// through the routed rows' tokens, and writing the pre-activation to zout
// too when it is non-null; which 2: the W2 pass.
int run_gemm(const moe_config_t& c, const Layout& L, void* ws, int which, const void* x_perm,
             const float* x_scale, const int32_t* offsets, const void* W1, const void* W2,
             void* h, float* y, cudaStream_t s, const int32_t* gather_src = nullptr,
             float* zout = nullptr) {
  const int R = c.T * c.k;
  if (R == 0) return MOE_OK;
  uint32_t* err = at<uint32_t>(ws, L.err);
  if (c.dtype == MOE_DTYPE_F32) {
    if (which == 1)
      return status_of(launch_gemm_simt(0, static_cast<const float*>(x_perm), soft(c) ? 1 : 0, R,
                                        static_cast<const float*>(W1), c.E, c.d, c.f, offsets,
                                        static_cast<float*>(h), err, s, zout));
    return status_of(launch_gemm_simt(1, static_cast<const float*>(h), 0, R,
                                      static_cast<const float*>(W2), c.E, c.f, c.d, offsets, y,
                                      err, s));
  }
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_LAUNCH;
  uint32_t* ctr = gemm_counters(ws) + (which - 1);
  if (which == 1) {
    // soft gating: x_perm is x itself, [T, d], read by every expert; the
    // FP8 payload is expanded to bf16 inside the GEMM (its prologue);
    // gathered rows: x_perm is x, [T, d], row r of the layout reads x[src[r]]
    return status_of(launch_gemm_tc(0, x_perm, c.payload_fp8 ? 1 : 0,
                                    soft(c) || gather_src ? c.T : R, soft(c) ? 1 : 0, R, W1, c.E,
                                    c.d, c.f, offsets, c.payload_fp8 ? x_scale : nullptr, h, err,
                                    ctr, gather_src, c.gemm_tile_n, sms, s, zout));
  }
  return status_of(launch_gemm_tc(1, h, 0, R, 0, R, W2, c.E, c.f, c.d, offsets, nullptr, y, err,
                                  ctr, nullptr, c.gemm_tile_n, sms, s));
}

int run_combine(const moe_config_t& c, const Layout& L, void* ws, const float* y,
                const int32_t* pos, const float* w, void* out, cudaStream_t s) {
  return status_of(launch_combine(c.dtype, y, pos, w, c.T, c.d, c.k, c.T * c.k, out,
                                  at<uint32_t>(ws, L.err), s));
}

bool ok_ptr(const void* p) { return p != nullptr && aligned(p, 16); }

int forward_impl(const moe_config_t* cfg, const void* x, const void* Wg, const float* bias,
                 const float* noise, const void* W1, const void* W2, void* out, void* ws,
                 size_t ws_bytes, void* const* events, void* stream) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_config_t& c = *cfg;
  if (!ok_ptr(x) || Wg == nullptr || !ok_ptr(W1) || !ok_ptr(W2) || !ok_ptr(out) ||
      ws == nullptr || !aligned(ws, kAlign) || (soft(c) && c.T > 0 && noise == nullptr))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(c);
  if (ws_bytes < L.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_stream(stream);
  int32_t* idx = at<int32_t>(ws, L.topk_idx);
  float* w = at<float>(ws, L.topk_w);
  int32_t* counts = at<int32_t>(ws, L.counts);
  int32_t* offsets = at<int32_t>(ws, L.offsets);
  int32_t* pos = at<int32_t>(ws, L.pos);
  int32_t* src = at<int32_t>(ws, L.src);
  // soft gating packs nothing: the W1 GEMM reads x for every expert; with
  // gathered rows the dispatch writes only the layout and the W1 GEMM reads
  // each routed row from x through src
  const bool ga = gathers(c);
  void* x_perm = soft(c) ? const_cast<void*>(x) : (ga ? nullptr : at<void>(ws, L.x_perm));
  float* x_scale = c.payload_fp8 ? at<float>(ws, L.x_scale) : nullptr;
  void* h = at<void>(ws, L.h);
  float* y = at<float>(ws, L.y);

  record(events, 0, s);
  if ((st = run_route(c, x, Wg, bias, noise, idx, w, nullptr, at<uint32_t>(ws, L.err), s)) !=
      MOE_OK)
    return st;
  record(events, 1, s);
  if ((st = run_dispatch(c, L, ws, x, idx, counts, offsets, pos, src, x_perm, x_scale, s)) !=
      MOE_OK)
    return st;
  record(events, 2, s);
  record(events, 3, s);  // (no kernel: the FP8 payload is expanded inside the W1 GEMM)
  // keep_z: the W1 pass also leaves the pre-activation Z in the workspace
  if ((st = run_gemm(c, L, ws, 1, ga ? x : x_perm, x_scale, offsets, W1, W2, h, y, s,
                     ga ? src : nullptr, c.keep_z ? at<float>(ws, L.z) : nullptr)) != MOE_OK)
    return st;
  record(events, 4, s);
  if ((st = run_gemm(c, L, ws, 2, x_perm, x_scale, offsets, W1, W2, h, y, s)) != MOE_OK)
    return st;
  record(events, 5, s);
  if (c.output_fp8) {
    uint8_t* yq = at<uint8_t>(ws, L.y_q);
    float* ys = at<float>(ws, L.y_scale);
    float* yz = at<float>(ws, L.y_zero);
    if ((st = status_of(launch_quantize_out(y, c.T * c.k, c.d, yq, ys, yz, s))) != MOE_OK)
      return st;
    record(events, 6, s);
    st = status_of(launch_combine_fp8(c.dtype, yq, ys, yz, pos, w, c.T, c.d, c.k, c.T * c.k, out,
                                      at<uint32_t>(ws, L.err), s));
    if (st != MOE_OK) return st;
  } else {
    record(events, 6, s);
    if ((st = run_combine(c, L, ws, y, pos, w, out, s)) != MOE_OK) return st;
  }
  record(events, 7, s);
  return MOE_OK;
}

// ---------------------------------------------------------------- backward
// The backward workspace: an error word and the GEMM tile counters, then the
// recomputed logits (and the route call's unused top-k), dw, dL, the single
// segment {0, T} of the gate GEMMs, dY (fp32 layers), the recomputed
// pre-activation Z (fp32 layers overwrite it with dZ; with keep_z, bf16
// layers read the forward's and fp32 layers copy it), dX_perm and the gate
// part of dx, all fp32 but the ints; bf16 layers add the tensor-core GEMMs'
// operands: the bf16 splits of dY (or, when 2f <= d, of w H: per routed row
// its routing weight times its H row), dZ and dL, and per routed row its
// token's dout row (hard routers) and its routing weight.
// bf16 layers: dW2 takes the routing weight on its H side, splitting w H
// ([R][2f]) instead of dY ([R][2d]), where that operand is at most half as
// wide (measured on GB300, same box: 256-expert layer, d = 3.5 f, backward
// 25.36 -> 24.67 ms; the balanced and 64-expert layers, f > d / 2, were
// 1.32 -> 1.36 and 1.02 -> 1.04 ms the other way)
bool split_h(const moe_config_t& c) { return 2 * static_cast<long long>(c.f) <= c.d; }

struct BwdLayout {
  size_t err, L, ridx, rw, dw, dL, seg01, segk, bpart, gpart, dY, Z, dXp, dxg, dYs, hs, dZs, dLs,
      doutp, wr, xp, total;
};

// Token chunks of the gate's weight gradient (split along T so that its few
// output tiles fill the GPU; the chunks' partial sums are added in chunk
// order) and of the bias gradient's partial sums.
// At most kTokChunks chunks, one per 64 tokens, and as many as 128 clusters
// of two CTAs need (the cap the workspace is sized for; GB300 has 76).
constexpr int kTokChunks = 32;
constexpr int kMaxClusters = 128;
int max_tok_chunks(const moe_config_t& c) {
  const int tiles = ceil_div(c.d, 256) * ceil_div(c.E, 256);
  int n = ceil_div(kMaxClusters, tiles);
  const int by_rows = ceil_div(c.T > 0 ? c.T : 1, 64);
  n = n < by_rows ? n : by_rows;
  return n < 1 ? 1 : (n > kTokChunks ? kTokChunks : n);
}
struct TokChunks {
  int n, len;
};
TokChunks tok_chunks(const moe_config_t& c, int sms) {
  const int tiles = ceil_div(c.d, 256) * ceil_div(c.E, 256);
  const int cap = max_tok_chunks(c);
  int n = ceil_div(sms / 2 > 0 ? sms / 2 : 1, tiles);
  n = n < 1 ? 1 : (n > cap ? cap : n);
  const int len = (ceil_div(c.T > 0 ? c.T : 1, n) + 63) / 64 * 64;
  return {ceil_div(c.T > 0 ? c.T : 1, len), len};  // <= n chunks
}

BwdLayout bwd_layout_of(const moe_config_t& c) {
  BwdLayout B;
  const size_t R = static_cast<size_t>(c.T) * c.k, T = c.T, E = c.E;
  size_t o = 0;
  auto take = [&](size_t bytes) {
    const size_t at = o;
    o = align_up(o + bytes, kAlign);
    return at;
  };
  B.err = take(kAlign);
  B.L = take(T * E * 4);
  B.ridx = take(R * 4);
  B.rw = take(R * 4);
  B.dw = take(R * 4);
  B.dL = take(T * E * 4);
  B.seg01 = take(8);
  const bool tc = c.dtype == MOE_DTYPE_BF16;
  const size_t nch = static_cast<size_t>(max_tok_chunks(c));
  B.segk = take((kTokChunks + 1) * 4);
  B.bpart = take(nch * E * 4);
  B.gpart = take(tc ? nch * E * static_cast<size_t>(c.d) * 4 : 0);
  B.dY = take(tc ? 0 : R * c.d * 4);  // fp32 layers (bf16 ones keep only the split)
  // Z: recomputed here, or kept by the forward (keep_z) and read there;
  // fp32 layers turn it into dZ in place, so they always hold a copy
  B.Z = take(c.keep_z && tc ? 0 : R * c.f * 4);
  B.dXp = take(R * c.d * 4);
  B.dxg = take(T * c.d * 4);
  B.dYs = take(tc && !split_h(c) ? R * 2 * c.d * 2 : 0);
  B.hs = take(tc && split_h(c) ? R * 2 * c.f * 2 : 0);
  B.dZs = take(tc ? R * 2 * c.f * 2 : 0);
  B.dLs = take(tc ? T * 2 * E * 2 : 0);
  B.doutp = take(tc && !soft(c) ? R * c.d * 2 : 0);
  B.wr = take(tc ? R * 4 : 0);
  // the packed rows, when the forward gathered them instead of writing them
  B.xp = take(gathers(c) ? R * c.d * 2 : 0);
  B.total = o;
  return B;
}

int backward_impl(const moe_config_t* cfg, const void* x, const void* Wg, const float* bias,
                  const float* noise, const void* W1, const void* W2, const void* fwd_ws,
                  size_t fwd_ws_bytes, const void* dout, float* dx, float* dWg, float* dbias,
                  float* dW1, float* dW2, void* bws, size_t bws_bytes, void* stream) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  const moe_config_t& c = *cfg;
  if (c.payload_fp8 || c.output_fp8) return MOE_ERR_UNSUPPORTED;
  // tensors read or written in 16-byte pieces or by TMA: 16-byte aligned
  if (!ok_ptr(x) || !ok_ptr(Wg) || !ok_ptr(W1) || !ok_ptr(W2) || fwd_ws == nullptr ||
      !aligned(fwd_ws, kAlign) || !ok_ptr(dout) || !ok_ptr(dx) || !ok_ptr(dWg) ||
      !ok_ptr(dW1) || !ok_ptr(dW2) || bws == nullptr || !aligned(bws, kAlign) ||
      (soft(c) && c.T > 0 && noise == nullptr))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(c);
  const BwdLayout B = bwd_layout_of(c);
  if (fwd_ws_bytes < L.total || bws_bytes < B.total) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_stream(stream);
  const int T = c.T, d = c.d, E = c.E, k = c.k, f = c.f, R = c.T * c.k;
  void* fws = const_cast<void*>(fwd_ws);
  const int32_t* idx = at<int32_t>(fws, L.topk_idx);
  const float* w = at<float>(fws, L.topk_w);
  const int32_t* offsets = at<int32_t>(fws, L.offsets);
  const int32_t* pos = at<int32_t>(fws, L.pos);
  // the packed rows: the forward's, or (gathered forward) packed here from x
  // through the forward's src
  const void* x_perm = soft(c) ? x : (gathers(c) ? at<void>(bws, B.xp) : at<void>(fws, L.x_perm));
  const void* h = at<void>(fws, L.h);
  const float* y = at<float>(fws, L.y);
  uint32_t* err = at<uint32_t>(bws, B.err);
  float* Lr = at<float>(bws, B.L);
  float* dw = at<float>(bws, B.dw);
  float* dL = at<float>(bws, B.dL);
  int32_t* seg01 = at<int32_t>(bws, B.seg01);
  float* dY = at<float>(bws, B.dY);
  // keep_z: the forward left Z in its workspace (read-only here)
  const bool kept = c.keep_z != 0;
  float* Z = kept && c.dtype == MOE_DTYPE_BF16 ? at<float>(fws, L.z) : at<float>(bws, B.Z);
  float* dXp = at<float>(bws, B.dXp);
  float* dxg = at<float>(bws, B.dxg);
  const int dt = c.dtype;
  if (T == 0) {
    // no tokens: every gradient is zero
    cudaError_t e = cudaMemsetAsync(dWg, 0, static_cast<size_t>(d) * E * 4, s);
    if (e == cudaSuccess && dbias) e = cudaMemsetAsync(dbias, 0, static_cast<size_t>(E) * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW1, 0, static_cast<size_t>(E) * d * f * 4, s);
    if (e == cudaSuccess) e = cudaMemsetAsync(dW2, 0, static_cast<size_t>(E) * f * d * 4, s);
    return status_of(e);
  }
  // the logits, recomputed by the forward's own gate kernel (bit for bit)
  if ((st = run_route(c, x, Wg, bias, noise, at<int32_t>(bws, B.ridx), at<float>(bws, B.rw), Lr,
                      err, s)) != MOE_OK)
    return st;
  const bool tc = dt == MOE_DTYPE_BF16;
  const int sms = num_sms();
  if (sms <= 0) return MOE_ERR_LAUNCH;
  const TokChunks ch = tok_chunks(c, sms);
  int32_t* segk = at<int32_t>(bws, B.segk);
  uint32_t* ctr = at<uint32_t>(bws, kGemmCounterOffset);  // four tile counters
  // (gathered forward) the packed rows dW1 reads, written token by token
  // through the forward's layout: each x row read once, written k times
  cudaError_t e = gathers(c) ? launch_scatter_rows(dt, x, pos, T, k, d, at<void>(bws, B.xp), s)
                             : cudaSuccess;
  if (e == cudaSuccess)
    e = launch_combine_bwd(dt, dout, y, pos, w, T, d, k, R, tc ? nullptr : dY,
                           tc && !split_h(c) ? at<void>(bws, B.dYs) : nullptr,
                           tc && split_h(c) ? h : nullptr, f,
                           tc && split_h(c) ? at<void>(bws, B.hs) : nullptr,
                           tc && !soft(c) ? at<void>(bws, B.doutp) : nullptr,
                           tc ? at<float>(bws, B.wr) : nullptr, dw, err, ctr, 4, seg01, segk,
                           ch.n, ch.len, s);
  void* dLs = tc ? at<void>(bws, B.dLs) : nullptr;
  if (e == cudaSuccess)
    e = launch_router_bwd(Lr, idx, w, dw, T, E, k, c.router, c.pre_k, c.tau, dL, dLs, s);
  // gate: dx_gate = dL W_g^T ([T, E] x [E, d]), dW_g = x^T dL, db = sum_t dL.
  // bf16 layers put them on the tensor cores with dL split into hi + lo
  // (dx_gate: W_g read K-major, K = E a multiple of 64; dW_g: E a multiple
  // of 8), else fp32 FMA.
  if (e == cudaSuccess)
    e = tc && E % 64 == 0 ? launch_gemm_tc_wt(dLs, T, Wg, 1, 2 * E, E, d, seg01, nullptr, dxg,
                                              err, ctr + 3, sms, s)
                          : launch_gemm_nt(dt, false, dL, Wg, 1, T, E, d, seg01, dxg, err, s);
  // dW_g on the tensor cores: one partial per token chunk (the chunks are
  // the "experts" of the weight-gradient GEMM), then summed in chunk order
  const bool wg_tc = tc && E % 8 == 0;
  const int wg_parts = wg_tc && ch.n > 1 ? ch.n : 0;
  float* gpart = at<float>(bws, B.gpart);
  if (e == cudaSuccess)
    e = wg_tc ? launch_wgrad_tc(x, T, 0, dLs, T, ch.n, d, E, segk, wg_parts ? gpart : dWg, err,
                                sms, s)
              : launch_gemm_tn(dt, x, 0, dL, 1, T, d, E, seg01, dWg, err, s);
  // db: partial sums per token chunk, then the same ordered sum
  const int b_parts = dbias != nullptr && ch.n > 1 ? ch.n : 0;
  float* bpart = at<float>(bws, B.bpart);
  if (e == cudaSuccess && dbias != nullptr)
    e = launch_bias_bwd(dL, T, E, ch.len, ch.n, b_parts ? bpart : dbias, s);
  if (e == cudaSuccess)
    e = launch_reduce_partials(gpart, wg_parts, static_cast<size_t>(d) * E, dWg, bpart, b_parts,
                               static_cast<size_t>(E), dbias, s);
  // experts: Z = X_e W1_e again (fp32; with keep_z the forward's), dZ =
  // (dY W2_e^T) * SiLU'(Z) over Z,
  // dW2 = H^T dY, dW1 = X^T dZ, dX_perm = dZ W1_e^T. bf16 layers run every
  // expert GEMM on the tensor cores (dY and dZ split into bf16 hi + lo; for
  // the dgrad GEMMs the weights transposed and stacked twice along K); fp32
  // layers run them in fp32 FMA.
  if (e == cudaSuccess) {
    if (!tc) {
      e = kept ? cudaMemcpyAsync(Z, at<float>(fws, L.z), static_cast<size_t>(R) * f * 4,
                                 cudaMemcpyDeviceToDevice, s)
               : launch_gemm_simt(1, static_cast<const float*>(x_perm), soft(c) ? 1 : 0, R,
                                  static_cast<const float*>(W1), E, d, f, offsets, Z, err, s);
    } else {
      if (!kept)
        e = launch_gemm_tc(1, x_perm, 0, soft(c) ? T : R, soft(c) ? 1 : 0, R, W1, E, d, f,
                           offsets, nullptr, Z, err, ctr, nullptr, c.gemm_tile_n, sms, s);
      // dH[r] = w_r (dout[t(r)] . W2_e^T): row r's routing weight comes out of
      // the sum, so the GEMM reads the exact bf16 dout rows (K = d; soft
      // gating: dout itself, every expert reading all T rows) and its
      // epilogue scales by w_r and writes the split of dZ = dH * SiLU'(Z);
      // dX_perm = [dZ hi | dZ lo] . [W1_e^T ; W1_e^T]: the stored weights
      // read K-major, K = 2f wrapping at f
      if (e == cudaSuccess)
        e = launch_gemm_tc_wt(soft(c) ? dout : at<void>(bws, B.doutp), R, W2, E, d, d, f,
                              offsets, Z, at<void>(bws, B.dZs), err, ctr + 1, sms, s,
                              at<float>(bws, B.wr), soft(c) ? T : R, soft(c) ? 1 : 0);
      if (e == cudaSuccess)
        e = launch_gemm_tc_wt(at<void>(bws, B.dZs), R, W1, E, 2 * f, f, d, offsets, nullptr, dXp,
                              err, ctr + 2, sms, s);
    }
  }
  if (e == cudaSuccess && tc) {
    // weight gradients on the tensor cores, contracted over each expert's
    // rows: dW2 = sum_r H_r^T dY_r with dY_r = w_r dout[t(r)]: H^T (dY hi +
    // lo), or, when 2f <= d, (w H hi + lo)^T . the bf16 dout rows (the split
    // on the narrower operand; soft gating: dout itself, every expert
    // reading all T rows); dW1 = X^T (dZ hi + lo)
    e = split_h(c) ? launch_wgrad_tc_split_a(at<void>(bws, B.hs), R,
                                             soft(c) ? dout : at<void>(bws, B.doutp),
                                             soft(c) ? T : R, soft(c) ? 1 : 0, E, f, d, offsets,
                                             dW2, err, sms, s)
                   : launch_wgrad_tc(h, R, 0, at<void>(bws, B.dYs), R, E, f, d, offsets, dW2, err,
                                     sms, s);
    if (e == cudaSuccess)
      e = launch_wgrad_tc(x_perm, soft(c) ? T : R, soft(c) ? 1 : 0, at<void>(bws, B.dZs), R, E, d,
                          f, offsets, dW1, err, sms, s);
  }
  if (e == cudaSuccess && !tc) {
    e = launch_gemm_nt(dt, true, dY, W2, E, R, d, f, offsets, Z, err, s);
    if (e == cudaSuccess) e = launch_gemm_tn(dt, h, 0, dY, E, R, f, d, offsets, dW2, err, s);
    if (e == cudaSuccess)
      e = launch_gemm_tn(dt, x_perm, soft(c) ? 1 : 0, Z, E, R, d, f, offsets, dW1, err, s);
    if (e == cudaSuccess) e = launch_gemm_nt(dt, false, Z, W1, E, R, f, d, offsets, dXp, err, s);
  }
  if (e == cudaSuccess) e = launch_undispatch(dxg, dXp, pos, T, d, k, R, dx, s);
  return status_of(e);
}

}  // namespace
}  // namespace moe

using namespace moe;

extern "C" {

int moe_check_config(const moe_config_t* cfg) { return check_cfg(cfg); }

int moe_set_gemm_epilogue_wait_ns(uint64_t ns) {
  set_gemm_epilogue_wait_ns(ns);
  return MOE_OK;
}

size_t moe_scratch_size(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return layout_of(*cfg).scratch_end;
}

size_t moe_workspace_size(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return layout_of(*cfg).total;
}

int moe_route(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
              const float* noise, int32_t* topk_idx, float* topk_w, float* logits,
              void* stream) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(x) || W_g == nullptr || topk_idx == nullptr || topk_w == nullptr ||
      (soft(*cfg) && noise == nullptr))
    return MOE_ERR_INVALID_ARG;
  return run_route(*cfg, x, W_g, bias, noise, topk_idx, topk_w, logits, nullptr,
                   as_stream(stream));
}

int moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                 int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src, void* x_perm,
                 float* x_scale, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (counts == nullptr || offsets == nullptr || ws == nullptr || !aligned(ws, kAlign))
    return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (pos == nullptr || src == nullptr ||
                     (!soft(*cfg) && (!ok_ptr(x) || topk_idx == nullptr || !ok_ptr(x_perm) ||
                                      (cfg->payload_fp8 && x_scale == nullptr)))))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  if (ws_bytes < L.scratch_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return run_dispatch(*cfg, L, ws, x, topk_idx, counts, offsets, pos, src, x_perm, x_scale,
                      as_stream(stream));
}

int moe_expert_ffn(const moe_config_t* cfg, const void* x_perm, const float* x_scale,
                   const int32_t* offsets, const void* W1, const void* W2, void* h,
                   float* y_perm, void* ws, size_t ws_bytes, void* stream) {
  int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (ws == nullptr || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 &&
      (!ok_ptr(x_perm) || offsets == nullptr || !ok_ptr(W1) || !ok_ptr(W2) || !ok_ptr(h) ||
       !ok_ptr(y_perm) || (cfg->payload_fp8 && x_scale == nullptr)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  if (ws_bytes < L.scratch_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  cudaStream_t s = as_stream(stream);
  if (cfg->T > 0 && cudaMemsetAsync(gemm_counters(ws), 0, kNumGemmCounters * sizeof(uint32_t),
                                    s) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  if ((st = run_gemm(*cfg, L, ws, 1, x_perm, x_scale, offsets, W1, W2, h, y_perm, s)) != MOE_OK)
    return st;
  return run_gemm(*cfg, L, ws, 2, x_perm, x_scale, offsets, W1, W2, h, y_perm, s);
}

int moe_combine(const moe_config_t* cfg, const float* y_perm, const int32_t* pos,
                const float* topk_w, void* out, void* ws, size_t ws_bytes, void* stream) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (ws == nullptr || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!ok_ptr(y_perm) || pos == nullptr || topk_w == nullptr || !ok_ptr(out)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  if (ws_bytes < L.scratch_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return run_combine(*cfg, L, ws, y_perm, pos, topk_w, out, as_stream(stream));
}

int moe_quantize_output(const moe_config_t* cfg, const float* y_perm, uint8_t* y_q,
                        float* y_scale, float* y_zero, void* stream) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (cfg->T == 0) return MOE_OK;
  if (!ok_ptr(y_perm) || !ok_ptr(y_q) || y_scale == nullptr || y_zero == nullptr)
    return MOE_ERR_INVALID_ARG;
  return status_of(launch_quantize_out(y_perm, cfg->T * cfg->k, cfg->d, y_q, y_scale, y_zero,
                                       as_stream(stream)));
}

int moe_combine_fp8(const moe_config_t* cfg, const uint8_t* y_q, const float* y_scale,
                    const float* y_zero, const int32_t* pos, const float* topk_w, void* out,
                    void* ws, size_t ws_bytes, void* stream) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (ws == nullptr || !aligned(ws, kAlign)) return MOE_ERR_INVALID_ARG;
  if (cfg->T > 0 && (!ok_ptr(y_q) || y_scale == nullptr || y_zero == nullptr ||
                     pos == nullptr || topk_w == nullptr || !ok_ptr(out)))
    return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  if (ws_bytes < L.scratch_end) return MOE_ERR_WORKSPACE_TOO_SMALL;
  return status_of(launch_combine_fp8(cfg->dtype, y_q, y_scale, y_zero, pos, topk_w, cfg->T,
                                      cfg->d, cfg->k, cfg->T * cfg->k, out,
                                      at<uint32_t>(ws, L.err), as_stream(stream)));
}

int moe_forward(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                const float* noise, const void* W1, const void* W2, void* out, void* ws,
                size_t ws_bytes, void* stream) {
  return forward_impl(cfg, x, W_g, bias, noise, W1, W2, out, ws, ws_bytes, nullptr, stream);
}

int moe_forward_with_events(const moe_config_t* cfg, const void* x, const void* W_g,
                            const float* bias, const float* noise, const void* W1, const void* W2,
                            void* out, void* ws, size_t ws_bytes, void* const* events,
                            int n_events, void* stream) {
  if (events != nullptr && n_events != MOE_NUM_EVENTS) return MOE_ERR_INVALID_ARG;
  return forward_impl(cfg, x, W_g, bias, noise, W1, W2, out, ws, ws_bytes, events, stream);
}

int moe_forward_views(const moe_config_t* cfg, void* ws, moe_forward_views_t* v) {
  const int st = check_cfg(cfg);
  if (st != MOE_OK) return st;
  if (ws == nullptr || v == nullptr) return MOE_ERR_INVALID_ARG;
  const Layout L = layout_of(*cfg);
  v->topk_idx = at<int32_t>(ws, L.topk_idx);
  v->topk_w = at<float>(ws, L.topk_w);
  v->counts = at<int32_t>(ws, L.counts);
  v->offsets = at<int32_t>(ws, L.offsets);
  v->pos = at<int32_t>(ws, L.pos);
  v->src = at<int32_t>(ws, L.src);
  v->x_perm = soft(*cfg) || gathers(*cfg) ? nullptr : at<void>(ws, L.x_perm);
  v->x_scale = cfg->payload_fp8 ? at<float>(ws, L.x_scale) : nullptr;
  v->h = at<void>(ws, L.h);
  v->y_perm = at<float>(ws, L.y);
  v->y_q = cfg->output_fp8 ? at<uint8_t>(ws, L.y_q) : nullptr;
  v->y_scale = cfg->output_fp8 ? at<float>(ws, L.y_scale) : nullptr;
  v->y_zero = cfg->output_fp8 ? at<float>(ws, L.y_zero) : nullptr;
  v->z = cfg->keep_z ? at<float>(ws, L.z) : nullptr;
  return MOE_OK;
}

int moe_get_device_error(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  cudaStream_t s = as_stream(stream);
  uint32_t v = 0;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_LAUNCH;
  if (cudaMemcpyAsync(&v, ws, sizeof(v), cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return MOE_ERR_LAUNCH;
  if (cudaMemsetAsync(ws, 0, sizeof(v), s) != cudaSuccess) return MOE_ERR_LAUNCH;
  if (cudaStreamSynchronize(s) != cudaSuccess) return MOE_ERR_LAUNCH;
  if (v & kErrTimeout) return MOE_ERR_TIMEOUT;
  if (v & kErrBadIndex) return MOE_ERR_BAD_INDEX;
  return MOE_OK;
}

int moe_clear_device_error(void* ws, void* stream) {
  if (ws == nullptr) return MOE_ERR_INVALID_ARG;
  return cudaMemsetAsync(ws, 0, sizeof(uint32_t), as_stream(stream)) == cudaSuccess
             ? MOE_OK
             : MOE_ERR_LAUNCH;
}

const char* moe_strerror(int status) {
  switch (status) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_UNSUPPORTED: return "unsupported configuration";
    case MOE_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MOE_ERR_LAUNCH: return "CUDA launch or runtime error";
    case MOE_ERR_BAD_INDEX: return "expert index or row position out of range (device)";
    case MOE_ERR_TIMEOUT: return "device wait timed out";
    default: return "unknown status";
  }
}

size_t moe_backward_workspace_size(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  return bwd_layout_of(*cfg).total;
}

int moe_backward(const moe_config_t* cfg, const void* x, const void* W_g, const float* bias,
                 const float* noise, const void* W1, const void* W2, const void* fwd_ws,
                 size_t fwd_ws_bytes, const void* dout, float* dx, float* dW_g, float* dbias,
                 float* dW1, float* dW2, void* ws, size_t ws_bytes, void* stream) {
  return backward_impl(cfg, x, W_g, bias, noise, W1, W2, fwd_ws, fwd_ws_bytes, dout, dx, dW_g,
                       dbias, dW1, dW2, ws, ws_bytes, stream);
}

int moe_forward_kernel_count(const moe_config_t* cfg) {
  if (check_cfg(cfg) != MOE_OK) return 0;
  if (cfg->T == 0) return 1;
  // dense layout, one fused kernel for small batches, or count + scan + scatter
  const int dispatch =
      soft(*cfg) || static_cast<long long>(cfg->T) * cfg->k <= kDispatchFusedMaxRows ? 1 : 3;
  return 1 + dispatch + 2 + (cfg->output_fp8 ? 1 : 0) + 1;
}

}  // extern "C"
