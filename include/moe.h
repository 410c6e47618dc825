/*
 * moe.h - C ABI of a routed mixture-of-experts (MoE) layer forward on one
 * NVIDIA GB300 (sm_103a).
 *
 * The layer, as the source pages describe it:
 *   gate      L = x W_g + b, one logit per expert
 *             (DeepSeek-V4 EP article, section 2.1)
 *   router    max-subtracted softmax, partial top-8, exact top-k; the lower
 *             expert id wins a tie (same article, section 3.2)
 *   dispatch  per-expert histogram, exclusive scan and a stable permutation
 *             that packs the routed rows contiguously by expert id - the
 *             single-GPU form of the expert-parallel all-to-all layout
 *             (same article, section 3.3; Deepseek-MoE sync-tax article,
 *             section 2.1), optionally as a per-token FP8 E4M3 payload
 *             (sync-tax article, section 3.1)
 *   FFN       per expert e: H = SiLU(X_e W1_e), Y = H W2_e ("L1 + Act + L2",
 *             DeepSeek V3/V4 parallel-strategy article, Waved-EP section)
 *   combine   out_t = sum_{j=0..k-1} w_tj * Y[pos(t, j)], in that order
 *             (sync-tax article, section 2.3)
 *
 * Conventions for every entry point
 * ---------------------------------
 *  - Pointers named as device pointers must point to device (or managed)
 *    memory of the current CUDA device. Host pointers are never accepted.
 *  - All tensors are dense, row-major, with no padding between rows.
 *  - Device pointers to activations, weights, payloads, H, Y and outputs must
 *    be 16-byte aligned; the workspace must be 256-byte aligned.
 *  - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *    stream). Every call is asynchronous on that stream: it only enqueues
 *    kernels, never allocates, frees or synchronises (except
 *    moe_get_device_error, which synchronises by design). The caller owns
 *    every buffer, including the workspace.
 *  - Calls return MOE_OK (0) or a negative moe_status. Argument errors are
 *    found on the host before anything is enqueued. Errors found by a kernel
 *    (an expert index or row position out of range, a device wait that ran
 *    past its bound) are recorded in the workspace's error word; the kernel
 *    skips the offending access instead of faulting. Read them with
 *    moe_get_device_error.
 *  - T = 0 is valid and produces empty outputs (counts/offsets are zeroed).
 */
#ifndef MOE_GB300_MOE_H_
#define MOE_GB300_MOE_H_

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define MOE_API __attribute__((visibility("default")))
#else
#define MOE_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* ---- status codes ------------------------------------------------------ */
typedef enum moe_status {
  MOE_OK = 0,
  MOE_ERR_INVALID_ARG = -1,         /* null pointer, misaligned pointer, bad shape */
  MOE_ERR_UNSUPPORTED = -2,         /* valid but unsupported combination */
  MOE_ERR_WORKSPACE_TOO_SMALL = -3, /* ws_bytes below the size query's answer */
  MOE_ERR_LAUNCH = -4,              /* a CUDA runtime/driver call failed */
  MOE_ERR_BAD_INDEX = -5,           /* device: expert id or row position out of range */
  MOE_ERR_TIMEOUT = -6              /* device: a bounded wait gave up */
} moe_status;

/* ---- configuration ----------------------------------------------------- */
enum { MOE_DTYPE_F32 = 0, MOE_DTYPE_BF16 = 1 };

enum {
  /* softmax over all E logits, keep the k largest, divide them by their sum */
  MOE_ROUTER_RENORM = 0,
  /* exact softmax over the pre_k largest logits only; keep its first k
   * entries without renormalising (the partial top-8 router of the
   * DeepSeek-V4 EP article, section 3.2) */
  MOE_ROUTER_PREK_SOFTMAX = 1,
  /* node-limited top-k (DeepSeek V3/V4 parallel-strategy article, EP
   * section: a token's experts come from its best nodes only). The E experts
   * form n_group equal groups of consecutive ids; a group's score is the
   * mean softmax probability of its experts; the topk_group best groups are
   * kept (equal scores: lower group id first); the k largest logits among
   * the kept groups' experts are chosen (lower id first on ties) and
   * weighted as in MOE_ROUTER_RENORM. pre_k is validated but not used. */
  MOE_ROUTER_GROUP_LIMITED = 2,
  /* soft gating (Deepseek-MoE sync-tax article, section 3.3: Gumbel-Softmax
   * instead of hard top-k, every expert output weighted): with g the
   * caller's Gumbel samples (the `noise` argument, [T, E] fp32),
   * w[t, e] = softmax_e((L[t, e] + g[t, e]) / tau), max-subtracted; k must
   * equal E (at most 16) and slot j holds expert j. Every token goes to
   * every expert in token order, so dispatch writes only the layout and the
   * W1 GEMM reads x itself (no packed rows, no FP8 payload). */
  MOE_ROUTER_SOFT_GUMBEL = 3
};

typedef struct moe_config {
  int32_t T;           /* tokens, >= 0 */
  int32_t d;           /* hidden size, multiple of 64 */
  int32_t E;           /* experts, 1..256 */
  int32_t k;           /* experts per token, 1..min(E, pre_k, 8) */
  int32_t f;           /* expert FFN inner size, multiple of 64 */
  int32_t dtype;       /* MOE_DTYPE_F32 or MOE_DTYPE_BF16: x, W_g, W1, W2, H, out */
  int32_t router;      /* MOE_ROUTER_* */
  int32_t pre_k;       /* partial top-k width, k..min(8, E) (8 on the pages) */
  int32_t payload_fp8; /* dispatch rows as FP8 E4M3 + an fp32 scale per row (bf16
                        * only): 1 = per-token absmax scale; 2 = one static
                        * scale, payload_scale, for every row (the sync-tax
                        * article's "static global" variant, section 3.1) */
  int32_t n_group;     /* MOE_ROUTER_GROUP_LIMITED: expert groups, 1..32, dividing E;
                        * ignored by the other routers */
  int32_t topk_group;  /* MOE_ROUTER_GROUP_LIMITED: groups kept per token,
                        * 1..n_group, with k <= topk_group * E / n_group */
  float payload_scale; /* payload_fp8 == 2: the scale, finite and > 0; values
                        * beyond 448 * payload_scale saturate to +-448 */
  int32_t output_fp8;  /* 1: moe_forward hands the expert outputs to the combine
                        * as an FP8 payload (moe_quantize_output, then
                        * moe_combine_fp8); 0: fp32 rows (moe_combine) */
  float tau;           /* MOE_ROUTER_SOFT_GUMBEL: temperature, finite and > 0 */
  int32_t gemm_tile_n; /* bf16 expert GEMMs: output features per 2-SM pair tile.
                        * 0 = the library's choice (512 for long-K SiLU passes
                        * with many tiles, else 256); 256 or 512 force it (the
                        * FP8 payload's W1 pass always takes 256). A tuning
                        * knob with no effect on the result beyond fp32
                        * summation order; other values: MOE_ERR_INVALID_ARG */
  int32_t x_perm_mode; /* moe_forward's packed rows (MOE_XPERM_*): packed by the
                        * dispatch into x_perm and read by the W1 GEMM, or
                        * gathered by the W1 GEMM from x through src, x_perm
                        * never written (the dispatch and the first expert
                        * GEMM in one pass: the single-GPU form of the
                        * Waved-EP fusion, DeepSeek V3/V4 parallel-strategy
                        * article). Gathering takes bf16 layers without an FP8
                        * payload or soft gating; asking for it elsewhere is
                        * MOE_ERR_UNSUPPORTED. The stage calls always pack. */
  int32_t keep_z;      /* 1: moe_forward also keeps the W1 GEMM's pre-activation
                        * Z = X_e W1_e [T k, f] (fp32, the value SiLU takes) in
                        * its workspace (moe_workspace_size grows by T k f 4
                        * bytes), and moe_backward, given the same config,
                        * reads it there instead of recomputing it. For a
                        * forward followed by a backward (training); not
                        * with an FP8 payload (those have no backward):
                        * MOE_ERR_UNSUPPORTED. Other values than 0 and 1:
                        * MOE_ERR_INVALID_ARG */
} moe_config_t;

enum {
  MOE_XPERM_AUTO = 0,     /* the library's choice: gathered where it can be and
                           * the packed rows (T k d bf16 values) would take
                           * 256 MiB or more, else packed */
  MOE_XPERM_PACKED = 1,   /* the dispatch writes x_perm */
  MOE_XPERM_GATHERED = 2  /* the W1 GEMM reads x[src[r]]; no x_perm */
};

/* Validate a configuration. Returns MOE_OK or MOE_ERR_INVALID_ARG /
 * MOE_ERR_UNSUPPORTED without touching the device. */
MOE_API int moe_check_config(const moe_config_t* cfg);

/* ---- workspace ----------------------------------------------------------
 * moe_scratch_size: bytes of workspace that moe_dispatch, moe_expert_ffn and
 *   moe_combine need (an error word, the GEMM tile counters and the dispatch
 *   per-block tables).
 * moe_workspace_size: bytes moe_forward needs: the scratch above followed by
 *   every intermediate of the layer (routing, permutation, payload, H, Y).
 *   A forward workspace therefore also serves the stage calls.
 * Both return 0 for an invalid configuration. The caller allocates the
 * workspace (256-byte aligned); zero it once before first use, or call
 * moe_clear_device_error, so the error word starts clear. */
MOE_API size_t moe_scratch_size(const moe_config_t* cfg);
MOE_API size_t moe_workspace_size(const moe_config_t* cfg);

/* ---- stage 1: gate + router ---------------------------------------------
 * The gate's per-expert logit (DeepSeek-V4 EP article, section 2.1) and the
 * router's max-subtracted softmax, partial top-8 and exact top-k (section
 * 3.2); the variants as cited at moe_config.router.
 * x [T, d] (dtype), W_g [d, E] (dtype), bias [E] fp32 or NULL (= zeros),
 * noise [T, E] fp32: the Gumbel samples of MOE_ROUTER_SOFT_GUMBEL (required
 * there, ignored by the other routers, may be NULL).
 * Outputs: topk_idx [T, k] int32, topk_w [T, k] fp32, slot j = j-th choice
 * (logit descending, lower id first on ties; soft gating: expert j);
 * logits [T, E] fp32 or NULL: the gate logits including the bias, as the
 * router saw them (before the noise).
 * Logits are accumulated in fp32 from exact products, in K-chunks combined
 * with compensated summation. */
MOE_API int moe_route(const moe_config_t* cfg, const void* x, const void* W_g,
              const float* bias, const float* noise, int32_t* topk_idx, float* topk_w,
              float* logits, void* stream);

/* ---- stage 2: dispatch ---------------------------------------------------
 * Packing by expert id (DeepSeek-V4 EP article, section 3.3; Deepseek-MoE
 * sync-tax article, section 2.1), with the optional FP8 payload (sync-tax
 * article, section 3.1).
 * Inputs: x [T, d] (dtype), topk_idx [T, k] int32.
 * (MOE_ROUTER_SOFT_GUMBEL: only counts, offsets, pos and src are written,
 * for the routing every token -> every expert in token order; x, topk_idx,
 * x_perm and x_scale are not used and may be NULL.)
 * Outputs (R = T*k):
 *   counts  [E]    int32  rows routed to each expert
 *   offsets [E+1]  int32  exclusive prefix sum of counts; offsets[E] = R
 *   pos     [R]    int32  flat entry i = t*k + j goes to row pos[i]; within an
 *                         expert, rows follow increasing i (stable)
 *   src     [R]    int32  src[pos[i]] = i / k (token of each packed row)
 *   x_perm  [R, d]        packed rows: x[src[r]] in dtype, or with
 *                         cfg->payload_fp8 the FP8 E4M3 bytes (uint8) of
 *                         x / scale, rounded to nearest even, saturating
 *   x_scale [R]    fp32   FP8 only (else may be NULL): scale = fp32(absmax of
 *                         the token's row / 448), 1 for an all-zero row
 * Entries of topk_idx outside [0, E) are skipped (pos = -1) and flag
 * MOE_ERR_BAD_INDEX in the error word. ws: >= moe_scratch_size bytes. */
MOE_API int moe_dispatch(const moe_config_t* cfg, const void* x, const int32_t* topk_idx,
                 int32_t* counts, int32_t* offsets, int32_t* pos, int32_t* src,
                 void* x_perm, float* x_scale, void* ws, size_t ws_bytes,
                 void* stream);

/* ---- dispatch without a workspace ---------------------------------------
 * The source pages have no counterpart to this entry point; it exists for
 * callers that cannot allocate device memory when they dispatch (a locked,
 * pre-sized memory pool; a plugin that is only handed its input and output
 * buffers; code that must not call cudaMalloc because it can synchronise
 * the device). It does what moe_dispatch does, with the same arguments
 * except the workspace: its scratch tables live in a fixed array compiled
 * into the library (4 MiB + 256 bytes, held on every GPU that loads the
 * library until the process exits), and it allocates nothing.
 * Limit: E * ceil(T / 8) <= 524288 (T = 16384 tokens over 256 experts
 * fits); larger requests return MOE_ERR_WORKSPACE_TOO_SMALL before anything
 * is enqueued. Out-of-range expert ids are skipped exactly as in
 * moe_dispatch (pos = -1); there is no error word to read back.
 * Every call shares the array and it keeps the last call's contents (each
 * call rewrites the tables and clears its error word first). Calls whose
 * kernels overlap on the GPU race on the array: order them on one stream.
 * The first call on each device looks up the array's device address (with
 * that device current) and keeps it for the life of the process; make that
 * first call before any stream capture. The kept address belongs to the
 * device's primary context: after cudaDeviceReset (or anything else that
 * destroys that context) it is stale, so do not call this entry point again
 * in a process that has reset the device. */
MOE_API int moe_dispatch_noalloc(const moe_config_t* cfg, const void* x,
                         const int32_t* topk_idx, int32_t* counts, int32_t* offsets,
                         int32_t* pos, int32_t* src, void* x_perm, float* x_scale,
                         void* stream);

/* ---- stage 3: grouped expert FFN -----------------------------------------
 * "L1 + Act + L2" per expert (DeepSeek V3/V4 parallel-strategy article,
 * Waved-EP section), read as one up projection, SiLU and one down projection:
 * For every expert e with rows [offsets[e], offsets[e+1]) of x_perm:
 *   h[r] = SiLU(s_r * x_perm[r] . W1[e])   (s_r = x_scale[r] with FP8, else 1)
 *   y_perm[r] = h[r] . W2[e]
 * x_perm [R, d] (dtype, or uint8 E4M3 with the FP8 payload), x_scale [R]
 * fp32 (FP8 only), offsets [E+1] int32 (non-decreasing, offsets[E] <= R;
 * rows past offsets[E] are not touched), W1 [E, d, f] and W2 [E, f, d]
 * (dtype, expert-major), h [R, f] (dtype) output, y_perm [R, d] fp32 output.
 * bf16 uses the tcgen05 tensor cores (fp32 accumulate in TMEM); fp32 uses
 * fp32 FMA. With the FP8 payload the GEMM reads the E4M3 bytes and expands
 * them to bf16 in shared memory (exact), applying s_r in its epilogue.
 * Experts with no rows read none of their weights.
 * MOE_ROUTER_SOFT_GUMBEL: x_perm is x itself, [T, d]; row r of expert e's
 * segment reads x[r - offsets[e]] (every expert reads all T rows).
 * ws: >= moe_scratch_size bytes. */
MOE_API int moe_expert_ffn(const moe_config_t* cfg, const void* x_perm,
                   const float* x_scale, const int32_t* offsets, const void* W1,
                   const void* W2, void* h, float* y_perm, void* ws,
                   size_t ws_bytes, void* stream);

/* ---- stage 4: combine ------------------------------------------------------
 * The weighted sum of a token's k expert outputs (Deepseek-MoE sync-tax
 * article, section 2.3):
 * out[t] = sum_{j=0..k-1} topk_w[t, j] * y_perm[pos[t*k + j]], accumulated in
 * fp32 in increasing j, then stored in dtype. No atomics: the result is
 * bitwise reproducible. y_perm [R, d] fp32, pos [R] int32, topk_w [T, k]
 * fp32, out [T, d] (dtype). A pos outside [0, R) contributes nothing and
 * flags MOE_ERR_BAD_INDEX. ws: >= moe_scratch_size bytes. */
MOE_API int moe_combine(const moe_config_t* cfg, const float* y_perm, const int32_t* pos,
                const float* topk_w, void* out, void* ws, size_t ws_bytes,
                void* stream);

/* ---- FP8 expert-output payload -------------------------------------------
 * The Deepseek-MoE sync-tax article (section 3.1) sends each expert output
 * vector to the combine as FP8, quantised on its own from its min and max by
 * an affine map.
 * moe_quantize_output: for each row r < R = T*k of y_perm [R, d] fp32:
 *   mn, mx = the row's min and max; zero = fp32(mx/2 + mn/2);
 *   half = fp32(mx/2 - mn/2); s = fp32(half / 448), IEEE division (1 when
 *   half = 0); y_q[r][c] = E4M3(fp32(fp32(y - zero) / s)), rounded to
 *   nearest even, saturating at +-448 (OCP E4M3, no infinities).
 *   Outputs: y_q [R, d] uint8, y_scale [R] fp32 (s), y_zero [R] fp32 (zero).
 *   No workspace; no device-side error is possible.
 * moe_combine_fp8: out[t] = sum_{j=0..k-1} topk_w[t, j] * (q * s + zero) of
 *   row pos[t*k + j], in fp32 in increasing j (each decoded value one fp32
 *   fma), stored in dtype; bitwise reproducible. A pos outside [0, R)
 *   contributes nothing and flags MOE_ERR_BAD_INDEX.
 *   ws: >= moe_scratch_size bytes (error word). */
MOE_API int moe_quantize_output(const moe_config_t* cfg, const float* y_perm, uint8_t* y_q,
                        float* y_scale, float* y_zero, void* stream);
MOE_API int moe_combine_fp8(const moe_config_t* cfg, const uint8_t* y_q, const float* y_scale,
                    const float* y_zero, const int32_t* pos, const float* topk_w,
                    void* out, void* ws, size_t ws_bytes, void* stream);

/* ---- whole layer -----------------------------------------------------------
 * Dispatch, L1 + Act + L2 and combine in sequence (DeepSeek V3/V4
 * parallel-strategy article, EP and Waved-EP sections), on one GPU:
 * moe_route -> moe_dispatch -> moe_expert_ffn -> moe_combine (or, with
 * output_fp8, moe_quantize_output -> moe_combine_fp8) on one stream, with
 * every intermediate in the workspace (>= moe_workspace_size bytes).
 * noise: as for moe_route (the soft router's Gumbel samples, else NULL).
 * No host synchronisation, so the call can be captured into a CUDA graph. */
MOE_API int moe_forward(const moe_config_t* cfg, const void* x, const void* W_g,
                const float* bias, const float* noise, const void* W1, const void* W2,
                void* out, void* ws, size_t ws_bytes, void* stream);

/* (No counterpart on the source pages: timing instrumentation.)
 * moe_forward that also records CUDA events (cudaEvent_t, passed as void*)
 * at the kernel boundaries, for per-kernel timing on the launching stream:
 *   events[0] before the route kernel      events[1] after route
 *   events[2] after dispatch (3 kernels; 1 with soft gating)
 *                                          events[3] = events[2] (kept for
 *   the slot; the FP8 payload is expanded  events[4] after the W1 GEMM
 *   inside the W1 GEMM)
 *   events[5] after the W2 GEMM            events[6] after the output
 *   quantisation (= events[5] without)     events[7] after combine
 * n_events must be MOE_NUM_EVENTS; any entry may be NULL (not recorded). */
#define MOE_NUM_EVENTS 8
MOE_API int moe_forward_with_events(const moe_config_t* cfg, const void* x,
                            const void* W_g, const float* bias, const float* noise,
                            const void* W1, const void* W2, void* out, void* ws,
                            size_t ws_bytes, void* const* events, int n_events,
                            void* stream);

/* (No counterpart on the source pages: inspection of intermediates.)
 * Pointers into a forward workspace, so a caller can inspect the
 * intermediates of the last moe_forward (routing, permutation, H, Y).
 * Any output pointer may be NULL. x_perm is NULL when that forward packs no
 * rows (gathered rows, soft gating). Returns MOE_ERR_INVALID_ARG for a bad
 * configuration. No device access. */
typedef struct moe_forward_views {
  int32_t* topk_idx; float* topk_w;
  int32_t* counts; int32_t* offsets; int32_t* pos; int32_t* src;
  void* x_perm; float* x_scale; void* h; float* y_perm;
  uint8_t* y_q; float* y_scale; float* y_zero;  /* NULL unless output_fp8 */
  float* z;                                     /* NULL unless keep_z */
} moe_forward_views_t;
MOE_API int moe_forward_views(const moe_config_t* cfg, void* ws, moe_forward_views_t* views);

/* ---- backward ------------------------------------------------------------
 * Gradients of a loss l through one moe_forward call, given dout = dl/dout
 * [T, d] (the output dtype): in backpropagation the gradient goes back only
 * to the activated experts (DeepSeek-V4 EP article, section 2.1), along the
 * mirror of the dispatch (Deepseek-MoE sync-tax article, section 2.4):
 *   dY[pos(t,j)] = w[t,j] dout[t]           dw[t,j] = <dout[t], Y[pos(t,j)]>
 *   dL = router Jacobian of dw (softmax over the chosen set; over the pre_k
 *        set for MOE_ROUTER_PREK_SOFTMAX; over all experts, / tau, for
 *        soft gating); no gradient flows through the choice itself
 *   dW_g = x^T dL   db = sum_t dL   dx = dL W_g^T + sum_j dX_perm[pos(t,j)]
 *   per expert e: Z = X_e W1_e (recomputed, or kept by the forward with
 *   keep_z), dW2_e = H_e^T dY_e,
 *   dZ = (dY_e W2_e^T) * SiLU'(Z), dW1_e = X_e^T dZ, dX_perm = dZ W1_e^T
 * x, W_g, bias, noise, W1, W2: the forward's inputs, unchanged. fwd_ws: the
 * workspace of that moe_forward call (>= moe_workspace_size bytes; its
 * routing, permutation, x_perm, H, Y and, with keep_z, Z are read, not
 * changed; keep_z must be the same on both calls). Outputs,
 * fp32, overwritten: dx [T, d], dW_g [d, E], dbias [E] (nullable), dW1 [E,
 * d, f], dW2 [E, f, d]; an expert with no rows gets zero gradients. ws: >=
 * moe_backward_workspace_size bytes, 256-byte aligned; its first word is
 * the backward's device error word (moe_get_device_error(ws, ...)). The
 * FP8 payloads (payload_fp8, output_fp8) have no backward:
 * MOE_ERR_UNSUPPORTED. Every tensor pointer (x, W_g, W1, W2, dout, dx,
 * dW_g, dW1, dW2) must be 16-byte aligned, else MOE_ERR_INVALID_ARG.
 * Precision: bf16 layers run the GEMMs on the tensor cores with each fp32
 * operand carried as two bf16 parts hi + lo (~2^-17 relative) against a
 * bf16 one, fp32 accumulation: dZ and dL against the weights or inputs,
 * and for dW2 either dY against H or, where 2f <= d, w H (each routed row's
 * weight times its H row) against the dout rows; dH takes the bf16 dout
 * rows themselves, the routing weight applied to the fp32 sum; fp32 layers
 * use fp32 FMA. Every sum runs in a fixed order (no atomics): the result is
 * bitwise reproducible. Asynchronous on `stream`. */
MOE_API size_t moe_backward_workspace_size(const moe_config_t* cfg);
MOE_API int moe_backward(const moe_config_t* cfg, const void* x, const void* W_g,
                 const float* bias, const float* noise, const void* W1, const void* W2,
                 const void* fwd_ws, size_t fwd_ws_bytes, const void* dout, float* dx,
                 float* dW_g, float* dbias, float* dW1, float* dW2, void* ws,
                 size_t ws_bytes, void* stream);

/* ---- errors --------------------------------------------------------------
 * moe_get_device_error synchronises `stream`, reads the workspace error
 * word, clears it, and returns MOE_OK, MOE_ERR_BAD_INDEX or MOE_ERR_TIMEOUT
 * (or MOE_ERR_LAUNCH if the stream itself reports an error).
 * moe_clear_device_error enqueues a clear of the error word on `stream`. */
MOE_API int moe_get_device_error(void* ws, void* stream);
MOE_API int moe_clear_device_error(void* ws, void* stream);
MOE_API const char* moe_strerror(int status);

/* Number of kernels one moe_forward call launches for cfg (0 if invalid). */
MOE_API int moe_forward_kernel_count(const moe_config_t* cfg);

/* ---- test hook: the bounded-wait path ---------------------------------------
 * Every wait inside the library's kernels gives up after a bound (2 s by
 * default: a wait that long means the GPU is not making progress), flags
 * MOE_ERR_TIMEOUT in the workspace's error word and lets the kernel finish
 * cleanly (copies and tensor-core work in flight are awaited, tensor memory
 * is freed), so the context stays usable. This call sets, for launches made
 * after it in this process, the bound of one of those waits in the grouped
 * expert GEMM: its epilogue's wait for a finished accumulator, the one a
 * test can make run out without a copy being left in flight (a tiny bound
 * such as 1 ns does it). The GEMM then reports MOE_ERR_TIMEOUT, having taken
 * up to the default bound to wind down. 0 restores the default. Not for use
 * outside tests: the library itself never shortens a bound. Returns
 * MOE_OK. */
MOE_API int moe_set_gemm_epilogue_wait_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif

#endif /* MOE_GB300_MOE_H_ */
