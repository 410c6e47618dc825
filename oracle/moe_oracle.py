"""Plain fp64 CPU oracle of one routed MoE layer forward (test infrastructure).

Each function follows one step of the method as the source pages state it;
page references name the article and its section:

  [V4-EP]    "DeepSeek-V4 Expert Parallelism and computation/communication
             overlap", sections 2.1 (per-expert logits), 3.2 (routing:
             max-subtracted softmax, partial top-8 then exact softmax over
             those 8, hard top-k), 3.3 (packing by expert id), 5.2 (expert
             weights laid out contiguously by expert id).
  [SYNC-TAX] "Deepseek-MoE sync tax", sections 2.1 (top-k gating, per-
             destination packed buffers), 2.3 (weighted sum of the k expert
             outputs per token), 3.1 (per-token FP8 payload quantisation of
             expert inputs and, by min/max affine maps, expert outputs).
  [V3V4-PAR] "DeepSeek V3/V4 parallel strategy", EP and Waved-EP sections
             (dispatch, expert L1 + Act + L2, combine; the V3 limit of a
             token's 8 experts to the 4 nodes that are best on average).

Readings taken where the pages leave a step open are listed with each
function (expert FFN form, selection order, FP8 scale form, rounding points).
"""
from __future__ import annotations

import numpy as np

from .numerics import round_to_bf16, round_to_f32, e4m3_round_satfinite

ROUTER_RENORM = 0
ROUTER_PREK_SOFTMAX = 1
ROUTER_GROUP_LIMITED = 2
ROUTER_SOFT_GUMBEL = 3
E4M3_MAX_F32 = np.float32(448.0)


# ----------------------------------------------------------------------------
# inputs
# ----------------------------------------------------------------------------
def _np64(t) -> np.ndarray:
    """fp64 numpy copy of a torch tensor or array (bf16/fp32 values are exact)."""
    if hasattr(t, "detach"):
        t = t.detach().cpu()            # the conversion itself runs on the host
        if t.dtype.is_floating_point:
            t = t.to(dtype=__import__("torch").float64)
        return t.numpy()
    return np.asarray(t, dtype=np.float64)


def inputs_to_numpy(inp: dict) -> dict:
    """x, Wg, bias (and the Gumbel samples of soft gating) as fp64 arrays;
    W1/W2 stay as given and are fetched one expert at a time by ``_expert``
    (the largest layer's weights are 15 GB)."""
    out = {"x": _np64(inp["x"]), "Wg": _np64(inp["Wg"]), "bias": _np64(inp["bias"]),
           "W1": inp["W1"], "W2": inp["W2"]}
    if inp.get("gumbel") is not None:
        out["gumbel"] = _np64(inp["gumbel"])
    return out


def _expert(W, e: int) -> np.ndarray:
    return _np64(W[e])


# ----------------------------------------------------------------------------
# gate [V4-EP 2.1]: each expert's logit is the token's dot product with that
# expert's gate column, plus the expert's bias.
# ----------------------------------------------------------------------------
def gate_logits(x: np.ndarray, Wg: np.ndarray, bias: np.ndarray | None) -> np.ndarray:
    L = np.asarray(x, np.float64) @ np.asarray(Wg, np.float64)
    if bias is not None:
        L = L + np.asarray(bias, np.float64)[None, :]
    return L


# ----------------------------------------------------------------------------
# router [V4-EP 3.2]
# ----------------------------------------------------------------------------
def _softmax_max_subtracted(L: np.ndarray) -> np.ndarray:
    """Softmax along the last axis after subtracting the row maximum
    ("logits - logits.max()" to avoid overflow)."""
    z = L - L.max(axis=-1, keepdims=True)
    ez = np.exp(z)
    return ez / ez.sum(axis=-1, keepdims=True)


def route(L: np.ndarray, k: int, router: int = ROUTER_RENORM, pre_k: int = 8,
          n_group: int = 1, topk_group: int = 1, gumbel: np.ndarray | None = None,
          tau: float = 1.0):
    """Top-k expert selection and gate weights.

    Order: logits descending, equal logits by expert id ascending (the lower
    id wins). The partial top-``pre_k`` is found first; the k chosen experts
    are its first k entries, and slot j of a token holds its j-th choice.

    * ROUTER_RENORM (hard top-k): p = softmax(L - max L) over all E experts;
      the k chosen probabilities are divided by their sum.
    * ROUTER_PREK_SOFTMAX: the exact softmax is taken over the pre_k largest
      logits only; the k chosen entries of that softmax are the weights, not
      renormalised (their sum is at most 1).
    * ROUTER_GROUP_LIMITED (node-limited, [V3V4-PAR] EP section): the E
      experts form n_group equal groups of consecutive ids (a node's
      experts). A group's score is the average softmax probability of its
      experts; the topk_group best groups are kept (equal scores: the lower
      group id first). The k chosen experts are the top-k logits among the
      kept groups' experts, weighted as in ROUTER_RENORM (their full-softmax
      probabilities divided by their sum). pre_k plays no part.
    * ROUTER_SOFT_GUMBEL (soft gating, [SYNC-TAX 3.3]): no top-k; the E
      logits plus the Gumbel samples ``gumbel`` [T, E], divided by the
      temperature tau, go through a (max-subtracted) softmax and every expert
      keeps its probability as weight. k must equal E; slot j holds expert j.

    Returns (topk_idx int32 [T, k], topk_w fp64 [T, k]).
    """
    L = np.asarray(L, np.float64)
    T, E = L.shape
    if router == ROUTER_GROUP_LIMITED:
        return _route_group_limited(L, k, n_group, topk_group)
    if router == ROUTER_SOFT_GUMBEL:
        return _route_soft_gumbel(L, k, gumbel, tau)
    pre_k = min(pre_k, E)
    if not (1 <= k <= pre_k):
        raise ValueError("need 1 <= k <= min(pre_k, E)")
    # stable sort of -L: descending logits, ties keep ascending expert id
    order = np.argsort(-L, axis=1, kind="stable")
    S = order[:, :pre_k]                              # partial top-pre_k
    sel = S[:, :k]
    rows = np.arange(T)[:, None]
    if router == ROUTER_RENORM:
        p = _softmax_max_subtracted(L)
        ps = p[rows, sel]
        w = ps / ps.sum(axis=1, keepdims=True)
    elif router == ROUTER_PREK_SOFTMAX:
        q = _softmax_max_subtracted(L[rows, S])
        w = q[:, :k]
    else:
        raise ValueError(f"unknown router mode {router}")
    return sel.astype(np.int32), w


def _route_group_limited(L: np.ndarray, k: int, n_group: int, topk_group: int):
    """Node-limited top-k [V3V4-PAR EP section]: keep the topk_group groups
    with the best average probability, then the k best experts inside them."""
    T, E = L.shape
    if n_group < 1 or E % n_group:
        raise ValueError("n_group must divide E")
    gs = E // n_group
    if not (1 <= topk_group <= n_group and 1 <= k <= topk_group * gs):
        raise ValueError("need 1 <= topk_group <= n_group and 1 <= k <= topk_group * E/n_group")
    p = _softmax_max_subtracted(L)
    score = p.reshape(T, n_group, gs).mean(axis=2)          # average affinity per group
    kept = np.argsort(-score, axis=1, kind="stable")[:, :topk_group]
    allowed = np.zeros((T, E), dtype=bool)
    for t in range(T):
        for g in kept[t]:
            allowed[t, g * gs:(g + 1) * gs] = True
    # experts outside the kept groups sort after every allowed one
    Lk = np.where(allowed, L, -np.inf)
    sel = np.argsort(-Lk, axis=1, kind="stable")[:, :k]
    ps = p[np.arange(T)[:, None], sel]
    return sel.astype(np.int32), ps / ps.sum(axis=1, keepdims=True)


def _route_soft_gumbel(L: np.ndarray, k: int, gumbel, tau: float):
    """Soft gating [SYNC-TAX 3.3]: Gumbel-softmax over all E experts, every
    expert weighted (none dropped)."""
    T, E = L.shape
    if k != E:
        raise ValueError("soft gating weights every expert: k must equal E")
    if gumbel is None or np.shape(gumbel) != (T, E):
        raise ValueError("soft gating needs Gumbel samples of shape [T, E]")
    if not (np.isfinite(tau) and tau > 0):
        raise ValueError("tau must be finite and positive")
    z = (L + np.asarray(gumbel, np.float64)) / float(np.float32(tau))
    w = _softmax_max_subtracted(z)
    idx = np.broadcast_to(np.arange(E, dtype=np.int32), (T, E)).copy()
    return idx, w


# ----------------------------------------------------------------------------
# dispatch [V4-EP 3.3; SYNC-TAX 2.1]: pack the (token, expert) pairs
# contiguously by expert id with a stable counting sort.
# ----------------------------------------------------------------------------
def dispatch(topk_idx: np.ndarray, E: int):
    """Returns counts [E], offsets [E+1], pos [R], src [R] (all int64).

    Flat entry i = t*k + j (token t's j-th choice, expert e) goes to row
    pos[i] = offsets[e] + (number of earlier flat entries with expert e);
    src[pos[i]] = t.
    """
    idx = np.asarray(topk_idx)
    T, k = idx.shape
    flat = idx.reshape(-1).astype(np.int64)
    R = flat.size
    if R and (flat.min() < 0 or flat.max() >= E):
        raise ValueError("expert index out of range")
    counts = np.zeros(E, dtype=np.int64)
    for e in flat:                      # histogram
        counts[e] += 1
    offsets = np.zeros(E + 1, dtype=np.int64)
    for e in range(E):                  # exclusive scan
        offsets[e + 1] = offsets[e] + counts[e]
    fill = offsets[:-1].copy()
    pos = np.empty(R, dtype=np.int64)
    for i in range(R):                  # stable placement, flat order
        e = flat[i]
        pos[i] = fill[e]
        fill[e] += 1
    src = np.empty(R, dtype=np.int64)
    src[pos] = np.arange(R) // k
    return counts, offsets, pos, src


# ----------------------------------------------------------------------------
# FP8 payload [SYNC-TAX 3.1]: per-token scale so the token's largest magnitude
# maps to the E4M3 maximum; symmetric (absmax) form, fp32 scale.
# ----------------------------------------------------------------------------
def quantize_payload_fp8(x_rows: np.ndarray, static_scale: float | None = None):
    """Per row t: a = max |x_t| (fp32), s = fp32(a / 448) with an fp32 IEEE
    division (s = 1 for an all-zero row), q = E4M3(fp32(x / s)) with an fp32
    IEEE division, rounded to nearest even and saturated to +-448.

    With ``static_scale`` (the "static global" variant [SYNC-TAX 3.1]: one
    scale fixed ahead of time for the whole tensor), s = fp32(static_scale)
    for every row and no absmax is taken; values beyond 448 s saturate.

    Returns (q as fp64 E4M3 values [T, d], s as fp64 holding fp32 values [T])."""
    x32 = np.asarray(x_rows, np.float64).astype(np.float32)
    if static_scale is not None:
        s = np.full(x32.shape[0], np.float32(static_scale), dtype=np.float32)
        if not (np.isfinite(s).all() and (s > 0).all()):
            raise ValueError("static scale must be finite and positive")
    else:
        a = np.abs(x32).max(axis=1)
        s = (a / E4M3_MAX_F32).astype(np.float32)
        s = np.where(a == 0, np.float32(1.0), s).astype(np.float32)
    ratio = (x32 / s[:, None]).astype(np.float32)     # fp32 division, RN
    q = e4m3_round_satfinite(ratio.astype(np.float64))
    return q, s.astype(np.float64)


# ----------------------------------------------------------------------------
# FP8 expert-output payload [SYNC-TAX 3.1]: each expert output vector is
# quantised on its own, from its min and max, by an affine map.
# ----------------------------------------------------------------------------
def quantize_output_fp8(Y_rows: np.ndarray):
    """Per row r of the fp32 expert outputs y: mn = min y, mx = max y;
    zero = fp32(mx/2 + mn/2) and half = fp32(mx/2 - mn/2) (each a single fp32
    rounding; halving is exact); s = fp32(half / 448) with an fp32 IEEE
    division (s = 1 for a constant row); q = E4M3(fp32(fp32(y - zero) / s)),
    rounded to nearest even and saturated to +-448. The row decodes as
    q * s + zero, so [mn, mx] spans the E4M3 range [-448, 448].

    Returns (q as fp64 E4M3 values [R, d], s and zero as fp64 holding fp32
    values [R])."""
    y = np.asarray(Y_rows, np.float64).astype(np.float32)
    half_f = np.float32(0.5)
    mn = y.min(axis=1)
    mx = y.max(axis=1)
    zero = (mx * half_f + mn * half_f).astype(np.float32)
    half = (mx * half_f - mn * half_f).astype(np.float32)
    s = (half / E4M3_MAX_F32).astype(np.float32)
    s = np.where(half == 0, np.float32(1.0), s).astype(np.float32)
    diff = (y - zero[:, None]).astype(np.float32)
    ratio = (diff / s[:, None]).astype(np.float32)
    q = e4m3_round_satfinite(ratio.astype(np.float64))
    return q, s.astype(np.float64), zero.astype(np.float64)


def dequantize_output_fp8(q: np.ndarray, s: np.ndarray, zero: np.ndarray) -> np.ndarray:
    """The expert outputs the combine sees: q * s + zero per row."""
    return np.asarray(q, np.float64) * np.asarray(s, np.float64)[:, None] + \
        np.asarray(zero, np.float64)[:, None]


# ----------------------------------------------------------------------------
# expert FFN [V3V4-PAR Waved-EP: "L1 + Act + L2"; V4-EP 2.3: W1 by columns,
# W2 by rows]: reading = one up projection, SiLU, one down projection, no
# biases and no gating branch.
# ----------------------------------------------------------------------------
def silu(z: np.ndarray) -> np.ndarray:
    """SiLU(z) = z / (1 + e^-z)."""
    with np.errstate(over="ignore"):
        return z / (1.0 + np.exp(-z))


def expert_ffn_rows(x_rows: np.ndarray, W1e: np.ndarray, W2e: np.ndarray,
                    h_storage: str = "bf16"):
    """y = round_storage(SiLU(x W1_e)) W2_e for the rows routed to expert e.

    ``h_storage`` mirrors the dtype the hidden activation is stored in
    between the two projections ("bf16", "f32", or "exact" for none)."""
    z = np.asarray(x_rows, np.float64) @ np.asarray(W1e, np.float64)
    h = silu(z)
    if h_storage == "bf16":
        h = round_to_bf16(h)
    elif h_storage == "f32":
        h = round_to_f32(h)
    return h @ np.asarray(W2e, np.float64), h


# ----------------------------------------------------------------------------
# combine [SYNC-TAX 2.3]: weighted sum of a token's k expert outputs.
# ----------------------------------------------------------------------------
def combine(Y: np.ndarray, pos: np.ndarray, topk_w: np.ndarray) -> np.ndarray:
    """out[t] = sum over j = 0..k-1 of w[t, j] * Y[pos[t*k + j]]."""
    w = np.asarray(topk_w, np.float64)
    T, k = w.shape
    Y = np.asarray(Y, np.float64)
    out = np.zeros((T, Y.shape[1]), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * Y[np.asarray(pos).reshape(T, k)[:, j]]
    return out


# ----------------------------------------------------------------------------
# whole layer
# ----------------------------------------------------------------------------
def _router_args(cfg, a, tokens=None):
    """Router arguments past (L, k): pre_k, groups, Gumbel samples, tau."""
    g = a.get("gumbel")
    if g is not None:
        g = _np64(g)
        if tokens is not None:
            g = g[tokens]
    return (cfg.pre_k, getattr(cfg, "n_group", 1), getattr(cfg, "topk_group", 1), g,
            getattr(cfg, "tau", 1.0))


def _payload(cfg, x):
    """The rows the experts see and the payload: (x_hat, q, s) or (x, None, None)."""
    if not cfg.payload_fp8:
        return x, None, None
    static = getattr(cfg, "payload_scale", 0.0) if int(cfg.payload_fp8) == 2 else None
    q, s = quantize_payload_fp8(x, static)
    return q * s[:, None], q, s


def _storage(cfg) -> str:
    return "bf16" if cfg.dtype == "bf16" else "f32"


def _round_out(cfg, v):
    return round_to_bf16(v) if cfg.dtype == "bf16" else round_to_f32(v)


def forward(cfg, inp: dict, keep_h: bool = True) -> dict:
    """Every intermediate of the layer for a (small) config.

    ``inp`` is the dict from ``workloads.make_inputs`` (or inputs_to_numpy of
    it). Returns a dict with L, topk_idx, topk_w, counts, offsets, pos, src,
    x_hat (the rows the experts see: x, or the dequantised FP8 payload),
    q / scale (FP8 only), H (optional), Y, out (fp64) and out_rounded (the
    output dtype's rounding of out)."""
    a = inputs_to_numpy(inp) if not isinstance(inp.get("x"), np.ndarray) else inp
    x = a["x"]
    L = gate_logits(x, a["Wg"], a["bias"])
    idx, w = route(L, cfg.k, cfg.router, *_router_args(cfg, a))
    counts, offsets, pos, src = dispatch(idx, cfg.E)
    res = {"L": L, "topk_idx": idx, "topk_w": w, "counts": counts,
           "offsets": offsets, "pos": pos, "src": src}
    x_hat_tok, q_tok, s_tok = _payload(cfg, x)
    if q_tok is not None:
        res["q"] = q_tok[src]
        res["scale"] = s_tok[src]
    R = idx.size
    Y = np.zeros((R, cfg.d), dtype=np.float64)
    H = np.zeros((R, cfg.f), dtype=np.float64) if keep_h else None
    for e in range(cfg.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue                    # an expert with no tokens does no work
        rows = x_hat_tok[src[lo:hi]]
        y, h = expert_ffn_rows(rows, _expert(a["W1"], e), _expert(a["W2"], e),
                               _storage(cfg))
        Y[lo:hi] = y
        if keep_h:
            H[lo:hi] = h
    if getattr(cfg, "output_fp8", 0):
        yq, ys, yz = quantize_output_fp8(Y)
        res.update({"y_q": yq, "y_scale": ys, "y_zero": yz})
        out = combine(dequantize_output_fp8(yq, ys, yz), pos, w)
    else:
        out = combine(Y, pos, w)
    res.update({"Y": Y, "out": out, "out_rounded": _round_out(cfg, out)})
    if keep_h:
        res["H"] = H
    return res


def forward_tokens(cfg, inp: dict, tokens) -> dict:
    """Route, FFN and combine for a subset of tokens only (a token's output
    does not depend on other tokens). Used for sampled checks on the large
    layers. Returns L, topk_idx, topk_w, out, out_rounded for ``tokens``
    (and, with the FP8 expert-output payload, y_q [n, k, d], y_scale and
    y_zero [n, k] per token slot)."""
    a = inputs_to_numpy(inp) if not isinstance(inp.get("x"), np.ndarray) else inp
    tokens = np.asarray(tokens, dtype=np.int64)
    x = a["x"][tokens]
    L = gate_logits(x, a["Wg"], a["bias"])
    idx, w = route(L, cfg.k, cfg.router, *_router_args(cfg, a, tokens))
    x_hat, _, _ = _payload(cfg, x)
    n, k = idx.shape
    y_slot = np.zeros((n, k, cfg.d), dtype=np.float64)
    for e in np.unique(idx):
        tt, jj = np.nonzero(idx == e)
        y, _ = expert_ffn_rows(x_hat[tt], _expert(a["W1"], int(e)),
                               _expert(a["W2"], int(e)), _storage(cfg))
        y_slot[tt, jj] = y
    res = {"tokens": tokens}
    if getattr(cfg, "output_fp8", 0):
        yq, ys, yz = quantize_output_fp8(y_slot.reshape(n * k, cfg.d))
        res.update({"y_q": yq.reshape(n, k, cfg.d), "y_scale": ys.reshape(n, k),
                    "y_zero": yz.reshape(n, k)})
        y_slot = dequantize_output_fp8(yq, ys, yz).reshape(n, k, cfg.d)
    out = np.zeros((n, cfg.d), dtype=np.float64)
    for j in range(k):
        out += w[:, j:j + 1] * y_slot[:, j]
    res.update({"L": L, "topk_idx": idx, "topk_w": w, "out": out,
                "out_rounded": _round_out(cfg, out)})
    return res


# ----------------------------------------------------------------------------
# backward [V4-EP 2.1: in backpropagation the gradient goes back only to the
# activated experts; SYNC-TAX 2.4: the backward exchange mirrors the
# dispatch]: gradients of a loss l whose gradient with respect to the layer
# output is dout = dl/dout. Readings: the expert choice itself is piecewise
# constant (no gradient through the top-k selection, only through the
# chosen experts' weights); the Gumbel samples are constants; storage
# roundings (H in the layer dtype, the output) pass the gradient unchanged,
# and dW2 uses the stored H, the value the forward multiplied by W2; the FP8
# payloads have no backward here.
# ----------------------------------------------------------------------------
def silu_grad(z: np.ndarray) -> np.ndarray:
    """d SiLU / dz = s (1 + z (1 - s)) with s = 1 / (1 + e^-z)."""
    with np.errstate(over="ignore"):
        s = 1.0 / (1.0 + np.exp(-z))
    return s * (1.0 + z * (1.0 - s))


def router_backward(L: np.ndarray, topk_idx: np.ndarray, topk_w: np.ndarray, dw: np.ndarray,
                    router: int = ROUTER_RENORM, pre_k: int = 8, tau: float = 1.0) -> np.ndarray:
    """dl/dL [T, E] from dl/dw [T, k] (dw[t, j] for the weight in slot j).

    * ROUTER_RENORM and ROUTER_GROUP_LIMITED: the weights are a softmax over
      the chosen set S (w_j = e^L_j / sum_S e^L_i), so dL_j = w_j (dw_j -
      sum_i w_i dw_i) for j in S and 0 elsewhere.
    * ROUTER_PREK_SOFTMAX: q = softmax over the pre_k largest logits P and
      w_j = q_j for the first k of P, so for i in P dL_i = q_i (g_i -
      sum_{j<k} dw_j q_j) with g_i = dw_i for the k chosen and 0 for the rest
      of P; 0 outside P.
    * ROUTER_SOFT_GUMBEL: w = softmax((L + g) / tau) over all E, slot j =
      expert j, so dL = (w / tau) (dw - sum_i w_i dw_i)."""
    L = np.asarray(L, np.float64)
    T, E = L.shape
    w = np.asarray(topk_w, np.float64)
    dw = np.asarray(dw, np.float64)
    idx = np.asarray(topk_idx, np.int64)
    dL = np.zeros((T, E), dtype=np.float64)
    rows = np.arange(T)[:, None]
    if router == ROUTER_SOFT_GUMBEL:
        s = (w * dw).sum(axis=1, keepdims=True)
        dL[rows, idx] = w * (dw - s) / float(np.float32(tau))
        return dL
    if router == ROUTER_PREK_SOFTMAX:
        pk = min(pre_k, E)
        P = np.argsort(-L, axis=1, kind="stable")[:, :pk]
        q = _softmax_max_subtracted(L[rows, P])
        k = idx.shape[1]
        g = np.zeros_like(q)
        g[:, :k] = dw
        s = (dw * q[:, :k]).sum(axis=1, keepdims=True)
        dL[rows, P] = q * (g - s)
        return dL
    s = (w * dw).sum(axis=1, keepdims=True)
    dL[rows, idx] = w * (dw - s)
    return dL


def _combine_backward(pos: np.ndarray, w: np.ndarray, Y: np.ndarray, g: np.ndarray):
    """Combine step backward: out[t] = sum_j w[t, j] Y[pos[t, j]] gives
    dY[pos[t, j]] = w[t, j] dout[t] and dw[t, j] = <dout[t], Y[pos[t, j]]>."""
    T, k = w.shape
    dY = np.zeros((T * k, Y.shape[1]), dtype=np.float64)
    dw = np.zeros((T, k), dtype=np.float64)
    for j in range(k):
        dY[pos[:, j]] = w[:, j:j + 1] * g
        dw[:, j] = (g * Y[pos[:, j]]).sum(axis=1)
    return dY, dw


def _expert_backward(xe: np.ndarray, W1e: np.ndarray, W2e: np.ndarray, dYe: np.ndarray,
                     hs: str):
    """One expert's rows: z = x_e W1_e, h = SiLU(z) (stored rounded), y = h W2_e.
    Returns dW1_e = x_e^T dZ, dW2_e = h^T dY_e and dX_e = dZ W1_e^T, with
    dZ = (dY_e W2_e^T) * SiLU'(z)."""
    z = xe @ W1e
    h = silu(z)
    if hs == "bf16":
        h = round_to_bf16(h)
    elif hs == "f32":
        h = round_to_f32(h)
    dW2e = h.T @ dYe
    dZ = (dYe @ W2e.T) * silu_grad(z)
    return xe.T @ dZ, dW2e, dZ @ W1e.T


def _backward_setup(cfg, inp, fwd, dout):
    if cfg.payload_fp8 or getattr(cfg, "output_fp8", 0):
        raise ValueError("the FP8 payloads have no backward")
    a = inputs_to_numpy(inp) if not isinstance(inp.get("x"), np.ndarray) else inp
    T, k = np.asarray(fwd["topk_idx"]).shape
    pos = np.asarray(fwd["pos"]).reshape(T, k)
    w = np.asarray(fwd["topk_w"], np.float64)
    g = np.asarray(dout, np.float64) if not hasattr(dout, "detach") else _np64(dout)
    return a, pos, w, g


def backward(cfg, inp: dict, fwd: dict, dout, h_storage: str | None = None) -> dict:
    """Gradients of the layer for dout = dl/dout [T, d]: dx [T, d], dWg [d, E],
    dbias [E], dW1 [E, d, f], dW2 [E, f, d], and the intermediates dY (per
    routed row), dw [T, k], dL [T, E]. ``fwd`` is forward(cfg, inp) (its
    routing, permutation, H and Y); ``h_storage`` (default: the layer's)
    must match the forward's."""
    a, pos, w, g = _backward_setup(cfg, inp, fwd, dout)
    x = a["x"]
    R = pos.size
    src = np.asarray(fwd["src"])
    offsets = np.asarray(fwd["offsets"])
    hs = h_storage or _storage(cfg)
    # combine: out[t] = sum_j w[t, j] Y[pos[t, j]]
    dY, dw = _combine_backward(pos, w, np.asarray(fwd["Y"], np.float64), g)
    # router and gate: L = x W_g + b
    dL = router_backward(fwd["L"], fwd["topk_idx"], w, dw, cfg.router, cfg.pre_k,
                         getattr(cfg, "tau", 1.0))
    Wg = np.asarray(a["Wg"], np.float64)
    dx = dL @ Wg.T
    dWg = x.T @ dL
    dbias = dL.sum(axis=0)
    # experts: z = x_e W1_e, h = SiLU(z) (stored rounded), y = h W2_e
    dW1 = np.zeros((cfg.E, cfg.d, cfg.f), dtype=np.float64)
    dW2 = np.zeros((cfg.E, cfg.f, cfg.d), dtype=np.float64)
    dXp = np.zeros((R, cfg.d), dtype=np.float64)
    for e in range(cfg.E):
        lo, hi = int(offsets[e]), int(offsets[e + 1])
        if hi == lo:
            continue                  # no rows: the expert's gradients are 0
        dW1[e], dW2[e], dXp[lo:hi] = _expert_backward(
            x[src[lo:hi]], _expert(a["W1"], e), _expert(a["W2"], e), dY[lo:hi], hs)
    # mirror of the dispatch: each routed row's gradient back to its token
    for j in range(pos.shape[1]):
        dx += dXp[pos[:, j]]
    return {"dx": dx, "dWg": dWg, "dbias": dbias, "dW1": dW1, "dW2": dW2, "dY": dY, "dw": dw,
            "dL": dL}


def backward_router(cfg, inp: dict, fwd: dict, dout) -> dict:
    """The gate's part of ``backward`` alone (no expert GEMMs): dw [T, k],
    dL [T, E], dWg [d, E], dbias [E]. Used for full checks of the gate's
    gradients on layers too large for the whole backward."""
    a, pos, w, g = _backward_setup(cfg, inp, fwd, dout)
    _, dw = _combine_backward(pos, w, np.asarray(fwd["Y"], np.float64), g)
    dL = router_backward(fwd["L"], fwd["topk_idx"], w, dw, cfg.router, cfg.pre_k,
                         getattr(cfg, "tau", 1.0))
    return {"dw": dw, "dL": dL, "dWg": a["x"].T @ dL, "dbias": dL.sum(axis=0)}


def backward_expert(cfg, inp: dict, fwd: dict, dout, e: int,
                    h_storage: str | None = None) -> dict:
    """Expert e's part of ``backward`` alone: dW1[e] [d, f] and dW2[e] [f, d]
    (zeros for an expert with no rows), from the rows routed to it."""
    a, pos, w, g = _backward_setup(cfg, inp, fwd, dout)
    offsets = np.asarray(fwd["offsets"])
    lo, hi = int(offsets[e]), int(offsets[e + 1])
    if hi == lo:
        return {"dW1": np.zeros((cfg.d, cfg.f)), "dW2": np.zeros((cfg.f, cfg.d))}
    k = pos.shape[1]
    # the flat entry t*k + j of each routed row r: dY[r] = w[t, j] dout[t]
    flat = np.empty(pos.size, dtype=np.int64)
    flat[pos.reshape(-1)] = np.arange(pos.size)
    i = flat[lo:hi]
    dYe = w.reshape(-1)[i][:, None] * g[i // k]
    src = np.asarray(fwd["src"])
    dW1e, dW2e, _ = _expert_backward(a["x"][src[lo:hi]], _expert(a["W1"], e),
                                     _expert(a["W2"], e), dYe, h_storage or _storage(cfg))
    return {"dW1": dW1e, "dW2": dW2e}


def backward_tokens(cfg, inp: dict, dout, tokens, h_storage: str | None = None) -> dict:
    """dx and dL for a subset of tokens only (a token's input gradient depends
    only on its own routing, expert rows and dout row). Used for sampled
    checks on the large layers. ``dout``: [T, d] (all tokens) or [n, d]."""
    if cfg.payload_fp8 or getattr(cfg, "output_fp8", 0):
        raise ValueError("the FP8 payloads have no backward")
    a = inputs_to_numpy(inp) if not isinstance(inp.get("x"), np.ndarray) else inp
    tokens = np.asarray(tokens, dtype=np.int64)
    x = a["x"][tokens]
    g = np.asarray(dout, np.float64) if not hasattr(dout, "detach") else _np64(dout)
    if g.shape[0] != len(tokens):
        g = g[tokens]
    L = gate_logits(x, a["Wg"], a["bias"])
    idx, w = route(L, cfg.k, cfg.router, *_router_args(cfg, a, tokens))
    hs = h_storage or _storage(cfg)
    n, k = idx.shape
    dw = np.zeros((n, k))
    dXp_slot = np.zeros((n, k, cfg.d))
    for e in np.unique(idx):
        tt, jj = np.nonzero(idx == e)
        W1e, W2e = _expert(a["W1"], int(e)), _expert(a["W2"], int(e))
        z = x[tt] @ W1e
        h = silu(z)
        if hs == "bf16":
            h = round_to_bf16(h)
        elif hs == "f32":
            h = round_to_f32(h)
        y = h @ W2e
        dw[tt, jj] = (g[tt] * y).sum(axis=1)
        dY = w[tt, jj][:, None] * g[tt]
        dZ = (dY @ W2e.T) * silu_grad(z)
        dXp_slot[tt, jj] = dZ @ W1e.T
    dL = router_backward(L, idx, w, dw, cfg.router, cfg.pre_k, getattr(cfg, "tau", 1.0))
    dx = dL @ np.asarray(a["Wg"], np.float64).T + dXp_slot.sum(axis=1)
    return {"tokens": tokens, "topk_idx": idx, "dL": dL, "dx": dx}
