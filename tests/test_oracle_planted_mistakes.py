"""The oracle's pins must fail when the oracle is wrong in a plausible way.

Each case below plants one mistake in the oracle (on the CPU: the oracle
function is replaced, in every module that holds it, by a wrong version)
and runs one of the pins written for that function; the pin must fail. The
mistakes are the ones a reader of the pages could make: a dropped bias, the
wrong tie order, weights not renormalised, a softmax without the max
subtracted, the top-pre_k softmax taken over every expert, group scores by
maximum or by mean logit, the temperature or the noise of soft gating
ignored, an unstable packing, a source index that forgets k, a combine
without its weights or with its slots crossed, E4M3 ties away from zero, no
subnormal range or no saturation, an fp64 payload scale or quotient, an
output payload mapped onto [0, 448] or decoded without its zero point, 240
for the E4M3 maximum, experts fed the rows before quantisation, H not
rounded to its storage type, ReLU for SiLU, bf16 rounding to seven bits or
by truncation, and backward passes that forget a term. (The FFN's planted
mistakes against its permutation pin sit beside that pin.)"""
import numpy as np
import pytest

import oracle
import oracle.moe_oracle as mo
import oracle.numerics as nu
import test_oracle_backward as backward_pins
import test_oracle_dispatch as dispatch_pins
import test_oracle_ffn as ffn_pins
import test_oracle_numerics as numerics_pins
import test_oracle_output_payload as outpay_pins
import test_oracle_router as router_pins
import test_oracle_router_groups as group_pins
import test_oracle_router_soft as soft_pins

HOLDERS = [oracle, mo, nu, backward_pins, dispatch_pins, ffn_pins, numerics_pins, outpay_pins,
           router_pins, group_pins, soft_pins]

REAL = {n: getattr(mo, n) for n in (
    "gate_logits", "route", "_softmax_max_subtracted", "_route_group_limited",
    "_route_soft_gumbel", "dispatch", "combine", "quantize_payload_fp8",
    "quantize_output_fp8", "dequantize_output_fp8", "router_backward", "silu_grad",
    "_combine_backward", "backward", "expert_ffn_rows", "silu", "_payload")}
REAL["e4m3_round_satfinite"] = nu.e4m3_round_satfinite
REAL["round_to_bf16"] = nu.round_to_bf16


def plant(monkeypatch, name, bad):
    """Replace the oracle function ``name`` by ``bad`` wherever it is bound."""
    real = REAL[name]
    for mod in HOLDERS:
        for attr, val in list(vars(mod).items()):
            if val is real:
                monkeypatch.setattr(mod, attr, bad)


def must_fail(pin, *args):
    with pytest.raises(AssertionError):
        pin(*args)


# ---------------------------------------------------------------- gate, router
def test_gate_bias_dropped(monkeypatch):
    plant(monkeypatch, "gate_logits", lambda x, Wg, b: REAL["gate_logits"](x, Wg, None))
    must_fail(router_pins.test_gate_matches_triple_loop)
    must_fail(router_pins.test_bias_moves_selection)


def test_gate_rows_of_the_wrong_token(monkeypatch):
    plant(monkeypatch, "gate_logits",
          lambda x, Wg, b: np.roll(REAL["gate_logits"](x, Wg, b), 1, axis=0))
    must_fail(router_pins.test_gate_matches_triple_loop)


def _route_ties_to_higher_id(L, k, router=0, pre_k=8, *a, **kw):
    L = np.asarray(L, np.float64)
    idx, w = REAL["route"](L[:, ::-1], k, router, pre_k, *a, **kw)
    return (L.shape[1] - 1 - idx).astype(np.int32), w


def _route_not_renormalised(L, k, router=0, pre_k=8, *a, **kw):
    idx, w = REAL["route"](L, k, router, pre_k, *a, **kw)
    if router == mo.ROUTER_RENORM:
        p = REAL["_softmax_max_subtracted"](np.asarray(L, np.float64))
        w = p[np.arange(idx.shape[0])[:, None], idx]
    return idx, w


def _route_prek_over_all(L, k, router=0, pre_k=8, *a, **kw):
    idx, w = REAL["route"](L, k, router, pre_k, *a, **kw)
    if router == mo.ROUTER_PREK_SOFTMAX:
        p = REAL["_softmax_max_subtracted"](np.asarray(L, np.float64))
        w = p[np.arange(idx.shape[0])[:, None], idx]
    return idx, w


def test_router_ties_go_to_the_higher_id(monkeypatch):
    plant(monkeypatch, "route", _route_ties_to_higher_id)
    must_fail(router_pins.test_topk_matches_bruteforce_with_ties, 0)


def test_router_weights_not_renormalised(monkeypatch):
    plant(monkeypatch, "route", _route_not_renormalised)
    must_fail(router_pins.test_renormalised_weights_sum_to_one)


def test_router_softmax_without_the_max_subtracted(monkeypatch):
    def naive(L):
        with np.errstate(over="ignore", invalid="ignore"):
            ez = np.exp(L)
            return ez / ez.sum(axis=-1, keepdims=True)
    plant(monkeypatch, "_softmax_max_subtracted", naive)
    must_fail(router_pins.test_huge_logits_do_not_overflow)


def test_router_prek_softmax_over_every_expert(monkeypatch):
    plant(monkeypatch, "route", _route_prek_over_all)
    must_fail(router_pins.test_prek_softmax_weights)


def _group_limited_scored_by(score):
    def bad(L, k, n_group, topk_group):
        T, E = L.shape
        gs = E // n_group
        p = REAL["_softmax_max_subtracted"](L)
        kept = np.argsort(-score(L, p, T, n_group, gs), axis=1, kind="stable")[:, :topk_group]
        allowed = np.zeros((T, E), dtype=bool)
        for t in range(T):
            for g in kept[t]:
                allowed[t, g * gs:(g + 1) * gs] = True
        sel = np.argsort(-np.where(allowed, L, -np.inf), axis=1, kind="stable")[:, :k]
        ps = p[np.arange(T)[:, None], sel]
        return sel.astype(np.int32), ps / ps.sum(axis=1, keepdims=True)
    return bad


def test_group_scored_by_its_best_expert(monkeypatch):
    plant(monkeypatch, "_route_group_limited", _group_limited_scored_by(
        lambda L, p, T, n, gs: p.reshape(T, n, gs).max(axis=2)))
    must_fail(group_pins.test_group_of_the_best_expert_can_lose)


def test_group_scored_by_mean_logit(monkeypatch):
    plant(monkeypatch, "_route_group_limited", _group_limited_scored_by(
        lambda L, p, T, n, gs: L.reshape(T, n, gs).mean(axis=2)))
    must_fail(group_pins.test_group_score_is_mean_probability_not_mean_logit)
    must_fail(group_pins.test_worked_example_three_groups)


def test_soft_gating_ignores_the_temperature(monkeypatch):
    plant(monkeypatch, "_route_soft_gumbel",
          lambda L, k, g, tau: REAL["_route_soft_gumbel"](L, k, g, 1.0))
    must_fail(soft_pins.test_two_experts_closed_form)
    must_fail(soft_pins.test_high_temperature_is_uniform)


def test_soft_gating_ignores_the_noise(monkeypatch):
    plant(monkeypatch, "_route_soft_gumbel",
          lambda L, k, g, tau: REAL["_route_soft_gumbel"](L, k, np.zeros(np.shape(g)), tau))
    must_fail(soft_pins.test_low_temperature_is_one_hot_at_the_gumbel_max)


# ---------------------------------------------------------------- dispatch, combine
def _dispatch_unstable(topk_idx, E):
    counts, offsets, pos, src = REAL["dispatch"](topk_idx, E)
    flat = np.asarray(topk_idx).reshape(-1)
    k = np.asarray(topk_idx).shape[1]
    bad = pos.copy()
    for e in range(E):
        members = np.nonzero(flat == e)[0]
        bad[members] = pos[members][::-1]         # last entry first
    src = np.empty_like(src)
    src[bad] = np.arange(flat.size) // k
    return counts, offsets, bad, src


def _dispatch_src_without_k(topk_idx, E):
    counts, offsets, pos, src = REAL["dispatch"](topk_idx, E)
    src = np.empty_like(src)
    src[pos] = np.arange(pos.size)                # the flat index, not the token
    return counts, offsets, pos, src


@pytest.mark.parametrize("bad", [_dispatch_unstable, _dispatch_src_without_k])
def test_dispatch_mistakes(monkeypatch, bad):
    plant(monkeypatch, "dispatch", bad)
    must_fail(dispatch_pins.test_random_routing, 0)


def test_combine_without_weights(monkeypatch):
    plant(monkeypatch, "combine",
          lambda Y, pos, w: REAL["combine"](Y, pos, np.ones_like(np.asarray(w, np.float64))))
    must_fail(ffn_pins.test_combine_matches_loops)


def test_combine_slots_crossed(monkeypatch):
    plant(monkeypatch, "combine",
          lambda Y, pos, w: REAL["combine"](Y, pos, np.asarray(w, np.float64)[:, ::-1]))
    must_fail(ffn_pins.test_combine_matches_loops)


# ---------------------------------------------------------------- FFN, storage roundings
def test_hidden_activation_not_rounded_to_its_storage(monkeypatch):
    plant(monkeypatch, "expert_ffn_rows",
          lambda x, W1e, W2e, h_storage="bf16": REAL["expert_ffn_rows"](x, W1e, W2e, "exact"))
    must_fail(ffn_pins.test_one_expert_bf16_storage_of_h)


def test_relu_for_silu(monkeypatch):
    plant(monkeypatch, "silu", lambda z: np.maximum(z, 0.0))
    must_fail(ffn_pins.test_one_expert_is_a_dense_ffn)


def test_bf16_rounding_keeps_seven_bits(monkeypatch):
    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        m, ex = np.frexp(v)
        return np.where(v == 0.0, v, np.ldexp(np.rint(np.ldexp(m, 7)), ex - 7))
    plant(monkeypatch, "round_to_bf16", bad)
    must_fail(numerics_pins.test_bf16_rounding_matches_torch)


def test_bf16_rounding_truncates(monkeypatch):
    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        m, ex = np.frexp(v)
        return np.where(v == 0.0, v, np.ldexp(np.trunc(np.ldexp(m, 8)), ex - 8))
    plant(monkeypatch, "round_to_bf16", bad)
    must_fail(numerics_pins.test_bf16_rounding_matches_torch)


# ---------------------------------------------------------------- E4M3, FP8 payloads
def test_experts_see_the_rows_before_quantisation(monkeypatch):
    def bad(cfg, x):
        x_hat, q, s = REAL["_payload"](cfg, x)
        return x, q, s                             # the payload computed, then not used
    plant(monkeypatch, "_payload", bad)
    must_fail(ffn_pins.test_fp8_payload_forward)


def test_payload_e4m3_maximum_taken_as_240(monkeypatch):
    monkeypatch.setattr(mo, "E4M3_MAX_F32", np.float32(240.0))
    must_fail(numerics_pins.test_payload_scale_and_saturation)


def test_output_payload_decoded_without_its_zero(monkeypatch):
    plant(monkeypatch, "dequantize_output_fp8",
          lambda q, s, zero: REAL["dequantize_output_fp8"](q, s, np.zeros_like(zero)))
    must_fail(outpay_pins.test_worked_row)
    must_fail(outpay_pins.test_constant_rows_decode_exactly)


def _e4m3_variant(rnd=np.rint, subnormals=True, saturate=True):
    def bad(v):
        v = np.asarray(v, dtype=np.float64)
        a = np.abs(v)
        _, ex = np.frexp(a)
        e = np.maximum(ex - 1, -6) if subnormals else ex - 1
        quantum = np.ldexp(1.0, e - 3)
        r = rnd(a / quantum) * quantum
        if saturate:
            r = np.minimum(r, 448.0)
        r = np.where(a == 0.0, 0.0, r)
        return np.copysign(r, v)
    return bad


@pytest.mark.parametrize("mistake", ["ties_away_from_zero", "no_subnormals"])
def test_e4m3_rounding_mistakes_fail_the_torch_pin(monkeypatch, mistake):
    bad = (_e4m3_variant(rnd=lambda u: np.floor(u + 0.5)) if mistake == "ties_away_from_zero"
           else _e4m3_variant(subnormals=False))
    plant(monkeypatch, "e4m3_round_satfinite", bad)
    must_fail(numerics_pins.test_e4m3_rounding_matches_torch_on_every_bf16_in_range)
    must_fail(numerics_pins.test_e4m3_handworked_values)


def test_e4m3_without_saturation(monkeypatch):
    plant(monkeypatch, "e4m3_round_satfinite", _e4m3_variant(saturate=False))
    must_fail(numerics_pins.test_e4m3_handworked_values)


def test_payload_scale_in_fp64(monkeypatch):
    def bad(x_rows, static_scale=None):
        x = np.asarray(x_rows, np.float64)
        a = np.abs(x).max(axis=1)
        s = np.where(a == 0, 1.0, a / 448.0)      # no fp32 rounding anywhere
        return REAL["e4m3_round_satfinite"](x / s[:, None]), s
    plant(monkeypatch, "quantize_payload_fp8", bad)
    must_fail(numerics_pins.test_payload_scale_and_saturation)


def test_payload_quotient_left_in_fp64(monkeypatch):
    def bad(x_rows, static_scale=None):
        x32 = np.asarray(x_rows, np.float64).astype(np.float32)
        a = np.abs(x32).max(axis=1)
        s = np.where(a == 0, np.float32(1), (a / np.float32(448)).astype(np.float32))
        ratio = x32.astype(np.float64) / s.astype(np.float64)[:, None]   # fp32 scale, fp64 quotient
        return REAL["e4m3_round_satfinite"](ratio), s.astype(np.float64)
    plant(monkeypatch, "quantize_payload_fp8", bad)
    must_fail(numerics_pins.test_payload_quotient_is_rounded_to_fp32_before_e4m3)


def test_output_payload_mapped_onto_zero_to_448(monkeypatch):
    def bad(Y_rows):
        y = np.asarray(Y_rows, np.float64).astype(np.float32)
        mn, mx = y.min(axis=1), y.max(axis=1)
        s = ((mx - mn) / np.float32(448.0)).astype(np.float32)
        s = np.where(mx == mn, np.float32(1.0), s).astype(np.float32)
        q = REAL["e4m3_round_satfinite"](((y - mn[:, None]) / s[:, None]).astype(np.float64))
        return q, s.astype(np.float64), mn.astype(np.float64)
    plant(monkeypatch, "quantize_output_fp8", bad)
    must_fail(outpay_pins.test_worked_row)
    must_fail(outpay_pins.test_matches_torch_e4m3_cast_of_the_fp32_division)


# ---------------------------------------------------------------- backward
def test_router_gradient_not_centred(monkeypatch):
    def bad(L, idx, w, dw, router=0, pre_k=8, tau=1.0):
        dL = np.zeros(np.shape(L))
        dL[np.arange(dL.shape[0])[:, None], np.asarray(idx, np.int64)] = \
            np.asarray(w) * np.asarray(dw)             # the "- sum w dw" term dropped
        return dL
    plant(monkeypatch, "router_backward", bad)
    must_fail(backward_pins.test_finite_differences_renorm, 0)


def test_prek_gradient_only_on_the_chosen(monkeypatch):
    def bad(L, idx, w, dw, router=0, pre_k=8, tau=1.0):
        dL = REAL["router_backward"](L, idx, w, dw, router, pre_k, tau)
        keep = np.zeros(dL.shape, dtype=bool)
        keep[np.arange(dL.shape[0])[:, None], np.asarray(idx, np.int64)] = True
        return np.where(keep, dL, 0.0)                 # the rest of the top pre_k dropped
    plant(monkeypatch, "router_backward", bad)
    must_fail(backward_pins.test_finite_differences_top_prek_softmax, 2)


def test_silu_derivative_is_the_sigmoid(monkeypatch):
    plant(monkeypatch, "silu_grad", lambda z: 1.0 / (1.0 + np.exp(-z)))
    must_fail(backward_pins.test_finite_differences_renorm, 0)


def test_combine_gradient_without_the_weight(monkeypatch):
    def bad(pos, w, Y, g):
        return REAL["_combine_backward"](pos, np.ones_like(w), Y, g)[0], \
            REAL["_combine_backward"](pos, w, Y, g)[1]
    plant(monkeypatch, "_combine_backward", bad)
    must_fail(backward_pins.test_finite_differences_renorm, 0)


def test_dx_without_the_gate_path(monkeypatch):
    def bad(cfg, inp, fwd, dout, h_storage=None):
        r = REAL["backward"](cfg, inp, fwd, dout, h_storage)
        r["dx"] = r["dx"] - r["dL"] @ np.asarray(inp["Wg"], np.float64).T
        return r
    plant(monkeypatch, "backward", bad)
    must_fail(backward_pins.test_finite_differences_renorm, 0)


def test_soft_gating_gradient_without_the_temperature(monkeypatch):
    def bad(L, idx, w, dw, router=0, pre_k=8, tau=1.0):
        return REAL["router_backward"](L, idx, w, dw, router, pre_k, 1.0)
    plant(monkeypatch, "router_backward", bad)
    must_fail(backward_pins.test_finite_differences_soft_gating)


def test_routing_weight_gradient_with_slots_crossed(monkeypatch):
    def bad(pos, w, Y, g):
        dY, dw = REAL["_combine_backward"](pos, w, Y, g)
        return dY, dw[:, ::-1]
    plant(monkeypatch, "_combine_backward", bad)
    must_fail(backward_pins.test_finite_differences_renorm, 0)
