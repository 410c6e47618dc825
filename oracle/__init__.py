"""CPU oracle for one routed mixture-of-experts layer forward.

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import anything under ``oracle/``. The
product path (the CUDA library and its Python binding) never calls it, and the
oracle never calls the product: they share no code except the seeded input
generator in ``workloads``, which holds none of the layer's arithmetic.

The oracle is plain numpy in fp64, written step by step in the order the
source pages give, with no blocking, fusion or reordering:

  gate      L = x W_g + b                   (DeepSeek-V4 EP article, sec. 2.1)
  router    max-subtracted softmax, partial top-8, exact top-k  (same, sec. 3.2);
            optionally limited to the best groups of experts (V3/V4 parallel
            strategy article, EP section); or soft gating: a Gumbel-softmax
            over all experts, none dropped (sync-tax article, sec. 3.3)
  dispatch  per-expert histogram, exclusive scan, stable packing (sec. 3.3;
            Deepseek-MoE sync-tax article, sec. 2.1)
  payload   optional per-token absmax FP8 E4M3                  (sync-tax, sec. 3.1)
  FFN       h = SiLU(x W1_e), y = h W2_e     ("L1 + Act + L2", V3/V4 parallel
            strategy article, Waved-EP section)
  payload   optional FP8 expert outputs, per-row min/max affine (sync-tax, 3.1)
  combine   out_t = sum_j w_tj y_(t,j)       (sync-tax article, sec. 2.3)
  backward  gradients of the above for a given dl/dout, flowing only to the
            chosen experts (DeepSeek-V4 EP article, sec. 2.1; sync-tax, 2.4)

Pins (tests/test_oracle_*.py) tie it to brute force, closed forms, special
cases and library routines; the FFN/combine absolute values are pinned only by
those special cases (dense FFN when E = 1, identical experts, linearity).
"""
from .moe_oracle import (  # noqa: F401
    gate_logits, route, dispatch, quantize_payload_fp8, quantize_output_fp8,
    dequantize_output_fp8, expert_ffn_rows,
    combine, forward, forward_tokens, inputs_to_numpy, backward, backward_tokens,
    backward_router, backward_expert, router_backward,
    silu_grad, ROUTER_RENORM,
    ROUTER_PREK_SOFTMAX, ROUTER_GROUP_LIMITED, ROUTER_SOFT_GUMBEL,
)
from .numerics import (  # noqa: F401
    round_to_bf16, round_to_f32, e4m3_round_satfinite, e4m3_encode, e4m3_decode,
)
