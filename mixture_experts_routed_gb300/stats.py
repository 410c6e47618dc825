"""Host-side load statistics of one routing (from the per-expert row counts
the dispatch produces).

The pages report these quantities for real training runs: per-expert
activation rates against the ideal 1/E (DeepSeek-V4 EP article, section 6.2:
64 experts, ideal 1.56%) and the entropy of the expert load (Deepseek-MoE
sync-tax article, section 5.1: 3.89 bits against the ideal 4.0 for 16
experts).
"""
from __future__ import annotations

import math


def load_stats(counts) -> dict:
    """counts: per-expert routed-row counts (any int sequence / tensor)."""
    c = [int(v) for v in (counts.tolist() if hasattr(counts, "tolist") else counts)]
    E = len(c)
    R = sum(c)
    if E == 0:
        raise ValueError("no experts")
    mean = R / E
    shares = [v / R for v in c] if R else [0.0] * E
    entropy = -sum(p * math.log2(p) for p in shares if p > 0)
    return {
        "experts": E,
        "rows": R,
        "max_over_mean": (max(c) / mean) if R else 0.0,
        "zero_experts": sum(1 for v in c if v == 0),
        "max_share": max(shares),
        "min_share": min(shares),
        "ideal_share": 1.0 / E,
        "entropy_bits": entropy,
        "ideal_entropy_bits": math.log2(E),
    }
