"""Roofline and score arithmetic -- TEST INFRASTRUCTURE ONLY.

Restated from muse_bf16_proj guide, ch. 1 "The problem, the judge and the
speed of light":
  * §1.7 "The speed of light": floor = max(bytes / bandwidth, FLOPs / peak),
    FLOPs = 2 * m * N * K (one multiply and one add per weight per token);
  * §1.3 "How the score is computed": a load's time is the sum of its five
    shapes; a load's speedup is the baseline time over ours; the score is the
    geometric mean of the six load speedups.

Bytes per shape (reading of §1.7, which counts weights plus "x and out"):
weights + x + out, with out in the layer's output dtype.
"""
from __future__ import annotations

import math


def shape_bytes(N_rows: int, K: int, m: int, w_bytes: float, out_bytes: int) -> float:
    """Weight bytes of the rows computed + bf16 x + output."""
    return N_rows * K * w_bytes + m * K * 2 + m * N_rows * out_bytes


def shape_flops(N_rows: int, K: int, m: int) -> float:
    return 2.0 * m * N_rows * K


def floor_seconds(bytes_moved: float, flops: float, bw_bytes_per_s: float,
                  flops_per_s: float) -> float:
    return max(bytes_moved / bw_bytes_per_s, flops / flops_per_s)


def score(baseline_load_us, ours_load_us) -> float:
    """Geometric mean over loads of baseline / ours."""
    ratios = [b / o for b, o in zip(baseline_load_us, ours_load_us)]
    return math.exp(sum(math.log(r) for r in ratios) / len(ratios))
