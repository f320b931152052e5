"""Nominal FLOP counts for attention throughput (TFLOP/s) reporting."""
from __future__ import annotations

from .inputs import Workload

# forward = 4*B*H*N^2*d (two N x N x d matmuls), halved under the causal mask.
# 'fwd_bwd' counts forward+backward as 2.5x the forward (the headline count);
# 'fwd_bwd_alg' as 3.5x (forward plus the five backward matmuls); 'bwd' 2.5x.
_MULT = {"fwd": 1.0, "fwd_bwd": 2.5, "fwd_bwd_alg": 3.5, "bwd": 2.5}


def visible_pairs(N: int, causal: bool, window: int = 0) -> float:
    """(query, key) pairs per head the FLOP count charges: N^2, N^2 / 2 under
    the causal mask, and with a causal window W < N the N W - W^2 / 2 pairs of
    the band (the same rounding as N^2 / 2, to which it reduces at W = N)."""
    if not causal:
        return float(N) * N
    if window > 0 and window < N:
        return float(N) * window - float(window) * window / 2.0
    return float(N) * N / 2.0


def attention_flops(w: Workload, passes: str = "fwd") -> float:
    f = 4.0 * w.B * w.H * w.d * visible_pairs(w.N, w.causal, getattr(w, "window", 0))
    return f * _MULT[passes]
