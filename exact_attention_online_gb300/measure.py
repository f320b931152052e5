"""Nominal FLOP counts for attention throughput (TFLOP/s) reporting."""
from __future__ import annotations

from .inputs import Workload

# forward = 4*B*H*N^2*d (two N x N x d matmuls), halved under the causal mask.
# 'fwd_bwd' counts forward+backward as 2.5x the forward (the headline count);
# 'fwd_bwd_alg' as 3.5x (forward plus the five backward matmuls); 'bwd' 2.5x.
_MULT = {"fwd": 1.0, "fwd_bwd": 2.5, "fwd_bwd_alg": 3.5, "bwd": 2.5}


def attention_flops(w: Workload, passes: str = "fwd") -> float:
    f = 4.0 * w.B * w.H * w.N * w.N * w.d
    if w.causal:
        f /= 2.0
    return f * _MULT[passes]
