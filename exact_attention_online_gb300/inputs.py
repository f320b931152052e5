"""Seeded synthetic inputs for the attention workloads.

This module only draws random numbers and shapes them; it holds none of the
attention arithmetic.  Both the CUDA-path tests and the oracle tests draw
their inputs here, so the two sides see the same bf16 values.

Recipe (all tensors drawn in fp32 on the CPU from one ``torch.Generator``
seeded with ``seed``, in the order Q, K, V, dO, then rounded to bf16 with
round-to-nearest-even):
  * Q, K, V, dO ~ N(0, 1) elementwise, dO optionally scaled by ``dout_std``.
  * ``k_outlier_channels`` > 0: that many head-dim channels of every key/value
    head are chosen with the same generator and multiplied by
    ``k_outlier_gain`` at every position and batch (before rounding).
  * ``outlier_frac`` > 0: independently for Q, K and V, round(frac * numel)
    element positions are chosen with the same generator and replaced by
    +-``outlier_mag`` with a random sign.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


@dataclass(frozen=True)
class Workload:
    """One attention problem: shapes, mask and input distribution."""
    name: str
    B: int
    H: int
    Hkv: int
    N: int
    d: int
    causal: bool
    seed: int
    dout_std: float = 1.0
    k_outlier_channels: int = 0
    k_outlier_gain: float = 20.0
    outlier_frac: float = 0.0
    outlier_mag: float = 30.0
    window: int = 0            # causal sliding window W (query i sees i - W < j <= i); 0 = none
    passes: tuple = ("fwd", "bwd")
    tags: tuple = field(default_factory=tuple)

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


def _cfg(idx: int, name: str, **kw) -> Workload:
    return Workload(name=name, seed=1000 + idx, **kw)


# The five attention workloads of the pages' setting (sizes, masks and value
# distributions), plus the FlashAttention-2 ablation shape.
WORKLOADS = {
    "tiny": _cfg(1, "tiny", B=1, H=1, Hkv=1, N=128, d=64, causal=False),
    "mha_d64": _cfg(2, "mha_d64", B=8, H=16, Hkv=16, N=2048, d=64, causal=True),
    "mha_d64_full": _cfg(2, "mha_d64_full", B=8, H=16, Hkv=16, N=2048, d=64, causal=False),
    "gpt_long": _cfg(3, "gpt_long", B=2, H=16, Hkv=16, N=8192, d=128, causal=True,
                     dout_std=0.1),
    "gqa": _cfg(4, "gqa", B=4, H=32, Hkv=8, N=4096, d=128, causal=True,
                k_outlier_channels=2),
    "long16k": _cfg(5, "long16k", B=1, H=16, Hkv=16, N=16384, d=128, causal=True,
                    outlier_frac=1e-3, passes=("fwd",)),
    "long32k": _cfg(5, "long32k", B=1, H=16, Hkv=16, N=32768, d=128, causal=True,
                    outlier_frac=1e-3, passes=("fwd",)),
    "ablation": _cfg(6, "ablation", B=8, H=16, Hkv=16, N=2048, d=128, causal=True,
                     passes=("fwd",)),
    # Local (sliding-window) attention, the variant the pages name for
    # Mistral-7B: that model's attention shape (32 query heads, 8 key/value
    # heads, d = 128) with a 4096-key window over a 16K sequence.
    "window": _cfg(7, "window", B=1, H=32, Hkv=8, N=16384, d=128, causal=True, window=4096),
}


def _channel_pick(gen: torch.Generator, d: int, n: int) -> torch.Tensor:
    return torch.randperm(d, generator=gen)[:n]


def _outliers(x: torch.Tensor, gen: torch.Generator, frac: float, mag: float) -> None:
    n = int(round(frac * x.numel()))
    if n == 0:
        return
    flat = x.view(-1)
    pos = torch.randperm(flat.numel(), generator=gen)[:n]
    sign = torch.randint(0, 2, (n,), generator=gen).to(torch.float32) * 2 - 1
    flat[pos] = sign * mag


def make_inputs(w: Workload, with_dout: bool = True):
    """Return (q, k, v, dout) as CPU bf16 tensors in [B, H(kv), N, d] layout.

    dout is None when ``with_dout`` is False (it is still drawn, so the other
    tensors do not depend on that flag).
    """
    gen = torch.Generator().manual_seed(int(w.seed))
    q = torch.randn((w.B, w.H, w.N, w.d), generator=gen, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.N, w.d), generator=gen, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.N, w.d), generator=gen, dtype=torch.float32)
    dout = torch.randn((w.B, w.H, w.N, w.d), generator=gen, dtype=torch.float32)
    if w.dout_std != 1.0:
        dout.mul_(w.dout_std)
    if w.k_outlier_channels:
        for g in range(w.Hkv):
            ch = _channel_pick(gen, w.d, w.k_outlier_channels)
            k[:, g, :, ch] *= w.k_outlier_gain
    if w.outlier_frac:
        for t in (q, k, v):
            _outliers(t, gen, w.outlier_frac, w.outlier_mag)
    out = [t.to(torch.bfloat16) for t in (q, k, v)]
    out.append(dout.to(torch.bfloat16) if with_dout else None)
    return tuple(out)


# ------------------------------------------------------------------ decoding
@dataclass(frozen=True)
class DecodeWorkload:
    """Nq new query rows against a cache of Nk keys and values (the queries
    are the last Nq positions)."""
    name: str
    B: int
    H: int
    Hkv: int
    Nq: int
    Nk: int
    d: int
    causal: bool
    seed: int

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)


# Decoding shapes (the pages describe the setting, not sizes): a GQA model
# decoding one token per sequence against a 32K cache (1.07 GB of K and V), a
# speculative step of 4 tokens against a 16K cache, and an MHA d = 64 step.
DECODE_WORKLOADS = {
    "decode_gqa": DecodeWorkload("decode_gqa", B=8, H=32, Hkv=8, Nq=1, Nk=32768, d=128,
                                 causal=True, seed=1101),
    "decode_spec4": DecodeWorkload("decode_spec4", B=8, H=32, Hkv=8, Nq=4, Nk=16384, d=128,
                                   causal=True, seed=1102),
    "decode_mha_d64": DecodeWorkload("decode_mha_d64", B=16, H=16, Hkv=16, Nq=1, Nk=8192, d=64,
                                     causal=True, seed=1103),
}


def make_decode_inputs(w: DecodeWorkload):
    """(q [B, H, Nq, d], k, v [B, Hkv, Nk, d]) as CPU bf16 tensors: one
    torch.Generator seeded with w.seed, N(0, 1) fp32 draws in the order Q, K,
    V, rounded to bf16 (round to nearest even)."""
    gen = torch.Generator().manual_seed(int(w.seed))
    q = torch.randn((w.B, w.H, w.Nq, w.d), generator=gen, dtype=torch.float32)
    k = torch.randn((w.B, w.Hkv, w.Nk, w.d), generator=gen, dtype=torch.float32)
    v = torch.randn((w.B, w.Hkv, w.Nk, w.d), generator=gen, dtype=torch.float32)
    return tuple(t.to(torch.bfloat16) for t in (q, k, v))


# ------------------------------------------------------------ packed batches
@dataclass(frozen=True)
class VarlenWorkload:
    """B sequences of different lengths packed without padding: q, dO
    [H][total][d], k, v [Hkv][total][d], sequence b at rows cu[b] .. cu[b+1] - 1."""
    name: str
    lens: tuple
    H: int
    Hkv: int
    d: int
    causal: bool
    seed: int

    @property
    def B(self) -> int:
        return len(self.lens)

    @property
    def total(self) -> int:
        return int(sum(self.lens))

    @property
    def max_seqlen(self) -> int:
        return int(max(self.lens))

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.d)

    def cu_seqlens(self) -> torch.Tensor:
        cu = [0]
        for n in self.lens:
            cu.append(cu[-1] + int(n))
        return torch.tensor(cu, dtype=torch.int32)


def varlen_lengths(n: int, lo: int, hi: int, seed: int) -> tuple:
    """n lengths drawn uniformly from [lo, hi] by a torch.Generator seeded
    with `seed` (the mix of a packed training batch)."""
    gen = torch.Generator().manual_seed(int(seed))
    return tuple(int(x) for x in torch.randint(lo, hi + 1, (n,), generator=gen))


# A packed causal training batch: 16 sequences of 128 to 4096 tokens (about
# 33K tokens), the GPT-style head shape of the long workloads (16 heads,
# d = 128).
VARLEN_WORKLOADS = {
    "varlen": VarlenWorkload("varlen", lens=varlen_lengths(16, 128, 4096, 1208), H=16, Hkv=16,
                             d=128, causal=True, seed=1008),
}


def make_varlen_inputs(w: VarlenWorkload):
    """(q, k, v, dout) as CPU bf16 tensors in the packed layout: one
    torch.Generator seeded with w.seed, N(0, 1) fp32 draws in the order Q, K,
    V, dO, rounded to bf16 (round to nearest even)."""
    gen = torch.Generator().manual_seed(int(w.seed))
    q = torch.randn((w.H, w.total, w.d), generator=gen, dtype=torch.float32)
    k = torch.randn((w.Hkv, w.total, w.d), generator=gen, dtype=torch.float32)
    v = torch.randn((w.Hkv, w.total, w.d), generator=gen, dtype=torch.float32)
    dout = torch.randn((w.H, w.total, w.d), generator=gen, dtype=torch.float32)
    return tuple(t.to(torch.bfloat16) for t in (q, k, v, dout))
