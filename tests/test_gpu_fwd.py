"""Forward parity: the sm_103a forward kernel (through the C ABI) against the
fp64 oracle on the same seeded bf16 inputs.  O max abs error <= 1e-2 and LSE
max abs error <= 1e-3."""
import numpy as np
import pytest
import torch

import oracle
from _gpu import check_fwd_heads, f64, run_fwd, sample_rows, stress
from exact_attention_online_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


def small(name, B, H, Hkv, N, d, causal, seed, **kw):
    return Workload(name=name, B=B, H=H, Hkv=Hkv, N=N, d=d, causal=causal, seed=seed, **kw)


# Small cases the oracle checks in full: several tiles, ragged tails, N = 1,
# MQA/GQA, both head dims, both masks.
SMALL = [
    WORKLOADS["tiny"],
    small("tiny_causal", 1, 1, 1, 128, 64, True, 11),
    small("n1", 1, 2, 1, 1, 64, False, 12),
    small("n1_causal_d128", 1, 2, 2, 1, 128, True, 13),
    small("n17", 2, 2, 1, 17, 128, True, 14),
    small("ragged200_d64", 1, 2, 1, 200, 64, True, 15),
    small("ragged333_d128", 1, 2, 2, 333, 128, True, 16),
    small("ragged257_full", 2, 4, 2, 257, 128, False, 17),
    small("tiles512_d64", 1, 2, 2, 512, 64, True, 18),
    small("tiles640_d128", 1, 1, 1, 640, 128, True, 19),
    small("mqa", 1, 4, 1, 300, 128, True, 20),
    small("full_d64_ragged", 1, 3, 3, 385, 64, False, 21),
    small("outliers", 1, 2, 1, 500, 128, True, 22, outlier_frac=1e-3),
    small("kchan", 1, 4, 2, 384, 128, True, 23, k_outlier_channels=2),
]


@pytest.mark.parametrize("precise", [False, True], ids=["bf16out", "precise"])
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fwd_small_full(w, precise):
    """bf16 output: O within 1e-2 (stress inputs - outliers of magnitude 30,
    key channels x20 - within the bf16 rounding bound, see
    _gpu.bf16_output_bound).  fa_fwd_precise: O within 1e-2 on every input."""
    q, k, v, _ = make_inputs(w, with_dout=False)
    o, lse, _ = run_fwd(q, k, v, w.causal, w.scale, precise=precise)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    check_fwd_heads(q, k, v, o, lse, w.causal, w.scale, heads,
                    bf16_bound=(stress(w) and not precise))


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_fwd_precise_rounding_bound(w):
    """fa_fwd_precise forms P V in fp16: each p is rounded to 11 significant
    bits (relative error <= 2^-11), V's bf16 values are exact in fp16, and O is
    fp32.  With weights w = p / l and the row sum corrected for the rounding of
    each block's largest p, a row of O moves by at most 2^-11 (sum over block
    maxima of w |v - O| + sum over the rest of w |v|) <= 2^-10 max|V| from the
    rounding of P; 1e-3 is left for the fp32 score, exponential and
    accumulation errors."""
    q, k, v, _ = make_inputs(w, with_dout=False)
    o, _, _ = run_fwd(q, k, v, w.causal, w.scale, precise=True)
    G = w.H // w.Hkv
    for b in range(w.B):
        for h in range(w.H):
            vh = f64(v[b:b + 1, h // G:h // G + 1])
            ro, _ = oracle.attn_fwd(f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, h // G:h // G + 1]),
                                    vh, w.causal, w.scale)
            err = np.abs(f64(o[b, h]) - ro[0, 0]).max()
            assert err <= 2.0 ** -10 * np.abs(vh).max() + 1e-3, (b, h, err)


def test_fwd_causal_row0_exact():
    """With the causal mask query 0 sees only key 0: O_0 = V_0 bit for bit and
    LSE_0 = scale*<q_0,k_0>."""
    w = small("row0", 2, 4, 2, 300, 128, True, 30)
    q, k, v, _ = make_inputs(w, with_dout=False)
    o, lse, _ = run_fwd(q, k, v, True, w.scale)
    G = w.H // w.Hkv
    for b in range(w.B):
        for h in range(w.H):
            assert torch.equal(o[b, h, 0], v[b, h // G, 0])
            want = w.scale * float(f64(q[b, h, 0]) @ f64(k[b, h // G, 0]))
            assert abs(float(lse[b, h, 0]) - want) <= 1e-4


def heads_to_check(w, seed=0):
    rng = np.random.default_rng(seed)
    last = (w.B - 1, w.H - 1)
    rand = (int(rng.integers(w.B)), int(rng.integers(w.H)))
    return sorted({(0, 0), last, rand})


FULL = ["mha_d64", "mha_d64_full", "gpt_long", "gqa", "long16k", "long32k", "ablation"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_fwd_full_size(name):
    """Full workload sizes, the same launch as the benchmark; the oracle checks
    whole heads (first, last, one random) for N <= 8192 and sampled rows of
    those heads beyond.  The stress workloads (outliers of magnitude 30, key
    channels x20) run fa_fwd_precise (fp32 O), as the benchmark does for them."""
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w, with_dout=False)
    precise = stress(w)
    o, lse, _ = run_fwd(q, k, v, w.causal, w.scale, precise=precise)
    assert torch.isfinite(o.float()).all() and torch.isfinite(lse).all()
    heads = heads_to_check(w)
    rows = None if w.N <= 8192 else sample_rows(w.N, seed=w.seed)
    if w.N == 8192:
        heads = heads[:2]
    check_fwd_heads(q, k, v, o, lse, w.causal, w.scale, heads, rows=rows)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["long16k", "gqa"])
def test_fwd_full_size_bf16_output_bound(name):
    """The bf16-output forward on the stress workloads: within 1e-2 plus its
    bf16 rounding bound (2^-8 (max|V| + |O|))."""
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w, with_dout=False)
    o, lse, _ = run_fwd(q, k, v, w.causal, w.scale)
    rows = None if w.N <= 8192 else sample_rows(w.N, seed=w.seed)
    check_fwd_heads(q, k, v, o, lse, w.causal, w.scale, heads_to_check(w)[:2],
                    rows=rows, bf16_bound=True)
