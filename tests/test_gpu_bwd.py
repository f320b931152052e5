"""Backward parity: fa_bwd (the preprocess, the dK/dV kernel with the dQ
reduction, the dQ conversion) on the GPU's own O and LSE, and the
training pair fa_fwd_train + fa_bwd_train, against the fp64 oracle on the same
seeded bf16 inputs.  dQ, dK, dV relative Frobenius error <= 2e-2 each; O and
LSE as in the forward tests."""
import numpy as np
import pytest
import torch

import exact_attention_online_gb300 as fa
from _gpu import GRAD_REL_FRO, check_bwd_groups, check_fwd_heads, f64, run_bwd, run_fwd, stress
from exact_attention_online_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


def small(name, B, H, Hkv, N, d, causal, seed, **kw):
    return Workload(name=name, B=B, H=H, Hkv=Hkv, N=N, d=d, causal=causal, seed=seed, **kw)


SMALL = [
    WORKLOADS["tiny"],
    small("tiny_causal", 1, 1, 1, 128, 64, True, 41),
    small("n1", 1, 2, 1, 1, 64, True, 42),
    small("n33_d128", 1, 2, 2, 33, 128, True, 43),
    small("ragged200_d64", 1, 2, 1, 200, 64, True, 44),
    small("ragged333_d128", 1, 2, 2, 333, 128, True, 45),
    small("ragged257_full_d128", 2, 4, 2, 257, 128, False, 46),
    small("full_d64", 1, 2, 2, 384, 64, False, 47),
    small("tiles512_d128", 1, 2, 1, 512, 128, True, 48),
    small("mqa_d64", 1, 4, 1, 300, 64, True, 49),
    small("gqa_kchan", 1, 4, 2, 384, 128, True, 50, k_outlier_channels=2),
    small("dout_small", 1, 2, 2, 256, 128, True, 51, dout_std=0.1),
]


@pytest.mark.parametrize("precise", [False, True], ids=["bf16out", "precise"])
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_bwd_small_full(w, precise):
    """fa_bwd after fa_fwd, and fa_bwd_precise after fa_fwd_precise."""
    q, k, v, do = make_inputs(w)
    _, _, dev = run_fwd(q, k, v, w.causal, w.scale, precise=precise)
    dq, dk, dv = run_bwd(dev, do, w.causal, w.scale)
    groups = [(b, g) for b in range(w.B) for g in range(w.Hkv)]
    check_bwd_groups(q, k, v, do, dq, dk, dv, w.causal, w.scale, groups)


def test_bwd_dv_column_sum_invariant():
    """Rows of P sum to 1, so sum_j dV_j equals the sum of dO over the group's
    query rows (checked on the GPU result alone, any size)."""
    w = small("inv", 2, 4, 2, 700, 64, True, 52)
    q, k, v, do = make_inputs(w)
    _, _, dev = run_fwd(q, k, v, w.causal, w.scale)
    _, _, dv = run_bwd(dev, do, w.causal, w.scale)
    G = w.H // w.Hkv
    for b in range(w.B):
        for g in range(w.Hkv):
            lhs = f64(dv[b, g]).sum(0)
            rhs = f64(do[b, g * G:(g + 1) * G]).sum(axis=(0, 1))
            assert np.abs(lhs - rhs).max() <= 2e-2 * np.abs(rhs).max() + 0.5


@pytest.mark.parametrize("causal", [True, False], ids=["causal", "full"])
def test_bwd_dkdv_reproducible(causal):
    """dK and dV are the same bit for bit from call to call: at d = 128 the
    even and odd query-block steps of a CTA run in two pipelines whose dV and
    dK MMAs add into the same accumulators, in step order.  Many CTAs, many
    steps each, GQA; five calls."""
    w = small("repro", 2, 8, 2, 2048 + 77, 128, causal, 57)
    q, k, v, do = make_inputs(w)
    _, _, dev = run_fwd(q, k, v, w.causal, w.scale)
    qd, kd, vd, o, lse = dev
    dod = do.cuda()
    first = None
    for _ in range(5):
        g = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=causal, scale=w.scale)
        torch.cuda.synchronize()
        if first is None:
            first = g
        else:
            assert torch.equal(g[1], first[1]) and torch.equal(g[2], first[2])
    assert fa.fa_device_status() == 0


def test_bwd_stages_equal_fused_call():
    """fa_bwd equals fa_bwd_preprocess + fa_bwd_dkdv + fa_bwd_dq_convert."""
    w = small("stages", 1, 4, 2, 300, 128, True, 53)
    q, k, v, do = make_inputs(w)
    _, _, dev = run_fwd(q, k, v, w.causal, w.scale)
    qd, kd, vd, o, lse = dev
    dod = do.cuda()
    dq1, dk1, dv1 = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True, scale=w.scale)
    ws = torch.empty(fa.fa_bwd_workspace_size(1, 4, 2, 300, 128), dtype=torch.uint8,
                     device="cuda")
    dq2, dk2, dv2 = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    fa.fa_bwd_preprocess(o, dod, lse, ws, w.Hkv)
    fa.fa_bwd_dkdv(qd, kd, vd, dod, dk2, dv2, ws, True, w.scale)
    fa.fa_bwd_dq_convert(ws, dq2, w.Hkv, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    assert (dq1.float() - dq2.float()).abs().max() <= 1e-2 * dq1.float().abs().max()


FULL = ["mha_d64", "mha_d64_full", "gpt_long", "gqa"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_bwd_full_size(name):
    """Full workload sizes, same launches as the benchmark (the stress workload
    with key channels x20 through the precise forward and backward); the oracle
    checks one (first) and one (last) key/value group in full (every query head
    of the group, every row)."""
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    _, _, dev = run_fwd(q, k, v, w.causal, w.scale, precise=stress(w))
    dq, dk, dv = run_bwd(dev, do, w.causal, w.scale)
    for t in (dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    groups = [(0, 0)] if w.N >= 8192 else [(0, 0), (w.B - 1, w.Hkv - 1)]
    check_bwd_groups(q, k, v, do, dq, dk, dv, w.causal, w.scale, groups)


def run_train_pair(w, q, k, v, do, precise):
    """fa_fwd_train then fa_bwd_train on a workspace filled with NaN bytes first,
    so that anything the training forward fails to prepare shows."""
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    ws = torch.full((fa.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d),), 0xFF,
                    dtype=torch.uint8, device=dev)
    o = torch.empty(qd.shape, dtype=torch.float32 if precise else torch.bfloat16, device=dev)
    lse = torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    fa.fa_fwd_train(qd, kd, vd, o, lse, ws, w.causal, w.scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    fa.fa_bwd_train(qd, kd, vd, o, dod, dq, dk, dv, ws, w.causal, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return o.cpu(), lse.cpu(), dq.cpu(), dk.cpu(), dv.cpu()


@pytest.mark.parametrize("precise", [False, True], ids=["bf16out", "precise"])
@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_train_pair_small_full(w, precise):
    """fa_fwd_train + fa_bwd_train: the same O, LSE and gradients as the oracle
    (every head, every row)."""
    q, k, v, do = make_inputs(w)
    o, lse, dq, dk, dv = run_train_pair(w, q, k, v, do, precise)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    check_fwd_heads(q, k, v, o, lse, w.causal, w.scale, heads,
                    bf16_bound=stress(w) and not precise)
    groups = [(b, g) for b in range(w.B) for g in range(w.Hkv)]
    check_bwd_groups(q, k, v, do, dq, dk, dv, w.causal, w.scale, groups)


@pytest.mark.parametrize("d", [64, 128])
def test_train_forward_prepares_the_workspace(d):
    """The -LSE table fa_fwd_train writes is bit-identical to the one the
    preprocess writes from the stored LSE (padding rows included), and the
    dQ accumulator it leaves is all zeros."""
    w = small("prep", 2, 3, 1, 300, d, True, 54)
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    n = fa.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d)
    ws1 = torch.full((n,), 0xFF, dtype=torch.uint8, device=dev)
    ws2 = torch.full((n,), 0x7F, dtype=torch.uint8, device=dev)
    o, lse = torch.empty_like(qd), torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    fa.fa_fwd_train(qd, kd, vd, o, lse, ws1, True, w.scale)
    fa.fa_bwd_preprocess(o, dod, lse, ws2, w.Hkv)
    torch.cuda.synchronize()
    rows = w.B * w.H * ((w.N + 127) // 128 * 128)
    a256 = lambda x: (x + 255) // 256 * 256
    ext = rows * 16 * 2
    assert torch.equal(ws1[:ext], ws2[:ext])
    acc0 = 2 * a256(ext)
    acc = ws1[acc0:acc0 + rows * d * 4].view(torch.float32)
    assert torch.count_nonzero(acc).item() == 0


TRAIN_FULL = ["gpt_long", "gqa"]


@pytest.mark.slow
@pytest.mark.parametrize("name", TRAIN_FULL)
def test_train_pair_full_size(name):
    """The training pair the benchmark times, at full size (the stress workload
    through the precise forms): O and LSE of sampled heads, and the gradients
    of the first key/value group in full, against the oracle."""
    w = WORKLOADS[name]
    q, k, v, do = make_inputs(w)
    o, lse, dq, dk, dv = run_train_pair(w, q, k, v, do, precise=stress(w))
    for t in (o, dq, dk, dv):
        assert torch.isfinite(t.float()).all()
    rows = list(range(0, w.N, 97)) + [w.N - 1]
    check_fwd_heads(q, k, v, o, lse, w.causal, w.scale, [(0, 0), (w.B - 1, w.H - 1)],
                    rows=rows)
    check_bwd_groups(q, k, v, do, dq, dk, dv, w.causal, w.scale, [(0, 0)])


def test_train_stages_equal_train_call():
    """fa_bwd_train equals fa_bwd_preprocess_train + fa_bwd_dkdv +
    fa_bwd_dq_convert, and both equal fa_bwd on the same forward (dK, dV
    bit-equal; dQ up to the order of the fp32 reductions)."""
    w = small("tstages", 2, 4, 2, 300, 128, True, 55)
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    n = fa.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d)
    ws = torch.empty(n, dtype=torch.uint8, device=dev)
    o, lse = torch.empty_like(qd), torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    outs = []
    for staged in (False, True):
        fa.fa_fwd_train(qd, kd, vd, o, lse, ws, True, w.scale)
        g = [torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)]
        if staged:
            fa.fa_bwd_preprocess_train(o, dod, ws, w.Hkv)
            fa.fa_bwd_dkdv(qd, kd, vd, dod, g[1], g[2], ws, True, w.scale)
            fa.fa_bwd_dq_convert(ws, g[0], w.Hkv, w.scale)
        else:
            fa.fa_bwd_train(qd, kd, vd, o, dod, *g, ws, True, w.scale)
        outs.append(g)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    ref = fa.attention_backward(qd, kd, vd, o, lse, dod, causal=True, scale=w.scale)
    for dq_, dk_, dv_ in outs:
        assert torch.equal(dk_, ref[1]) and torch.equal(dv_, ref[2])
        assert (dq_.float() - ref[0].float()).abs().max() <= 1e-2 * ref[0].float().abs().max()
