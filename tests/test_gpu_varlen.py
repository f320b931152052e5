"""Packed variable-length batches on the GPU, through the C ABI
(fa_fwd_varlen, fa_bwd_varlen), against the fp64 oracle's packed attention
(each sequence its own problem) on the same seeded bf16 inputs: O max abs
<= 1e-2, LSE max abs <= 1e-3, dQ/dK/dV relative Frobenius <= 2e-2."""
import numpy as np
import pytest
import torch

import exact_attention_online_gb300 as fa
import oracle
from _gpu import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, f64, rel_fro
from exact_attention_online_gb300.inputs import (VARLEN_WORKLOADS, VarlenWorkload,
                                                 make_varlen_inputs)

pytestmark = pytest.mark.gpu


def wl(name, lens, H, Hkv, d, causal, seed):
    return VarlenWorkload(name=name, lens=tuple(lens), H=H, Hkv=Hkv, d=d, causal=causal,
                          seed=seed)


# Ragged lengths around the 128-row tiles and the 256-row query-block pairs,
# an empty sequence, one-row sequences, MQA/GQA, both head dims and masks.
SMALL = [
    wl("mix_d64_causal", [1, 130, 0, 257, 64, 511], 2, 1, 64, True, 601),
    wl("mix_d128_causal", [300, 17, 128, 256, 1], 4, 2, 128, True, 602),
    wl("mix_d64_full", [77, 385, 200], 3, 3, 64, False, 603),
    wl("mix_d128_full", [129, 1, 640, 33], 2, 1, 128, False, 604),
    wl("mqa_long_short", [1000, 3, 260], 4, 1, 128, True, 605),
    wl("single", [700], 2, 2, 64, True, 606),
]


def run(w, max_seqlen=None, dout=True):
    q, k, v, do = make_varlen_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    cu = w.cu_seqlens().to(dev)
    ms = w.max_seqlen if max_seqlen is None else max_seqlen
    o, lse = fa.attention_varlen(qd, kd, vd, cu, ms, w.causal, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    grads = None
    if dout:
        grads = fa.attention_varlen_backward(qd, kd, vd, o, lse, dod, cu, ms, w.causal, w.scale)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        grads = tuple(t.cpu() for t in grads)
    return (q, k, v, do), o.cpu(), lse.cpu(), grads


def check(w, ins, o, lse, grads, rows=None):
    """Against the oracle; rows (optional) = the sequences to compare."""
    q, k, v, do = ins
    cu = w.cu_seqlens().numpy()
    seqs = range(w.B) if rows is None else rows
    for b in seqs:
        a, e = int(cu[b]), int(cu[b + 1])
        if e == a:
            continue
        sub = np.array([0, e - a])
        ro, rl = oracle.attn_fwd_varlen(f64(q[:, a:e]), f64(k[:, a:e]), f64(v[:, a:e]), sub,
                                        w.causal, w.scale)
        assert np.abs(f64(o[:, a:e]) - ro).max() <= O_MAX_ABS, f"O, sequence {b}"
        assert np.abs(lse[:, a:e].double().numpy() - rl).max() <= LSE_MAX_ABS, f"LSE, seq {b}"
        if grads is None:
            continue
        rq, rk, rv, _ = oracle.attn_bwd_varlen(f64(q[:, a:e]), f64(k[:, a:e]), f64(v[:, a:e]),
                                               f64(do[:, a:e]), sub, w.causal, w.scale)
        for name, got, ref in (("dq", grads[0], rq), ("dk", grads[1], rk), ("dv", grads[2], rv)):
            err = rel_fro(got[:, a:e], ref)
            assert err <= GRAD_REL_FRO, f"{name} sequence {b}: relative Frobenius {err:.3e}"


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_varlen_small(w):
    ins, o, lse, grads = run(w)
    check(w, ins, o, lse, grads)
    # the whole packed batch at once, through the oracle's own packing
    q, k, v, do = ins
    ro, rl = oracle.attn_fwd_varlen(f64(q), f64(k), f64(v), w.cu_seqlens().numpy(), w.causal,
                                    w.scale)
    assert np.abs(f64(o) - ro).max() <= O_MAX_ABS
    assert np.abs(lse.double().numpy() - rl).max() <= LSE_MAX_ABS


def test_varlen_larger_max_seqlen_same_result():
    """max_seqlen above the longest sequence only adds work items that have no
    rows: the outputs are the same bit for bit (dQ up to the order of its fp32
    additions)."""
    w = SMALL[0]
    _, o1, l1, g1 = run(w)
    _, o2, l2, g2 = run(w, max_seqlen=w.max_seqlen + 300)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(g1[1], g2[1]) and torch.equal(g1[2], g2[2])
    assert rel_fro(g1[0], f64(g2[0])) <= 1e-3


def test_varlen_equal_lengths_match_dense():
    """Equal lengths: the packed batch is the dense batch laid out head-major;
    the same tiles and masks give the dense kernels' O, LSE, dK and dV bit for
    bit."""
    B, N, H, d = 3, 333, 2, 64
    w = wl("equal", [N] * B, H, H, d, True, 607)
    ins, o, lse, grads = run(w)
    q, k, v, do = ins
    dense = lambda x: x.reshape(x.shape[0], B, N, d).transpose(0, 1).contiguous()
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (dense(t).to(dev) for t in (q, k, v, do))
    od, ld = fa.attention(qd, kd, vd, causal=True, scale=w.scale)
    gd = fa.attention_backward(qd, kd, vd, od, ld, dod, causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(dense(o), od.cpu())
    assert torch.equal(lse.reshape(H, B, N).transpose(0, 1), ld.cpu())
    assert torch.equal(dense(grads[1]), gd[1].cpu()) and torch.equal(dense(grads[2]), gd[2].cpu())
    assert rel_fro(dense(grads[0]), f64(gd[0].cpu())) <= 1e-3


def test_varlen_backward_reads_only_what_the_preprocess_writes():
    """The preprocess writes a sequence's workspace rows only up to its length
    rounded up to 128, not up to max_seqlen: a workspace filled with NaN bytes
    and one filled with zeros give the same gradients (dK, dV bit for bit, dQ
    up to the order of its fp32 additions), so nothing past those rows is
    read.  Mixed lengths, with max_seqlen well above the longest one."""
    for w in (SMALL[0], SMALL[4]):
        q, k, v, do = make_varlen_inputs(w)
        dev = torch.device("cuda:0")
        qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
        cu = w.cu_seqlens().to(dev)
        ms = w.max_seqlen + 200
        o, lse = fa.attention_varlen(qd, kd, vd, cu, ms, w.causal, w.scale)
        n = fa.fa_bwd_varlen_workspace_size(w.B, w.H, w.Hkv, ms, w.d)
        out = []
        for fill in (0xFF, 0x00):
            ws = torch.full((n,), fill, dtype=torch.uint8, device=dev)
            out.append(fa.attention_varlen_backward(qd, kd, vd, o, lse, dod, cu, ms, w.causal,
                                                    w.scale, workspace=ws))
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        (dq1, dk1, dv1), (dq2, dk2, dv2) = ([t.cpu() for t in g] for g in out)
        for t in (dq1, dk1, dv1):
            assert torch.isfinite(t.float()).all()
        assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
        assert rel_fro(dq1, f64(dq2)) <= 1e-3


def test_varlen_rejects():
    dev = torch.device("cuda:0")
    q = torch.zeros((2, 100, 64), dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty((2, 100), dtype=torch.float32, device=dev)
    cu = torch.tensor([0, 100], dtype=torch.int32, device=dev)
    lib = fa.lib()
    import ctypes
    p = lambda t: ctypes.c_void_p(t.data_ptr())
    st = lib.fa_fwd_varlen(p(q), p(q), p(q), p(o), p(lse), None, 1, 100, 100, 2, 2, 64, 1,
                           0.125, None)
    assert st == fa.FA_ERR_INVALID_ARG
    st = lib.fa_fwd_varlen(p(q), p(q), p(q), p(o), p(lse), p(cu), 1, 100, 0, 2, 2, 64, 1,
                           0.125, None)
    assert st == fa.FA_ERR_INVALID_ARG
    st = lib.fa_fwd_varlen(p(q), p(q), p(q), p(o), p(lse), p(cu), 1, 100, 100, 2, 2, 96, 1,
                           0.125, None)
    assert st == fa.FA_ERR_UNSUPPORTED


def test_varlen_offsets_out_of_range_stay_in_bounds():
    """Offsets that break the rules (a sequence longer than max_seqlen, one
    running past the end of the tensor) give unspecified values but no access
    outside the tensors: rows outside every clamped sequence are left as they
    were, and the context still works."""
    dev = torch.device("cuda:0")
    H, T, d = 2, 300, 64
    q = torch.randn((H, T, d), device=dev).to(torch.bfloat16)
    o = torch.full_like(q, 7.0)
    lse = torch.full((H, T), 7.0, dtype=torch.float32, device=dev)
    cu = torch.tensor([0, 200, 450], dtype=torch.int32, device=dev)   # 2nd runs past T
    fa.fa_fwd_varlen(q, q, q, o, lse, cu, 128, True, 0.125)   # 1st longer than max_seqlen
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    oc = o.cpu()
    # sequence 0 clamped to 128 rows: rows 128..199 untouched
    assert torch.all(oc[:, 128:200] == 7.0)
    x = torch.ones(4, device=dev) * 2
    assert float(x.sum()) == 8.0


@pytest.mark.slow
def test_varlen_full_size():
    """The benchmark's packed batch (16 causal sequences of 128-4096 tokens,
    H 16, d 128), the same launches; the oracle checks the first, the
    shortest and the last sequence in full (every head, every row)."""
    w = VARLEN_WORKLOADS["varlen"]
    ins, o, lse, grads = run(w)
    for t in (o,) + grads:
        assert torch.isfinite(t.float()).all()
    shortest = int(np.argmin(w.lens))
    check(w, ins, o, lse, grads, rows=sorted({0, shortest, w.B - 1}))
