"""Causal sliding-window ("local") attention on the GPU, through the C ABI
(fa_fwd_window, fa_bwd_window), against the fp64 oracle's windowed attention
on the same seeded bf16 inputs: O max abs <= 1e-2, LSE max abs <= 1e-3,
dQ/dK/dV relative Frobenius <= 2e-2.

At the full workload size the oracle runs on slices of the sequence: rows of
windowed attention depend only on the W keys before them, so the oracle on
positions [s, e) gives the exact forward of every row i >= s + W - 1 (and of
every row when s = 0), dQ of the same rows, and dK, dV of keys j with
s + W - 1 <= j and (j + W <= e or e = N).
"""
import numpy as np
import pytest
import torch

import exact_attention_online_gb300 as fa
import oracle
from _gpu import GRAD_REL_FRO, LSE_MAX_ABS, O_MAX_ABS, f64, rel_fro
from exact_attention_online_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu


def small(name, B, H, Hkv, N, d, window, seed):
    return Workload(name=name, B=B, H=H, Hkv=Hkv, N=N, d=d, causal=True, seed=seed,
                    window=window)


# Several tiles, ragged tails, windows below, at and above the 128-key block,
# a window that is not a block multiple, a window >= N (plain causal), MQA/GQA.
SMALL = [
    small("w1_d64", 1, 2, 1, 300, 64, 1, 501),
    small("w1_d128", 1, 2, 2, 300, 128, 1, 502),
    small("w64_d64", 1, 2, 2, 600, 64, 64, 503),
    small("w128_d128", 1, 2, 1, 640, 128, 128, 504),
    small("w129_d64", 2, 2, 1, 517, 64, 129, 505),
    small("w300_d128", 1, 4, 2, 1000, 128, 300, 506),
    small("w200_mqa", 1, 4, 1, 777, 128, 200, 507),
    small("w256_d64_ragged", 1, 3, 3, 1111, 64, 256, 508),
    small("w_ge_n", 1, 2, 1, 333, 128, 5000, 509),
    small("n1", 1, 2, 2, 1, 64, 3, 510),
    small("n100_w7", 2, 2, 2, 100, 128, 7, 511),
]


def run(w, q, k, v, dout=None):
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    o, lse = fa.attention_window(qd, kd, vd, w.window, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    grads = None
    if dout is not None:
        grads = fa.attention_window_backward(qd, kd, vd, o, lse, dout.to(dev), w.window, w.scale)
        torch.cuda.synchronize()
        assert fa.fa_device_status() == 0
        grads = tuple(t.cpu() for t in grads)
    return o.cpu(), lse.cpu(), grads


@pytest.mark.parametrize("w", SMALL, ids=lambda w: w.name)
def test_window_small_full(w):
    q, k, v, do = make_inputs(w)
    o, lse, (dq, dk, dv) = run(w, q, k, v, do)
    ro, rl = oracle.attn_fwd_window(f64(q), f64(k), f64(v), w.window, w.scale)
    assert np.abs(f64(o) - ro).max() <= O_MAX_ABS
    assert np.abs(lse.double().numpy() - rl).max() <= LSE_MAX_ABS
    rq, rk, rv, _ = oracle.attn_bwd_window(f64(q), f64(k), f64(v), f64(do), w.window, w.scale)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = rel_fro(got, ref)
        assert e <= GRAD_REL_FRO, f"{name} relative Frobenius error {e:.3e}"


@pytest.mark.parametrize("w", [SMALL[3], SMALL[5], SMALL[6], SMALL[7]], ids=lambda w: w.name)
def test_window_train_pair_equals_window_pair(w):
    """fa_fwd_window_train + fa_bwd_window_train on a workspace of NaN bytes
    give the O, LSE, dK and dV of fa_fwd_window + fa_bwd_window bit for bit
    and the same dQ up to the order of its fp32 additions: the training
    forward leaves the backward a complete workspace."""
    q, k, v, do = make_inputs(w)
    dev = torch.device("cuda:0")
    qd, kd, vd, dod = (t.to(dev) for t in (q, k, v, do))
    n = fa.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d)
    ws = torch.full((n,), 0xFF, dtype=torch.uint8, device=dev)
    o, lse = torch.empty_like(qd), torch.empty((w.B, w.H, w.N), dtype=torch.float32, device=dev)
    fa.fa_fwd_window_train(qd, kd, vd, o, lse, ws, w.window, w.scale)
    dq, dk, dv = torch.empty_like(qd), torch.empty_like(kd), torch.empty_like(vd)
    fa.fa_bwd_window_train(qd, kd, vd, o, dod, dq, dk, dv, ws, w.window, w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    o2, l2 = fa.attention_window(qd, kd, vd, w.window, w.scale)
    g2 = fa.attention_window_backward(qd, kd, vd, o2, l2, dod, w.window, w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o, o2) and torch.equal(lse, l2)
    assert torch.equal(dk, g2[1]) and torch.equal(dv, g2[2])
    assert rel_fro(dq.cpu(), f64(g2[0].cpu())) <= 1e-3
    rq, rk, rv, _ = oracle.attn_bwd_window(f64(q), f64(k), f64(v), f64(do), w.window, w.scale)
    for name, got, ref in (("dq", dq, rq), ("dk", dk, rk), ("dv", dv, rv)):
        e = rel_fro(got.cpu(), ref)
        assert e <= GRAD_REL_FRO, f"{name} relative Frobenius error {e:.3e}"


def test_window_one_is_value_row():
    """W = 1: each query sees only its own key, so O_i = V_i bit for bit, LSE_i
    = scale <q_i, k_i>, dV_i = dO_i (up to bf16 rounding of the fp32 sum of
    one term) and dQ = dK = 0 (P = 1 gives dS = P (dP - D) = 0 exactly in
    exact arithmetic)."""
    w = small("w1", 1, 2, 2, 260, 128, 1, 520)
    q, k, v, do = make_inputs(w)
    o, lse, (dq, dk, dv) = run(w, q, k, v, do)
    assert torch.equal(o, v)
    want = w.scale * np.einsum("bhnd,bhnd->bhn", f64(q), f64(k))
    assert np.abs(lse.double().numpy() - want).max() <= 1e-4
    assert torch.equal(dv, do)
    assert np.abs(f64(dq)).max() <= 1e-2 and np.abs(f64(dk)).max() <= 1e-2


def test_window_ge_n_equals_causal_bitwise():
    """A window that reaches back past position 0 for every query is plain
    causal attention: the same key blocks and masks, so the windowed forward
    and backward give the causal kernels' outputs bit for bit."""
    w = small("wide", 1, 4, 2, 700, 64, 700, 521)
    q, k, v, do = make_inputs(w)
    o, lse, (dq, dk, dv) = run(w, q, k, v, do)
    dev = torch.device("cuda:0")
    qd, kd, vd = (t.to(dev) for t in (q, k, v))
    oc, lc = fa.attention(qd, kd, vd, causal=True, scale=w.scale)
    gc = fa.attention_backward(qd, kd, vd, oc, lc, do.to(dev), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert torch.equal(o, oc.cpu()) and torch.equal(lse, lc.cpu())
    # dK and dV accumulate inside one CTA in a fixed order; dQ partials are
    # added into fp32 by several CTAs in whatever order they finish.
    assert torch.equal(dk, gc[1].cpu()) and torch.equal(dv, gc[2].cpu())
    assert rel_fro(dq, f64(gc[0].cpu())) <= 1e-3


def test_window_rejects_nonpositive():
    q = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    o = torch.empty_like(q)
    lse = torch.empty((1, 1, 128), dtype=torch.float32, device="cuda")
    for bad in (0, -5):
        with pytest.raises(fa.FAError) as e:
            fa.fa_fwd_window(q, q, q, o, lse, bad, 0.125)
        assert e.value.status == fa.FA_ERR_INVALID_ARG


def slice_check(w, q, k, v, do, o, lse, grads, s, e, b, g):
    """Oracle on positions [s, e) of batch b, key/value head g (every query
    head of its group); compares the rows that the slice determines exactly."""
    W, N = w.window, w.N
    G = w.H // w.Hkv
    hs = slice(g * G, (g + 1) * G)
    qs, ks, vs, ds = (f64(t[b:b + 1, hh, s:e]) for t, hh in
                      ((q, hs), (k, slice(g, g + 1)), (v, slice(g, g + 1)), (do, hs)))
    ro, rl = oracle.attn_fwd_window(qs, ks, vs, W, w.scale)
    rq, rk, rv, _ = oracle.attn_bwd_window(qs, ks, vs, ds, W, w.scale)
    r0 = 0 if s == 0 else W - 1                                  # exact query rows
    k1 = (e - s) if e == N else (e - s) - W + 1                  # exact key rows: [r0, k1)
    assert k1 > r0
    go = f64(o[b:b + 1, hs, s:e])
    assert np.abs(go[..., r0:, :] - ro[..., r0:, :]).max() <= O_MAX_ABS
    assert np.abs(lse[b:b + 1, hs, s:e].double().numpy()[..., r0:] - rl[..., r0:]).max() \
        <= LSE_MAX_ABS
    dq, dk, dv = grads
    errs = {"dq": rel_fro(f64(dq[b:b + 1, hs, s:e])[..., r0:, :], rq[..., r0:, :]),
            "dk": rel_fro(f64(dk[b:b + 1, g:g + 1, s:e])[..., r0:k1, :], rk[..., r0:k1, :]),
            "dv": rel_fro(f64(dv[b:b + 1, g:g + 1, s:e])[..., r0:k1, :], rv[..., r0:k1, :])}
    for name, err in errs.items():
        assert err <= GRAD_REL_FRO, f"{name} [{s}, {e}) relative Frobenius error {err:.3e}"


@pytest.mark.slow
def test_window_full_size():
    """The benchmark's windowed workload (B 1, H 32, Hkv 8, N 16384, d 128,
    W 4096), the same launches; the oracle checks three slices: the prefix
    [0, W + 256) and a middle slice [7000, 7000 + 2W + 256) of the first
    key/value group, the suffix [N - W - 256, N) of the last one."""
    w = WORKLOADS["window"]
    q, k, v, do = make_inputs(w)
    o, lse, grads = run(w, q, k, v, do)
    for t in (o,) + grads:
        assert torch.isfinite(t.float()).all()
    W, N = w.window, w.N
    for (b, g), (s, e) in (((0, 0), (0, W + 256)), ((0, 0), (7000, 7000 + 2 * W + 256)),
                           ((w.B - 1, w.Hkv - 1), (N - W - 256, N))):
        slice_check(w, q, k, v, do, o, lse, grads, s, e, b, g)
