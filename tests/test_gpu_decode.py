"""Split-KV decoding forward on the GPU, through the C ABI, against the fp64
oracle for fewer queries than keys (the queries are the last positions,
bottom-right causal): O max abs <= 1e-2, LSE max abs <= 1e-3 on the same
seeded bf16 inputs."""
import numpy as np
import pytest
import torch

import exact_attention_online_gb300 as fa
import oracle
from _gpu import LSE_MAX_ABS, O_MAX_ABS, f64
from exact_attention_online_gb300.inputs import (DECODE_WORKLOADS, DecodeWorkload,
                                                 make_decode_inputs)

pytestmark = pytest.mark.gpu


def dw(name, B, H, Hkv, Nq, Nk, d, causal, seed):
    return DecodeWorkload(name, B=B, H=H, Hkv=Hkv, Nq=Nq, Nk=Nk, d=d, causal=causal, seed=seed)


CASES = [
    dw("one_key", 1, 2, 1, 1, 1, 128, True, 401),
    dw("mha_d64", 2, 4, 4, 1, 300, 64, True, 402),
    dw("gqa4_d128", 1, 8, 2, 1, 1000, 128, True, 403),
    dw("nq3_causal", 1, 4, 2, 3, 777, 128, True, 404),
    dw("nq3_full", 1, 4, 2, 3, 777, 128, False, 405),
    dw("nq_eq_nk", 1, 2, 1, 5, 5, 64, True, 406),
    dw("rows16", 1, 8, 2, 4, 5000, 128, True, 407),
    dw("mqa_d64", 2, 16, 1, 1, 2049, 64, True, 408),
    dw("tile_edge", 1, 2, 2, 2, 256, 128, True, 409),
    dw("many_splits", 1, 2, 1, 1, 70000, 64, True, 410),
]


def run(w, q, k, v):
    qd, kd, vd = q.cuda(), k.cuda(), v.cuda()
    o, lse = fa.attention_decode(qd, kd, vd, causal=w.causal, scale=w.scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return o.cpu(), lse.cpu()


def check(w, q, k, v, o, lse, heads=None):
    if heads is None:
        ro, rl = oracle.attn_fwd_decode(f64(q), f64(k), f64(v), w.causal, w.scale)
        go, gl = f64(o), lse.double().numpy()
    else:
        G = w.H // w.Hkv
        ro, rl, go, gl = [], [], [], []
        for (b, h) in heads:
            g = h // G
            a, c = oracle.attn_fwd_decode(f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, g:g + 1]),
                                          f64(v[b:b + 1, g:g + 1]), w.causal, w.scale)
            ro.append(a[0, 0]); rl.append(c[0, 0])
            go.append(f64(o[b, h])); gl.append(lse[b, h].double().numpy())
        ro, rl, go, gl = map(np.array, (ro, rl, go, gl))
    assert np.isfinite(go).all() and np.isfinite(gl).all()
    eo, el = np.abs(go - ro).max(), np.abs(gl - rl).max()
    assert eo <= O_MAX_ABS and el <= LSE_MAX_ABS, (eo, el)


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_decode_small(w):
    q, k, v = make_decode_inputs(w)
    o, lse = run(w, q, k, v)
    check(w, q, k, v, o, lse)


def test_decode_matches_square_forward_last_rows():
    """Nq == Nk: the decode path and fa_fwd give the same rows (within the
    parity bound of each against the oracle)."""
    w = dw("square", 1, 4, 2, 8, 8, 128, True, 411)
    q, k, v = make_decode_inputs(w)
    o, lse = run(w, q, k, v)
    o2, lse2 = fa.attention(q.cuda(), k.cuda(), v.cuda(), causal=True, scale=w.scale)
    torch.cuda.synchronize()
    assert (o.float() - o2.cpu().float()).abs().max() <= 2 * O_MAX_ABS
    assert (lse - lse2.cpu()).abs().max() <= 2 * LSE_MAX_ABS


def test_decode_rejects():
    q = torch.zeros((1, 8, 4, 128), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((1, 1, 64, 128), dtype=torch.bfloat16, device="cuda")
    assert fa.fa_fwd_decode_workspace_size(1, 8, 1, 4, 64, 128) == 0     # G * Nq = 32 > 16
    assert fa.fa_fwd_decode_workspace_size(1, 8, 1, 4, 3, 128) == 0      # Nk < Nq
    assert fa.fa_fwd_decode_workspace_size(1, 8, 1, 1, 64, 96) == 0      # d
    o = torch.empty_like(q)
    lse = torch.empty((1, 8, 4), dtype=torch.float32, device="cuda")
    work = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    before = fa.fa_kernel_launches()
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_decode(q, k, k, o, lse, work, True, 0.1)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    q1 = q[:, :, :1].contiguous()
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd_decode(q1, k, k, o[:, :, :1].contiguous(), lse[:, :, :1].contiguous(),
                         work[:16], True, 0.1)
    assert e.value.status == fa.FA_ERR_WORKSPACE
    assert fa.fa_kernel_launches() == before


@pytest.mark.slow
@pytest.mark.parametrize("name", sorted(DECODE_WORKLOADS))
def test_decode_full_size(name):
    """The benchmark's decoding shapes; the oracle checks the first and the
    last query head in full."""
    w = DECODE_WORKLOADS[name]
    q, k, v = make_decode_inputs(w)
    o, lse = run(w, q, k, v)
    check(w, q, k, v, o, lse, heads=[(0, 0), (w.B - 1, w.H - 1)])
