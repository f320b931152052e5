"""FP8 (e4m3) forward on the GPU, through the C ABI: S = Q K^T from the bf16
inputs, P and V in e4m3 (the placement tests/test_fp8_error_model.py derives).

- fa_fp8_quantize against the oracle's quantiser of V: every code byte and
  every block scale bit-exact (integer/byte work).
- fa_fwd_fp8 against the fp64 oracle on the unquantised bf16 inputs: O's
  relative RMS error sqrt(mean((o - ref)^2)) / sqrt(mean(ref^2)) <= 5e-2, the
  bar for an FP8 forward; LSE max abs <= 1e-3 (LSE depends on S alone, which
  is computed as in the bf16 forward).
- fa_fwd_fp8 against the fp64 oracle on the unquantised Q, K and the values
  V's codes stand for: what remains is the kernel's own rounding of P to e4m3
  (about 2.7 % RMS per element) and of O to bf16: relative RMS <= 3e-2.
"""
import numpy as np
import pytest
import torch

import exact_attention_online_gb300 as fa
import oracle
from _gpu import LSE_MAX_ABS, f64
from exact_attention_online_gb300.inputs import WORKLOADS, Workload, make_inputs

pytestmark = pytest.mark.gpu

FP8_O_REL_RMS = 5e-2          # against the unquantised inputs
FP8_O_REL_RMS_DEQ_V = 3e-2    # against the unquantised Q, K and the dequantised V


def rel_rms(a, ref):
    return float(np.sqrt(np.mean((a - ref) ** 2)) / np.sqrt(np.mean(ref ** 2)))


def small(name, B, H, Hkv, N, causal, seed, **kw):
    return Workload(name=name, B=B, H=H, Hkv=Hkv, N=N, d=128, causal=causal, seed=seed, **kw)


CASES = [
    small("tiny", 1, 1, 1, 128, False, 301),
    small("causal_ragged", 1, 2, 1, 333, True, 302),
    small("gqa", 1, 4, 2, 384, True, 303),
    small("n1", 1, 2, 2, 1, True, 304),
    small("full_600", 2, 2, 1, 600, False, 305),
    small("outliers", 1, 2, 2, 512, True, 306, outlier_frac=0.001),
    small("k_channels", 1, 2, 1, 300, True, 307, k_outlier_channels=2),
]


def quantize_gpu(v, H):
    B, Hkv, N, d = v.shape
    n = fa.fa_fp8_buffer_size(B, H, Hkv, N, d)
    assert n > 0
    buf = torch.zeros(n, dtype=torch.uint8, device="cuda")
    fa.fa_fp8_quantize(v.cuda(), buf, H)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return buf


def carve(buf, B, Hkv, N, d):
    """Views of the documented buffer layout (fa.h), on the host."""
    Np = (N + 127) // 128 * 128
    nblk = Np // 128
    a = lambda x: (x + 255) // 256 * 256
    h = buf.cpu().numpy()
    off = 0
    out = {}
    for name, count, dt, shape in (("v8t", B * Hkv * Np * d, np.uint8, (B * Hkv, d, Np)),
                                   ("sv", B * Hkv * nblk, np.float32, (B * Hkv, nblk)),
                                   ("svmax", B * Hkv, np.float32, (B * Hkv,))):
        nbytes = count * np.dtype(dt).itemsize
        out[name] = h[off:off + nbytes].view(dt).reshape(shape)
        off += a(nbytes)
    return out


@pytest.mark.parametrize("w", CASES[:3] + CASES[5:], ids=lambda w: w.name)
def test_fp8_quantize_bit_exact(w):
    _, _, v, _ = make_inputs(w)
    got = carve(quantize_gpu(v, w.H), w.B, w.Hkv, w.N, w.d)
    want = oracle.fp8_quantize_v(v.float().numpy())
    for name in ("v8t", "sv", "svmax"):
        g, r = got[name], want[name]
        if g.dtype == np.float32:
            assert np.array_equal(g.view(np.uint32), r.view(np.uint32)), name
        else:
            diff = np.argwhere(g != r)
            assert diff.size == 0, f"{name}: {len(diff)} codes differ, first at {diff[0]}"


def test_fp8_quantize_zero_block_and_saturation():
    """An all-zero block gets scale 1 and zero codes; an element at the block
    amax encodes to +-448 exactly."""
    w = small("zero", 1, 1, 1, 256, False, 308)
    _, _, v, _ = make_inputs(w)
    v[0, 0, :128] = 0
    v[0, 0, 200, 5] = -64.0
    got = carve(quantize_gpu(v, 1), 1, 1, 256, 128)
    assert got["sv"][0, 0] == 1.0 and not got["v8t"][0, :, :128].any()
    assert got["v8t"][0, 5, 200] == 0xFE
    assert got["sv"][0, 1] == np.float32(np.float32(64.0) / np.float32(448.0))


def run_fp8(q, k, v, causal, scale):
    B, H, N, d = q.shape
    buf = quantize_gpu(v, H)
    o = torch.empty((B, H, N, d), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((B, H, N), dtype=torch.float32, device="cuda")
    fa.fa_fwd_fp8(q.cuda(), k.cuda(), buf, o, lse, causal, scale)
    torch.cuda.synchronize()
    assert fa.fa_device_status() == 0
    return buf, o.cpu(), lse.cpu()


def check_heads(w, q, k, v, buf, o, lse, heads):
    d = w.d
    G = w.H // w.Hkv
    v_deq = oracle.fp8_dequantize_v(carve(buf, w.B, w.Hkv, w.N, d), w.B, w.Hkv, w.N, d)
    worst = {"rel_rms": 0.0, "rel_rms_deq_v": 0.0, "lse": 0.0}
    for (b, h) in heads:
        g = h // G
        qh, kh = f64(q[b:b + 1, h:h + 1]), f64(k[b:b + 1, g:g + 1])
        ref_o, ref_l = oracle.attn_fwd(qh, kh, f64(v[b:b + 1, g:g + 1]), w.causal, w.scale)
        dq_o, _ = oracle.attn_fwd(qh, kh, v_deq[b:b + 1, g:g + 1], w.causal, w.scale)
        go = f64(o[b, h])
        assert np.isfinite(go).all()
        worst["rel_rms"] = max(worst["rel_rms"], rel_rms(go, ref_o[0, 0]))
        worst["rel_rms_deq_v"] = max(worst["rel_rms_deq_v"], rel_rms(go, dq_o[0, 0]))
        worst["lse"] = max(worst["lse"],
                           float(np.abs(lse[b, h].double().numpy() - ref_l[0, 0]).max()))
    assert worst["rel_rms"] <= FP8_O_REL_RMS, worst
    assert worst["rel_rms_deq_v"] <= FP8_O_REL_RMS_DEQ_V, worst
    assert worst["lse"] <= LSE_MAX_ABS, worst
    return worst


@pytest.mark.parametrize("w", CASES, ids=lambda w: w.name)
def test_fp8_fwd_small(w):
    q, k, v, _ = make_inputs(w)
    buf, o, lse = run_fp8(q, k, v, w.causal, w.scale)
    heads = [(b, h) for b in range(w.B) for h in range(w.H)]
    check_heads(w, q, k, v, buf, o, lse, heads)


def test_fp8_entry_points_reject():
    v = torch.zeros((1, 1, 128, 64), dtype=torch.bfloat16, device="cuda")
    assert fa.fa_fp8_buffer_size(1, 1, 1, 128, 64) == 0
    buf = torch.zeros(1 << 20, dtype=torch.uint8, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fp8_quantize(v, buf, 1)
    assert e.value.status == fa.FA_ERR_UNSUPPORTED
    v = torch.zeros((1, 1, 128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fa.FAError) as e:
        fa.fa_fp8_quantize(v, buf[:1024], 1)
    assert e.value.status == fa.FA_ERR_WORKSPACE


FULL = ["long16k", "long32k"]


@pytest.mark.slow
@pytest.mark.parametrize("name", FULL)
def test_fp8_fwd_full_size(name):
    """The long-sequence stress workloads (0.1 % outliers of magnitude 30), the
    same launches as the benchmark's FP8 line; the oracle checks the first and
    the last head in full."""
    w = WORKLOADS[name]
    q, k, v, _ = make_inputs(w)
    buf, o, lse = run_fp8(q, k, v, w.causal, w.scale)
    assert torch.isfinite(o.float()).all()
    check_heads(w, q, k, v, buf, o, lse, [(0, 0), (w.B - 1, w.H - 1)])
