"""The C ABI without a GPU: the library loads, exports every symbol that
include/fa.h declares, and rejects bad arguments with the documented status
before touching the device (no compute calls here)."""
import ctypes
import os
import re

import pytest

import exact_attention_online_gb300 as fa
from exact_attention_online_gb300 import _native

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    fa.build()
    return fa.lib()


def declared_symbols():
    with open(os.path.join(ROOT, "include", "fa.h")) as f:
        text = f.read()
    return re.findall(r"^FA_API\s+[\w\s\*]*?\b(fa_\w+)\s*\(", text, flags=re.M)


def test_header_declares_the_exports():
    assert sorted(declared_symbols()) == sorted(_native.EXPORTS)


def test_library_exports_every_declared_symbol(L):
    for name in declared_symbols():
        assert hasattr(L, name), name


def test_status_strings(L):
    names = {0: "FA_OK", -1: "FA_ERR_INVALID_ARG", -2: "FA_ERR_UNSUPPORTED",
             -3: "FA_ERR_ALIGNMENT", -4: "FA_ERR_WORKSPACE", -5: "FA_ERR_CUDA",
             -6: "FA_ERR_TIMEOUT"}
    for code, name in names.items():
        assert fa.fa_status_string(code) == name
    assert fa.fa_status_string(-99) == "FA_ERR_UNKNOWN"


A = 1 << 20          # a 16-byte aligned fake address (never dereferenced)
MIS = A + 8          # misaligned


def fwd(L, q=A, k=A, v=A, o=A, lse=A, B=1, H=2, Hkv=1, N=128, d=64, causal=1, scale=0.125):
    return L.fa_fwd(q, k, v, o, lse, B, H, Hkv, N, d, causal, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=96), fa.FA_ERR_UNSUPPORTED),
    (dict(d=256), fa.FA_ERR_UNSUPPORTED),
    (dict(H=3, Hkv=2), fa.FA_ERR_INVALID_ARG),
    (dict(N=0), fa.FA_ERR_INVALID_ARG),
    (dict(N=-5), fa.FA_ERR_INVALID_ARG),
    (dict(B=0), fa.FA_ERR_INVALID_ARG),
    (dict(Hkv=0), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("nan")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=float("inf")), fa.FA_ERR_INVALID_ARG),
    (dict(scale=0.0), fa.FA_ERR_INVALID_ARG),
    (dict(q=0), fa.FA_ERR_INVALID_ARG),
    (dict(lse=0), fa.FA_ERR_INVALID_ARG),
    (dict(v=MIS), fa.FA_ERR_ALIGNMENT),
    (dict(o=MIS), fa.FA_ERR_ALIGNMENT),
    (dict(B=4096, H=64, Hkv=64, N=4096, d=128), fa.FA_ERR_UNSUPPORTED),
])
def test_fwd_rejects_before_launch(L, kw, code):
    before = fa.fa_kernel_launches()
    assert fwd(L, **kw) == code
    assert fa.fa_kernel_launches() == before


def test_workspace_size(L):
    # -LSE and -D extension tables: bf16 [B][H][Np][16] each, accumulator fp32
    # [B][H][Np][d], the dK/dV kernel's work counter (int32, 256-byte region);
    # Np = N rounded to 128.
    B, H, Hkv, N, d = 2, 4, 2, 200, 64
    Np = 256
    rows = B * H * Np
    r256 = lambda x: (x + 255) // 256 * 256
    assert fa.fa_bwd_workspace_size(B, H, Hkv, N, d) == \
        2 * r256(rows * 32) + r256(rows * d * 4) + 256
    assert fa.fa_bwd_workspace_size(B, H, 3, N, d) == 0
    assert fa.fa_bwd_workspace_size(B, H, Hkv, N, 80) == 0


def bwd(L, ws=A, ws_bytes=None, dq=A, B=1, H=2, Hkv=1, N=128, d=64, scale=0.125):
    if ws_bytes is None:
        ws_bytes = L.fa_bwd_workspace_size(B, H, Hkv, N, d)
    return L.fa_bwd(A, A, A, A, A, A, dq, A, A, ws, ws_bytes, B, H, Hkv, N, d, 1, scale, None)


@pytest.mark.parametrize("kw,code", [
    (dict(ws=0), fa.FA_ERR_WORKSPACE),
    (dict(ws_bytes=16), fa.FA_ERR_WORKSPACE),
    (dict(ws=MIS), fa.FA_ERR_ALIGNMENT),
    (dict(dq=0), fa.FA_ERR_INVALID_ARG),
    (dict(dq=MIS), fa.FA_ERR_ALIGNMENT),
    (dict(d=32), fa.FA_ERR_UNSUPPORTED),
    (dict(H=2, Hkv=4), fa.FA_ERR_INVALID_ARG),
    (dict(scale=-1.0), fa.FA_ERR_INVALID_ARG),
])
def test_bwd_rejects_before_launch(L, kw, code):
    before = fa.fa_kernel_launches()
    assert bwd(L, **kw) == code
    assert fa.fa_kernel_launches() == before


def test_stage_entry_points_validate(L):
    ws = L.fa_bwd_workspace_size(1, 2, 1, 128, 64)
    assert L.fa_bwd_preprocess(A, A, A, A, 8, 1, 2, 1, 128, 64, None) == fa.FA_ERR_WORKSPACE
    assert L.fa_bwd_preprocess(0, A, A, A, ws, 1, 2, 1, 128, 64, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_bwd_dkdv(A, A, A, A, A, MIS, A, ws, 1, 2, 1, 128, 64, 0, 0.1, None) == \
        fa.FA_ERR_ALIGNMENT
    assert L.fa_bwd_dq_convert(A, ws, A, 1, 2, 1, 128, 64, float("nan"), None) == \
        fa.FA_ERR_INVALID_ARG


def test_training_entry_points_validate(L):
    """The training pair and its stages reject bad arguments before any launch."""
    before = fa.fa_kernel_launches()
    ws = L.fa_bwd_workspace_size(1, 2, 1, 128, 64)
    args = (1, 2, 1, 128, 64, 1, 0.125, None)
    assert L.fa_fwd_train(A, A, A, A, A, A, 8, *args) == fa.FA_ERR_WORKSPACE
    assert L.fa_fwd_train(A, A, A, A, 0, A, ws, *args) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_train_precise(A, A, A, MIS, A, A, ws, *args) == fa.FA_ERR_ALIGNMENT
    assert L.fa_fwd_train(A, A, A, A, A, A, ws, 1, 2, 1, 128, 80, 1, 0.125, None) == \
        fa.FA_ERR_UNSUPPORTED
    assert L.fa_bwd_train(A, A, A, A, A, A, A, A, 0, ws, *args) == fa.FA_ERR_WORKSPACE
    assert L.fa_bwd_train(A, A, A, A, A, 0, A, A, A, ws, *args) == fa.FA_ERR_INVALID_ARG
    assert L.fa_bwd_train_precise(A, A, A, A, A, A, A, A, A, ws, 1, 2, 1, 128, 64, 1,
                                  float("inf"), None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_bwd_preprocess_train(A, A, A, 8, 1, 2, 1, 128, 64, None) == fa.FA_ERR_WORKSPACE
    assert L.fa_bwd_preprocess_train_precise(0, A, A, ws, 1, 2, 1, 128, 64, None) == \
        fa.FA_ERR_INVALID_ARG
    assert fa.fa_kernel_launches() == before


def test_python_binding_rejects_cpu_tensors():
    import torch
    q = torch.zeros(1, 1, 8, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        fa.fa_fwd(q, q, q, q, torch.zeros(1, 1, 8), False, 0.125, stream=0)


def test_window_entry_points_validate(L):
    """window < 1 and the shape rules of fa_fwd / fa_bwd, before any launch."""
    before = fa.fa_kernel_launches()
    for w in (0, -3):
        assert L.fa_fwd_window(A, A, A, A, A, 1, 2, 1, 128, 64, w, 0.125, None) == \
            fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_window(A, A, A, A, A, 1, 2, 1, 128, 96, 16, 0.125, None) == \
        fa.FA_ERR_UNSUPPORTED
    assert L.fa_fwd_window(A, A, A, MIS, A, 1, 2, 1, 128, 64, 16, 0.125, None) == \
        fa.FA_ERR_ALIGNMENT
    ws = L.fa_bwd_workspace_size(1, 2, 1, 128, 64)
    assert L.fa_bwd_window(A, A, A, A, A, A, A, A, A, A, ws, 1, 2, 1, 128, 64, 0, 0.125,
                           None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_bwd_window(A, A, A, A, A, A, A, A, A, A, 16, 1, 2, 1, 128, 64, 8, 0.125,
                           None) == fa.FA_ERR_WORKSPACE
    assert L.fa_bwd_dkdv_window(A, A, A, A, A, A, A, ws, 1, 2, 1, 128, 64, 0, 0.125,
                                None) == fa.FA_ERR_INVALID_ARG
    # the training pair of the window: window < 1, a short workspace
    for w in (0, -1):
        assert L.fa_fwd_window_train(A, A, A, A, A, A, ws, 1, 2, 1, 128, 64, w, 0.125,
                                     None) == fa.FA_ERR_INVALID_ARG
        assert L.fa_bwd_window_train(A, A, A, A, A, A, A, A, A, ws, 1, 2, 1, 128, 64, w, 0.125,
                                     None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_window_train(A, A, A, A, A, A, 16, 1, 2, 1, 128, 64, 8, 0.125,
                                 None) == fa.FA_ERR_WORKSPACE
    assert L.fa_bwd_window_train(A, A, A, A, A, A, A, A, A, 16, 1, 2, 1, 128, 64, 8, 0.125,
                                 None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_kernel_launches() == before


def test_varlen_entry_points_validate(L):
    """Packed batches: a null offsets array, total < 1, a misaligned offsets
    pointer and the shape rules, before any launch."""
    before = fa.fa_kernel_launches()
    f = lambda cu, B, ms, total, d=64: L.fa_fwd_varlen(A, A, A, A, A, cu, B, ms, total, 2, 1, d,
                                                       1, 0.125, None)
    assert f(None, 2, 128, 200) == fa.FA_ERR_INVALID_ARG
    assert f(A, 2, 128, 0) == fa.FA_ERR_INVALID_ARG
    assert f(A + 2, 2, 128, 200) == fa.FA_ERR_ALIGNMENT
    assert f(A, 2, 128, 200, d=96) == fa.FA_ERR_UNSUPPORTED
    assert f(A, 0, 128, 200) == fa.FA_ERR_INVALID_ARG
    ws = L.fa_bwd_varlen_workspace_size(2, 2, 1, 128, 64)
    assert ws == L.fa_bwd_workspace_size(2, 2, 1, 128, 64)
    assert L.fa_bwd_varlen(A, A, A, A, A, A, A, A, A, A, 16, A, 2, 128, 200, 2, 1, 64, 1, 0.125,
                           None) == fa.FA_ERR_WORKSPACE
    assert fa.fa_kernel_launches() == before


def test_decode_entry_points_validate(L):
    """Decoding: more query rows than keys, more than 16 rows per kv group, an
    unsupported head dim and a short workspace, before any launch."""
    before = fa.fa_kernel_launches()
    assert L.fa_fwd_decode_workspace_size(1, 4, 1, 8, 4, 64) == 0        # Nq > Nk
    assert L.fa_fwd_decode_workspace_size(1, 32, 1, 1, 1024, 64) == 0    # G * Nq = 32 > 16
    assert L.fa_fwd_decode_workspace_size(1, 4, 1, 1, 1024, 96) == 0     # d = 96
    ws = L.fa_fwd_decode_workspace_size(2, 8, 2, 1, 4096, 128)
    assert ws > 0
    d = lambda wsb, Nq=1, Nk=4096: L.fa_fwd_decode(A, A, A, A, A, A, wsb, 2, 8, 2, Nq, Nk, 128, 1,
                                                   0.088, None)
    assert d(ws, Nq=8, Nk=4) != fa.FA_OK
    assert d(16) == fa.FA_ERR_WORKSPACE
    assert fa.fa_kernel_launches() == before


def test_fp8_entry_points_validate(L):
    """FP8: d = 64 is not supported and a short buffer is rejected."""
    before = fa.fa_kernel_launches()
    assert L.fa_fp8_buffer_size(1, 2, 1, 256, 64) == 0
    n = L.fa_fp8_buffer_size(1, 2, 1, 256, 128)
    assert n > 0
    assert L.fa_fp8_quantize(A, A, 16, 1, 2, 1, 256, 128, None) == fa.FA_ERR_WORKSPACE
    assert L.fa_fp8_quantize(0, A, n, 1, 2, 1, 256, 128, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_fp8(A, A, A, 16, A, A, 1, 2, 1, 256, 128, 1, 0.088, None) == \
        fa.FA_ERR_WORKSPACE
    assert L.fa_fwd_fp8(A, 0, A, n, A, A, 1, 2, 1, 256, 128, 1, 0.088, None) == \
        fa.FA_ERR_INVALID_ARG
    assert L.fa_fwd_fp8(A, A, MIS, n, A, A, 1, 2, 1, 256, 128, 1, 0.088, None) == \
        fa.FA_ERR_ALIGNMENT
    # the buffer holds V only: its size depends on B, Hkv, N, not on H
    assert L.fa_fp8_buffer_size(1, 8, 1, 256, 128) == n
    assert fa.fa_kernel_launches() == before


class FakeCuda:
    """Stands in for a contiguous CUDA tensor of a given shape and dtype: the
    binding reads only these attributes before it calls the library, and the
    library rejects its null pointer before any launch."""

    def __init__(self, shape, dtype, index=0):
        import torch
        self.shape, self.dtype, self.is_cuda = torch.Size(shape), dtype, True
        self.device = torch.device("cuda", index)
        self._esize = torch.empty(0, dtype=dtype).element_size()

    def dim(self):
        return len(self.shape)

    def numel(self):
        n = 1
        for x in self.shape:
            n *= x
        return n

    def element_size(self):
        return self._esize

    def is_contiguous(self):
        return True

    def data_ptr(self):
        return 0


def test_python_binding_checks_every_tensor_shape():
    """The C entry points see only pointers, so the binding checks the shape of
    every tensor against the one q and k imply before anything reaches the
    library."""
    import torch
    bf, f32 = torch.bfloat16, torch.float32
    T = FakeCuda
    q, k = T((1, 4, 8, 64), bf), T((1, 2, 8, 64), bf)
    lse, ws = T((1, 4, 8), f32), T((16,), torch.uint8)
    short_k, short_lse = T((1, 2, 7, 64), bf), T((1, 4, 7), f32)
    cases = [
        ("v", lambda: fa.fa_fwd(q, k, short_k, q, lse, True, 0.125, stream=0)),
        ("o", lambda: fa.fa_fwd(q, k, k, k, lse, True, 0.125, stream=0)),
        ("lse", lambda: fa.fa_fwd(q, k, k, q, short_lse, True, 0.125, stream=0)),
        ("o", lambda: fa.fa_fwd_precise(q, k, k, T((1, 4, 8, 32), f32), lse, True, 0.125,
                                        stream=0)),
        ("lse", lambda: fa.fa_fwd_window(q, k, k, q, short_lse, 4, 0.125, stream=0)),
        ("dout", lambda: fa.fa_bwd(q, k, k, q, k, lse, q, k, k, ws, True, 0.125, stream=0)),
        ("dq", lambda: fa.fa_bwd(q, k, k, q, q, lse, k, k, k, ws, True, 0.125, stream=0)),
        ("dk", lambda: fa.fa_bwd_window(q, k, k, q, q, lse, q, q, k, ws, 4, 0.125, stream=0)),
        ("dv", lambda: fa.fa_bwd_dkdv(q, k, k, q, k, short_k, ws, True, 0.125, stream=0)),
        ("dout", lambda: fa.fa_bwd_preprocess(q, k, lse, ws, 2, stream=0)),
        ("lse", lambda: fa.fa_fwd_fp8(q, k, ws, q, short_lse, True, 0.125, stream=0)),
        ("o", lambda: fa.fa_fwd_fp8(q, k, ws, k, lse, True, 0.125, stream=0)),
        ("o", lambda: fa.fa_fwd_decode(q, k, k, T((1, 4, 1, 64), bf), lse, ws, True, 0.125,
                                       stream=0)),
    ]
    for name, call in cases:
        with pytest.raises(ValueError, match=rf"^{name} has shape"):
            call()
    # the same tensors with the right shapes pass the binding and reach the
    # library, which rejects the null pointers before any launch
    with pytest.raises(fa.FAError) as e:
        fa.fa_fwd(q, k, k, q, lse, True, 0.125, stream=0)
    assert e.value.status == fa.FA_ERR_INVALID_ARG
    # packed layout: [H, total, d] and [H, total]
    pq, pk, cu = T((4, 10, 64), bf), T((2, 10, 64), bf), T((3,), torch.int32)
    with pytest.raises(ValueError, match=r"^lse has shape"):
        fa.fa_fwd_varlen(pq, pk, pk, pq, T((4, 9), f32), cu, 6, True, 0.125, stream=0)
    with pytest.raises(ValueError, match=r"^dk has shape"):
        fa.fa_bwd_varlen(pq, pk, pk, pq, pq, T((4, 10), f32), pq, pq, pk, ws, cu, 6, True,
                         0.125, stream=0)
    with pytest.raises(ValueError, match=r"cu_seqlens must be 1-D"):
        fa.fa_fwd_varlen(pq, pk, pk, pq, T((4, 10), f32), T((1, 3), torch.int32), 6, True,
                         0.125, stream=0)


def test_python_binding_accepts_consistent_shapes():
    """Every wrapper, given tensors of the shapes its documentation states, passes
    the binding's checks and reaches the library (which rejects the null
    pointers of the stand-ins before any launch)."""
    import torch
    bf, f32, u8, i32 = torch.bfloat16, torch.float32, torch.uint8, torch.int32
    T = FakeCuda
    B, H, Hkv, N, d = 2, 4, 2, 8, 64
    q, k, lse = T((B, H, N, d), bf), T((B, Hkv, N, d), bf), T((B, H, N), f32)
    o32, ws = T((B, H, N, d), f32), T((1 << 20,), u8)
    pq, pk, plse = T((H, 20, d), bf), T((Hkv, 20, d), bf), T((H, 20), f32)
    cu = T((B + 1,), i32)
    dq, dlse = T((B, H, 1, d), bf), T((B, H, 1), f32)
    calls = [
        lambda: fa.fa_fwd(q, k, k, q, lse, True, 0.125, stream=0),
        lambda: fa.fa_fwd_precise(q, k, k, o32, lse, True, 0.125, stream=0),
        lambda: fa.fa_fwd_window(q, k, k, q, lse, 4, 0.125, stream=0),
        lambda: fa.fa_bwd(q, k, k, q, q, lse, q, k, k, ws, True, 0.125, stream=0),
        lambda: fa.fa_bwd_precise(q, k, k, o32, q, lse, q, k, k, ws, True, 0.125, stream=0),
        lambda: fa.fa_bwd_window(q, k, k, q, q, lse, q, k, k, ws, 4, 0.125, stream=0),
        lambda: fa.fa_bwd_preprocess(q, q, lse, ws, Hkv, stream=0),
        lambda: fa.fa_bwd_preprocess_precise(o32, q, lse, ws, Hkv, stream=0),
        lambda: fa.fa_bwd_dkdv(q, k, k, q, k, k, ws, True, 0.125, stream=0),
        lambda: fa.fa_bwd_dkdv_window(q, k, k, q, k, k, ws, 4, 0.125, stream=0),
        lambda: fa.fa_bwd_dq_convert(ws, q, Hkv, 0.125, stream=0),
        lambda: fa.fa_fwd_varlen(pq, pk, pk, pq, plse, cu, 12, True, 0.125, stream=0),
        lambda: fa.fa_bwd_varlen(pq, pk, pk, pq, pq, plse, pq, pk, pk, ws, cu, 12, True, 0.125,
                                 stream=0),
        lambda: fa.fa_fp8_quantize(T((B, Hkv, N, 128), bf), ws, H, stream=0),
        lambda: fa.fa_fwd_fp8(T((B, H, N, 128), bf), T((B, Hkv, N, 128), bf), ws,
                              T((B, H, N, 128), bf), lse, True, 0.125, stream=0),
        lambda: fa.fa_fwd_decode(dq, k, k, dq, dlse, ws, True, 0.125, stream=0),
    ]
    for i, call in enumerate(calls):
        with pytest.raises(fa.FAError) as e:
            call()
        assert e.value.status == fa.FA_ERR_INVALID_ARG, i


def test_python_binding_rejects_tensors_of_another_device():
    """Every pointer must be memory of the current device: an operand (or the
    workspace, or the FP8 buffer) on another GPU is rejected before any
    library call, so no kernel or tensor map is built over another GPU's
    memory."""
    import torch
    bf, f32, u8 = torch.bfloat16, torch.float32, torch.uint8
    T = FakeCuda
    B, H, Hkv, N, d = 1, 4, 2, 8, 64
    q, k, lse, ws = T((B, H, N, d), bf), T((B, Hkv, N, d), bf), T((B, H, N), f32), T((64,), u8)
    other = lambda shape, dt: T(shape, dt, index=1)
    before = fa.fa_kernel_launches()
    cases = [
        ("q", lambda: fa.fa_fwd(other(q.shape, bf), k, k, q, lse, True, 0.125, stream=0)),
        ("v", lambda: fa.fa_fwd(q, k, other(k.shape, bf), q, lse, True, 0.125, stream=0)),
        ("lse", lambda: fa.fa_fwd(q, k, k, q, other(lse.shape, f32), True, 0.125, stream=0)),
        ("workspace", lambda: fa.fa_bwd(q, k, k, q, q, lse, q, k, k, other((64,), u8), True,
                                        0.125, stream=0)),
        ("dk", lambda: fa.fa_bwd_dkdv(q, k, k, q, other(k.shape, bf), k, ws, True, 0.125,
                                      stream=0)),
        ("workspace", lambda: fa.fa_fwd_fp8(T((B, H, N, 128), bf), T((B, Hkv, N, 128), bf),
                                            other((64,), u8), T((B, H, N, 128), bf), lse,
                                            True, 0.125, stream=0)),
    ]
    for name, call in cases:
        with pytest.raises(ValueError, match=rf"^{name} is on cuda:1 but the current device"):
            call()
    assert fa.fa_kernel_launches() == before


def test_ex2_rate_validates(L):
    """The exponential-unit microbenchmark rejects a null output and block or
    round counts out of range before any launch."""
    before = fa.fa_kernel_launches()
    assert L.fa_ex2_rate(None, 8, 16, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_ex2_rate(A, 0, 16, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_ex2_rate(A, 8, 0, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_ex2_rate(A, (1 << 20) + 1, 16, None) == fa.FA_ERR_INVALID_ARG
    assert L.fa_ex2_rate(A, 8, (1 << 24) + 1, None) == fa.FA_ERR_INVALID_ARG
    assert fa.fa_kernel_launches() == before
