"""fa_bwd_static_scratch: the backward for callers that cannot allocate device
memory (a runtime that owns all device memory in a fixed pool, a loop that
must not risk the synchronisation cudaMalloc can cause, a plugin without the
host's allocator).  Its scratch is a fixed array inside the library instead of
a caller workspace; its results must equal fa_bwd's.

This file is collected last so that a run stopping at the first failure has
already run every other test.  It builds and loads the library itself, so it
also passes when run alone in a fresh process.
"""
import ctypes

import pytest
import torch

import exact_attention_online_gb300 as fa
from exact_attention_online_gb300.inputs import Workload, make_inputs

GRAD_REL_FRO = 2e-2          # the gradient tolerance used by the parity tests
SCRATCH_BYTES = 32 << 20     # the fixed array's size, as documented in include/fa.h


def _lib():
    fa.build()
    return fa.lib()


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr())


def _call(L, w, q, k, v, o, do, lse, dq, dk, dv):
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    return L.fa_bwd_static_scratch(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(do), _ptr(lse),
                                   _ptr(dq), _ptr(dk), _ptr(dv), w.B, w.H, w.Hkv, w.N, w.d,
                                   int(w.causal), float(w.scale), stream)


def _rel(a, b):
    a, b = a.double(), b.double()
    return float((a - b).norm() / max(float(b.norm()), 1e-30))


def test_sizes_beyond_the_array_are_rejected():
    """A problem whose backward workspace exceeds the fixed array is refused
    with FA_ERR_WORKSPACE before anything is launched (no GPU needed)."""
    L = _lib()
    B, H, Hkv, N, d = 2, 16, 16, 8192, 128
    assert L.fa_bwd_workspace_size(B, H, Hkv, N, d) > SCRATCH_BYTES
    A = ctypes.c_void_p(1 << 20)
    before = fa.fa_kernel_launches()
    st = L.fa_bwd_static_scratch(A, A, A, A, A, A, A, A, A, B, H, Hkv, N, d, 1, 0.088, None)
    assert st == fa.FA_ERR_WORKSPACE
    assert fa.fa_kernel_launches() == before


@pytest.mark.gpu
def test_static_scratch_matches_fa_bwd_on_two_calls_in_a_row():
    """Two calls in a row (different shapes, so the second sees what the first
    left in the shared array) give fa_bwd's dQ, dK, dV within the gradient
    tolerance of the parity tests.  Each call launches exactly its three
    kernels and leaves device memory as it was: neither PyTorch's reserve nor
    the driver's free bytes move (measured after a first round of both shapes,
    so that the lazy loading of the kernels' code is not counted)."""
    L = _lib()
    dev = torch.device("cuda:0")
    cases = [
        Workload(name="noalloc_a", B=1, H=4, Hkv=2, N=333, d=128, causal=True, seed=71),
        Workload(name="noalloc_b", B=2, H=2, Hkv=2, N=512, d=64, causal=False, seed=72),
    ]
    prepared = []
    for w in cases:
        assert L.fa_bwd_workspace_size(w.B, w.H, w.Hkv, w.N, w.d) <= SCRATCH_BYTES
        q, k, v, do = (t.to(dev) for t in make_inputs(w))
        o, lse = fa.attention(q, k, v, causal=w.causal, scale=w.scale)
        ref = fa.attention_backward(q, k, v, o, lse, do, causal=w.causal, scale=w.scale)
        out = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
        prepared.append((w, q, k, v, o, do, lse, ref, out))
    torch.cuda.synchronize()
    for w, q, k, v, o, do, lse, ref, out in prepared:          # warm-up round
        assert _call(L, w, q, k, v, o, do, lse, *out) == fa.FA_OK
    torch.cuda.synchronize()
    assert fa.fa_device_status() == fa.FA_OK
    for w, q, k, v, o, do, lse, ref, out in prepared:          # checked round
        for t in out:
            t.fill_(float("nan"))
        torch.cuda.synchronize()
        reserved, (free, _) = torch.cuda.memory_reserved(dev), torch.cuda.mem_get_info(dev)
        launches = fa.fa_kernel_launches()
        assert _call(L, w, q, k, v, o, do, lse, *out) == fa.FA_OK
        torch.cuda.synchronize()
        assert fa.fa_kernel_launches() - launches == 3, w.name
        assert torch.cuda.memory_reserved(dev) == reserved, w.name
        assert torch.cuda.mem_get_info(dev)[0] == free, w.name
        assert fa.fa_device_status() == fa.FA_OK
        for name, a, b in zip(("dq", "dk", "dv"), out, ref):
            assert torch.isfinite(a.float()).all(), name
            assert _rel(a, b) <= GRAD_REL_FRO, (w.name, name, _rel(a, b))
