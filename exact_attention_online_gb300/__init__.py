"""GB300-native exact attention: online-softmax forward and recomputation
backward, as hand-written sm_103a kernels behind the C ABI of include/fa.h.

This module is the thin Python binding: each function has the name of the C
entry point it calls and does argument marshalling only (tensor -> pointer,
shape -> ints, current CUDA stream).  Every step of the computation runs in
libfa.so; there is no other code path.  A nonzero fa_status raises FAError.

Layouts (as in include/fa.h): q, o, dout, dq bf16 [B, H, N, d]; k, v, dk, dv
bf16 [B, Hkv, N, d]; lse fp32 [B, H, N]; all contiguous CUDA tensors.
"""
from __future__ import annotations

import ctypes

from ._native import EXPORTS, LIB_PATH, build, lib

FA_OK = 0
FA_ERR_INVALID_ARG = -1
FA_ERR_UNSUPPORTED = -2
FA_ERR_ALIGNMENT = -3
FA_ERR_WORKSPACE = -4
FA_ERR_CUDA = -5
FA_ERR_TIMEOUT = -6

__all__ = ["build", "lib", "LIB_PATH", "EXPORTS", "FAError", "fa_fwd", "fa_fwd_precise", "fa_bwd",
           "fa_bwd_workspace_size", "fa_bwd_precise", "fa_bwd_preprocess",
           "fa_bwd_preprocess_precise", "fa_bwd_dkdv", "fa_bwd_dq_convert",
           "fa_device_status", "fa_device_status_detail", "fa_status_string",
           "fa_kernel_launches", "fa_watchdog_selftest", "attention", "attention_backward",
           "fa_fwd_window", "fa_bwd_window", "fa_bwd_dkdv_window", "attention_window",
           "attention_window_backward", "fa_fwd_varlen", "fa_bwd_varlen",
           "fa_bwd_varlen_workspace_size", "attention_varlen", "attention_varlen_backward",
           "fa_fp8_buffer_size", "fa_fp8_quantize", "fa_fwd_fp8", "attention_fp8",
           "fa_fwd_decode_workspace_size", "fa_fwd_decode", "attention_decode",
           "fa_fwd_train", "fa_bwd_train", "fa_bwd_preprocess_train", "fa_exp2_check",
           "fa_ex2_rate",
           "fa_fwd_window_train", "fa_bwd_window_train"]


class FAError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {fa_status_string(status)} ({status})")


def fa_status_string(status: int) -> str:
    return lib().fa_status_string(int(status)).decode()


def _check(status: int, where: str) -> None:
    if status != FA_OK:
        raise FAError(status, where)


def _current_index() -> int:
    """Index of the current CUDA device: every pointer the library receives
    must be memory of this device (its kernels and tensor maps are built
    there)."""
    import torch
    try:
        return torch.cuda.current_device()
    except Exception:   # no CUDA runtime in this process: the library rejects the call
        return 0


def _on_current_device(t, name) -> None:
    dev = getattr(t, "device", None)
    idx = getattr(dev, "index", None)
    cur = _current_index()
    if idx is not None and idx != cur:
        raise ValueError(f"{name} is on cuda:{idx} but the current device is cuda:{cur}")


def _stream(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    if hasattr(stream, "cuda_stream"):
        _on_current_device(stream, "stream")
        return ctypes.c_void_p(stream.cuda_stream)
    return ctypes.c_void_p(int(stream))


def _ptr(t, name, dtype, shape):
    """Device pointer of t after checking its shape (the C entry points see
    only pointers, so a short buffer would be read or written past its end),
    dtype, contiguity and device: a CUDA tensor of the current device, so that
    every operand of a call shares one device."""
    if shape is not None and tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if t.dtype != dtype or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA {str(dtype)[6:]} tensor")
    _on_current_device(t, name)
    return ctypes.c_void_p(t.data_ptr())


def _bf16(t, name, shape=None):
    import torch
    return _ptr(t, name, torch.bfloat16, shape)


def _f32(t, name, shape=None):
    import torch
    return _ptr(t, name, torch.float32, shape)


def _dims(q, k):
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D [B, H(kv), N, d]")
    B, H, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d:
        raise ValueError(f"q {tuple(q.shape)} and k {tuple(k.shape)} disagree")
    return B, H, k.shape[1], N, d


def _shapes(B, H, Hkv, N, d):
    """Shapes of the query-side tensors (q, o, dout, dq), the key-side tensors
    (k, v, dk, dv) and lse: [B, H, N, d], [B, Hkv, N, d], [B, H, N]."""
    return (B, H, N, d), (B, Hkv, N, d), (B, H, N)


def fa_fwd(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    _check(lib().fa_fwd(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _bf16(o, "o", qs),
                        _f32(lse, "lse", ls), B, H, Hkv, N, d, int(bool(causal)), float(scale),
                        _stream(stream)), "fa_fwd")


def fa_fwd_precise(q, k, v, o, lse, causal: bool, scale: float, stream=None) -> None:
    """o: fp32 [B, H, N, d]."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    _check(lib().fa_fwd_precise(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _f32(o, "o", qs),
                                _f32(lse, "lse", ls), B, H, Hkv, N, d, int(bool(causal)),
                                float(scale), _stream(stream)), "fa_fwd_precise")


def fa_fwd_window(q, k, v, o, lse, window: int, scale: float, stream=None) -> None:
    """Causal sliding window: query i attends to keys i - window < j <= i."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    _check(lib().fa_fwd_window(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _bf16(o, "o", qs),
                               _f32(lse, "lse", ls), B, H, Hkv, N, d, int(window), float(scale),
                               _stream(stream)), "fa_fwd_window")


def _i32(t, name, shape=None):
    import torch
    return _ptr(t, name, torch.int32, shape)


def _varlen_dims(q, k, cu_seqlens):
    if q.dim() != 3 or k.dim() != 3:
        raise ValueError("packed q and k must be 3-D [H(kv), total, d]")
    H, total, d = q.shape
    if k.shape[1] != total or k.shape[2] != d:
        raise ValueError(f"q {tuple(q.shape)} and k {tuple(k.shape)} disagree")
    if cu_seqlens.dim() != 1:
        raise ValueError("cu_seqlens must be 1-D [B + 1]")
    return cu_seqlens.numel() - 1, H, k.shape[0], total, d


def fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen: int, causal: bool, scale: float,
                  stream=None) -> None:
    """Packed sequences: q, o [H, total, d], k, v [Hkv, total, d], lse [H, total],
    cu_seqlens int32 [B + 1] on the device."""
    B, H, Hkv, total, d = _varlen_dims(q, k, cu_seqlens)
    qs, ks = (H, total, d), (Hkv, total, d)
    _check(lib().fa_fwd_varlen(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _bf16(o, "o", qs),
                               _f32(lse, "lse", (H, total)), _i32(cu_seqlens, "cu_seqlens"), B,
                               int(max_seqlen), total, H, Hkv, d, int(bool(causal)),
                               float(scale), _stream(stream)), "fa_fwd_varlen")


def fa_bwd_varlen_workspace_size(B: int, H: int, Hkv: int, max_seqlen: int, d: int) -> int:
    return int(lib().fa_bwd_varlen_workspace_size(B, H, Hkv, max_seqlen, d))


def fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens, max_seqlen: int,
                  causal: bool, scale: float, stream=None) -> None:
    B, H, Hkv, total, d = _varlen_dims(q, k, cu_seqlens)
    qs, ks = (H, total, d), (Hkv, total, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_varlen(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _bf16(o, "o", qs),
                               _bf16(dout, "dout", qs), _f32(lse, "lse", (H, total)),
                               _bf16(dq, "dq", qs), _bf16(dk, "dk", ks), _bf16(dv, "dv", ks),
                               wp, wb,
                               _i32(cu_seqlens, "cu_seqlens"), B, int(max_seqlen), total, H, Hkv,
                               d, int(bool(causal)), float(scale), _stream(stream)),
           "fa_bwd_varlen")


def fa_bwd_workspace_size(B: int, H: int, Hkv: int, N: int, d: int) -> int:
    return int(lib().fa_bwd_workspace_size(B, H, Hkv, N, d))


def _ws(workspace):
    import torch
    if not workspace.is_cuda or not workspace.is_contiguous():
        raise ValueError("workspace must be a contiguous CUDA tensor")
    _on_current_device(workspace, "workspace")
    return ctypes.c_void_p(workspace.data_ptr()), workspace.numel() * workspace.element_size()


def fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal: bool, scale: float,
           stream=None) -> None:
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _bf16(o, "o", qs),
                        _bf16(dout, "dout", qs), _f32(lse, "lse", ls), _bf16(dq, "dq", qs),
                        _bf16(dk, "dk", ks), _bf16(dv, "dv", ks), wp, wb, B, H, Hkv, N, d,
                        int(bool(causal)),
                        float(scale), _stream(stream)), "fa_bwd")


def fa_bwd_precise(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal: bool, scale: float,
                   stream=None) -> None:
    """o: the fp32 output of fa_fwd_precise."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_precise(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _f32(o, "o", qs),
                                _bf16(dout, "dout", qs), _f32(lse, "lse", ls), _bf16(dq, "dq", qs),
                                _bf16(dk, "dk", ks), _bf16(dv, "dv", ks), wp, wb, B, H, Hkv, N, d,
                                int(bool(causal)), float(scale), _stream(stream)),
           "fa_bwd_precise")


def fa_fwd_train(q, k, v, o, lse, workspace, causal: bool, scale: float, stream=None) -> None:
    """fa_fwd, plus the backward's workspace prepared for fa_bwd_train; o is
    bf16, or fp32 (the precise forward)."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    import torch
    if o.dtype == torch.float32:
        fn, op, name = lib().fa_fwd_train_precise, _f32(o, "o", qs), "fa_fwd_train_precise"
    else:
        fn, op, name = lib().fa_fwd_train, _bf16(o, "o", qs), "fa_fwd_train"
    _check(fn(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), op, _f32(lse, "lse", ls), wp, wb,
              B, H, Hkv, N, d, int(bool(causal)), float(scale), _stream(stream)), name)


def fa_bwd_train(q, k, v, o, dout, dq, dk, dv, workspace, causal: bool, scale: float,
                 stream=None) -> None:
    """The backward of fa_fwd_train, on the workspace it prepared; o is bf16 or
    fp32 as that forward wrote it."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    import torch
    if o.dtype == torch.float32:
        fn, op, name = lib().fa_bwd_train_precise, _f32(o, "o", qs), "fa_bwd_train_precise"
    else:
        fn, op, name = lib().fa_bwd_train, _bf16(o, "o", qs), "fa_bwd_train"
    _check(fn(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), op, _bf16(dout, "dout", qs),
              _bf16(dq, "dq", qs), _bf16(dk, "dk", ks), _bf16(dv, "dv", ks), wp, wb,
              B, H, Hkv, N, d, int(bool(causal)), float(scale), _stream(stream)), name)


def fa_exp2_check(x, y_fma, y_ex2, stream=None) -> None:
    """2^x on the FMA pipe (y_fma) and from ex2.approx (y_ex2) for fp32 CUDA x."""
    n = x.numel()
    _check(lib().fa_exp2_check(_f32(x, "x"), _f32(y_fma, "y_fma", tuple(x.shape)),
                               _f32(y_ex2, "y_ex2", tuple(x.shape)), n, _stream(stream)),
           "fa_exp2_check")


def fa_ex2_rate(out, blocks: int, iters: int, stream=None) -> None:
    """One launch of the exponential-unit microbenchmark: blocks x 256 threads,
    8 x iters ex2.approx each; out is an fp32 CUDA tensor of blocks x 256."""
    if out.numel() < int(blocks) * 256:
        raise ValueError(f"out must hold blocks x 256 = {int(blocks) * 256} floats")
    _check(lib().fa_ex2_rate(_f32(out, "out"), int(blocks), int(iters), _stream(stream)),
           "fa_ex2_rate")


def fa_bwd_preprocess_train(o, dout, workspace, Hkv: int, stream=None) -> None:
    """Stage 1 of fa_bwd_train: -D into the workspace fa_fwd_train prepared (o
    bf16, or fp32 from the precise forward)."""
    import torch
    if o.dim() != 4:
        raise ValueError("o must be 4-D [B, H, N, d]")
    B, H, N, d = o.shape
    wp, wb = _ws(workspace)
    if o.dtype == torch.float32:
        fn, op, name = (lib().fa_bwd_preprocess_train_precise, _f32(o, "o"),
                        "fa_bwd_preprocess_train_precise")
    else:
        fn, op, name = lib().fa_bwd_preprocess_train, _bf16(o, "o"), "fa_bwd_preprocess_train"
    _check(fn(op, _bf16(dout, "dout", (B, H, N, d)), wp, wb, B, H, int(Hkv), N, d,
              _stream(stream)), name)


def fa_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, workspace, window: int, scale: float,
                  stream=None) -> None:
    """Backward of fa_fwd_window."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_window(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks), _bf16(o, "o", qs),
                               _bf16(dout, "dout", qs), _f32(lse, "lse", ls), _bf16(dq, "dq", qs),
                               _bf16(dk, "dk", ks), _bf16(dv, "dv", ks), wp, wb, B, H, Hkv, N, d,
                               int(window), float(scale), _stream(stream)), "fa_bwd_window")


def fa_fwd_window_train(q, k, v, o, lse, workspace, window: int, scale: float,
                        stream=None) -> None:
    """fa_fwd_window, plus the backward's workspace prepared for
    fa_bwd_window_train."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_fwd_window_train(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks),
                                     _bf16(o, "o", qs), _f32(lse, "lse", ls), wp, wb, B, H, Hkv,
                                     N, d, int(window), float(scale), _stream(stream)),
           "fa_fwd_window_train")


def fa_bwd_window_train(q, k, v, o, dout, dq, dk, dv, workspace, window: int, scale: float,
                        stream=None) -> None:
    """The backward of fa_fwd_window_train, on the workspace it prepared."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_window_train(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks),
                                     _bf16(o, "o", qs), _bf16(dout, "dout", qs),
                                     _bf16(dq, "dq", qs), _bf16(dk, "dk", ks), _bf16(dv, "dv", ks),
                                     wp, wb, B, H, Hkv, N, d, int(window), float(scale),
                                     _stream(stream)), "fa_bwd_window_train")


def _dims_of(t, name):
    if t.dim() != 4:
        raise ValueError(f"{name} must be 4-D [B, H, N, d]")
    return tuple(t.shape)


def fa_bwd_preprocess(o, dout, lse, workspace, Hkv: int, stream=None) -> None:
    B, H, N, d = _dims_of(o, "o")
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_preprocess(_bf16(o, "o"), _bf16(dout, "dout", (B, H, N, d)),
                                   _f32(lse, "lse", (B, H, N)), wp, wb,
                                   B, H, Hkv, N, d, _stream(stream)), "fa_bwd_preprocess")


def fa_bwd_preprocess_precise(o, dout, lse, workspace, Hkv: int, stream=None) -> None:
    """o: the fp32 output of fa_fwd_precise."""
    B, H, N, d = _dims_of(o, "o")
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_preprocess_precise(_f32(o, "o"), _bf16(dout, "dout", (B, H, N, d)),
                                           _f32(lse, "lse", (B, H, N)),
                                           wp, wb, B, H, Hkv, N, d, _stream(stream)),
           "fa_bwd_preprocess_precise")


def fa_bwd_dkdv(q, k, v, dout, dk, dv, workspace, causal: bool, scale: float,
                stream=None) -> None:
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, _ = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_dkdv(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks),
                             _bf16(dout, "dout", qs), _bf16(dk, "dk", ks), _bf16(dv, "dv", ks),
                             wp, wb, B, H, Hkv, N, d,
                             int(bool(causal)), float(scale), _stream(stream)), "fa_bwd_dkdv")


def fa_bwd_dkdv_window(q, k, v, dout, dk, dv, workspace, window: int, scale: float,
                       stream=None) -> None:
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, _ = _shapes(B, H, Hkv, N, d)
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_dkdv_window(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v", ks),
                                    _bf16(dout, "dout", qs), _bf16(dk, "dk", ks),
                                    _bf16(dv, "dv", ks), wp, wb,
                                    B, H, Hkv, N, d, int(window), float(scale), _stream(stream)),
           "fa_bwd_dkdv_window")


def fa_bwd_dq_convert(workspace, dq, Hkv: int, scale: float, stream=None) -> None:
    B, H, N, d = _dims_of(dq, "dq")
    wp, wb = _ws(workspace)
    _check(lib().fa_bwd_dq_convert(wp, wb, _bf16(dq, "dq"), B, H, Hkv, N, d, float(scale),
                                   _stream(stream)), "fa_bwd_dq_convert")


def fa_device_status(stream=None) -> int:
    return int(lib().fa_device_status(_stream(stream)))


def fa_device_status_detail():
    site, block = ctypes.c_int(0), ctypes.c_int(0)
    lib().fa_device_status_detail(ctypes.byref(site), ctypes.byref(block))
    return site.value, block.value


def fa_kernel_launches() -> int:
    return int(lib().fa_kernel_launches())


def fa_watchdog_selftest(timeout_ns: int, stream=None) -> None:
    _check(lib().fa_watchdog_selftest(int(timeout_ns), _stream(stream)), "fa_watchdog_selftest")


# Convenience wrappers that allocate outputs with PyTorch (the library itself
# never allocates).
def fa_fp8_buffer_size(B: int, H: int, Hkv: int, N: int, d: int) -> int:
    return int(lib().fa_fp8_buffer_size(B, H, Hkv, N, d))


def fa_fp8_quantize(v, fp8_buf, H: int, stream=None) -> None:
    """e4m3 codes (transposed) and block scales of v [B, Hkv, N, d] into fp8_buf,
    a contiguous CUDA tensor of at least fa_fp8_buffer_size() bytes; H is the
    number of query heads (checked against Hkv)."""
    B, Hkv, N, d = _dims_of(v, "v")
    bp, bb = _ws(fp8_buf)
    _check(lib().fa_fp8_quantize(_bf16(v, "v"), bp, bb, B, int(H), Hkv, N, d, _stream(stream)),
           "fa_fp8_quantize")


def fa_fwd_fp8(q, k, fp8_buf, o, lse, causal: bool, scale: float, stream=None) -> None:
    """S from the bf16 q, k; P V in e4m3 with V from fp8_buf; o: bf16 [B, H, N, d],
    lse: fp32 [B, H, N]."""
    B, H, Hkv, N, d = _dims(q, k)
    qs, ks, ls = _shapes(B, H, Hkv, N, d)
    bp, bb = _ws(fp8_buf)
    _check(lib().fa_fwd_fp8(_bf16(q, "q"), _bf16(k, "k"), bp, bb, _bf16(o, "o", qs),
                            _f32(lse, "lse", ls), B, H, Hkv, N, d, int(bool(causal)),
                            float(scale), _stream(stream)), "fa_fwd_fp8")


def attention_fp8(q, k, v, causal: bool = False, scale: float | None = None, stream=None):
    """FP8 forward: quantize V (into a new buffer) and attend; returns (O, LSE, buffer)."""
    import torch
    B, H, Hkv, N, d = _dims(q, k)
    if scale is None:
        scale = d ** -0.5
    n = fa_fp8_buffer_size(B, H, Hkv, N, d)
    if n == 0:
        raise FAError(FA_ERR_UNSUPPORTED, "fa_fp8_buffer_size")
    buf = torch.empty(n, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fa_fp8_quantize(v, buf, H, stream)
    fa_fwd_fp8(q, k, buf, o, lse, causal, scale, stream)
    return o, lse, buf


def fa_fwd_decode_workspace_size(B: int, H: int, Hkv: int, Nq: int, Nk: int, d: int) -> int:
    return int(lib().fa_fwd_decode_workspace_size(B, H, Hkv, Nq, Nk, d))


def fa_fwd_decode(q, k, v, o, lse, workspace, causal: bool, scale: float, stream=None) -> None:
    """q, o: bf16 [B, H, Nq, d]; k, v: bf16 [B, Hkv, Nk, d]; lse: fp32 [B, H, Nq]."""
    if q.dim() != 4 or k.dim() != 4:
        raise ValueError("q and k must be 4-D")
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d or v.shape != k.shape:
        raise ValueError(f"q {tuple(q.shape)}, k {tuple(k.shape)}, v {tuple(v.shape)} disagree")
    wp, wb = _ws(workspace)
    _check(lib().fa_fwd_decode(_bf16(q, "q"), _bf16(k, "k"), _bf16(v, "v"),
                               _bf16(o, "o", (B, H, Nq, d)), _f32(lse, "lse", (B, H, Nq)),
                               wp, wb, B, H, Hkv, Nq, Nk, d,
                               int(bool(causal)), float(scale), _stream(stream)), "fa_fwd_decode")


def attention_decode(q, k, v, causal: bool = True, scale: float | None = None, stream=None):
    """Decoding forward; allocates the output, LSE and workspace."""
    import torch
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if scale is None:
        scale = d ** -0.5
    n = fa_fwd_decode_workspace_size(B, H, Hkv, Nq, Nk, d)
    if n == 0:
        raise FAError(FA_ERR_UNSUPPORTED, "fa_fwd_decode_workspace_size")
    work = torch.empty(n, dtype=torch.uint8, device=q.device)
    o = torch.empty_like(q)
    lse = torch.empty((B, H, Nq), dtype=torch.float32, device=q.device)
    fa_fwd_decode(q, k, v, o, lse, work, causal, scale, stream)
    return o, lse


def attention(q, k, v, causal: bool = False, scale: float | None = None, stream=None,
              precise: bool = False):
    """Returns (o, lse) for bf16 CUDA q [B,H,N,d], k/v [B,Hkv,N,d]; o is bf16, or
    fp32 from fa_fwd_precise when precise=True."""
    import torch
    d = q.shape[-1]
    scale = d ** -0.5 if scale is None else scale
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    if precise:
        o = torch.empty(q.shape, dtype=torch.float32, device=q.device)
        fa_fwd_precise(q, k, v, o, lse, causal, scale, stream)
    else:
        o = torch.empty_like(q)
        fa_fwd(q, k, v, o, lse, causal, scale, stream)
    return o, lse


def attention_window(q, k, v, window: int, scale: float | None = None, stream=None):
    """Causal sliding-window attention (query i sees keys i - window < j <= i);
    returns (o, lse)."""
    import torch
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    lse = torch.empty(q.shape[:3], dtype=torch.float32, device=q.device)
    o = torch.empty_like(q)
    fa_fwd_window(q, k, v, o, lse, window, scale, stream)
    return o, lse


def attention_window_backward(q, k, v, o, lse, dout, window: int, scale: float | None = None,
                              workspace=None, stream=None):
    """Returns (dq, dk, dv) for attention_window."""
    import torch
    B, H, Hkv, N, d = _dims(q, k)
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(B, H, Hkv, N, d), dtype=torch.uint8,
                                device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_window(q, k, v, o, dout, lse, dq, dk, dv, workspace, window, scale, stream)
    return dq, dk, dv


def attention_varlen(q, k, v, cu_seqlens, max_seqlen: int, causal: bool = False,
                     scale: float | None = None, stream=None):
    """Packed variable-length sequences; returns (o [H, total, d], lse [H, total])."""
    import torch
    scale = q.shape[-1] ** -0.5 if scale is None else scale
    o = torch.empty_like(q)
    lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    fa_fwd_varlen(q, k, v, o, lse, cu_seqlens, max_seqlen, causal, scale, stream)
    return o, lse


def attention_varlen_backward(q, k, v, o, lse, dout, cu_seqlens, max_seqlen: int,
                              causal: bool = False, scale: float | None = None, workspace=None,
                              stream=None):
    """Returns (dq, dk, dv) for attention_varlen."""
    import torch
    B, H, Hkv, total, d = _varlen_dims(q, k, cu_seqlens)
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(fa_bwd_varlen_workspace_size(B, H, Hkv, max_seqlen, d),
                                dtype=torch.uint8, device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    fa_bwd_varlen(q, k, v, o, dout, lse, dq, dk, dv, workspace, cu_seqlens, max_seqlen, causal,
                  scale, stream)
    return dq, dk, dv


def attention_backward(q, k, v, o, lse, dout, causal: bool = False, scale: float | None = None,
                       workspace=None, stream=None):
    """Returns (dq, dk, dv)."""
    import torch
    B, H, Hkv, N, d = _dims(q, k)
    scale = d ** -0.5 if scale is None else scale
    if workspace is None:
        workspace = torch.empty(fa_bwd_workspace_size(B, H, Hkv, N, d), dtype=torch.uint8,
                                device=q.device)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    if o.dtype == torch.float32:
        fa_bwd_precise(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal, scale, stream)
    else:
        fa_bwd(q, k, v, o, dout, lse, dq, dk, dv, workspace, causal, scale, stream)
    return dq, dk, dv
