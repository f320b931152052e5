"""fp64 CPU oracle for exact attention.  TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The CUDA library never calls it,
and the two share no code: this package holds its own C source
(``attn_oracle.c``), built with the host C compiler, and a ctypes binding.

Functions (NumPy float64 in, NumPy float64 out; layouts as in the C file):
    attn_fwd          standard attention, materialised score rows, 3-loop safe
                      softmax (FlashAttention blog, "(Safe) Softmax"); optional
                      row subset and optional P output.
    attn_fwd_online   one-pass online-softmax attention in key blocks, normalised
                      (blog "FlashAttention", o_N = o'_N) or deferred division
                      (FlashAttention-2 answer on non-matmul FLOPs).
    attn_fwd_window / attn_bwd_window
                      causal sliding window: query i sees keys i - W < j <= i.
    attn_fwd_varlen / attn_bwd_varlen
                      packed variable-length sequences ([H][T][d], offsets
                      cu_seqlens), each sequence its own attention problem.
    attn_fwd_decode   fewer query rows than keys (the decoding setting), the
                      queries being the last positions (bottom-right causal).
    attn_bwd          analytic gradients dQ, dK, dV and D = rowsum(dO * O).
    e4m3_encode/decode  the e4m3 format from its definition (round to nearest,
                      ties to even, saturating at 448).
    fp8_quantize      per-(batch, head, 128-row block) quantisation of Q, K, V
                      with scale amax / 448 (FlashAttention-3 summary, "block
                      quantization"; the granularity is this repository's
                      reading), V also transposed; fp8_quantize_v for V alone,
                      fp8_dequantize(_v) for the values the codes stand for.
    incoherent_rotate x times diag(signs) Hd / sqrt(d), the reading of the
                      FlashAttention-3 summary's "incoherent processing".
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "attn_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_lock = threading.Lock()
_libs: dict[int, ctypes.CDLL] = {}


def lib_path(mutant: int = 0) -> str:
    name = "liboracle.so" if mutant == 0 else f"liboracle_mutant{mutant}.so"
    return os.path.join(_BUILD, name)


def build(mutant: int = 0, force: bool = False) -> str:
    """Compile the oracle (or one planted-mistake copy of it) with gcc."""
    out = lib_path(mutant)
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(_SRC):
        return out
    os.makedirs(_BUILD, exist_ok=True)
    tmp = f"{out}.{os.getpid()}.tmp"
    cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
           f"-DORACLE_MUTANT={int(mutant)}", "-o", tmp, _SRC, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib: ctypes.CDLL) -> ctypes.CDLL:
    dp = ctypes.POINTER(ctypes.c_double)
    i, d = ctypes.c_int, ctypes.c_double
    lib.oracle_attn_fwd.argtypes = [dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, d,
                                    ctypes.POINTER(ctypes.c_longlong), ctypes.c_longlong]
    lib.oracle_attn_fwd.restype = i
    lib.oracle_attn_fwd_online.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, d, i, i]
    lib.oracle_attn_fwd_online.restype = i
    lib.oracle_attn_bwd.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, d]
    lib.oracle_attn_bwd.restype = i
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = i
    lib.oracle_attn_fwd_window.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, d]
    lib.oracle_attn_fwd_window.restype = i
    lib.oracle_attn_bwd_window.argtypes = [dp, dp, dp, dp, dp, dp, dp, dp, i, i, i, i, i, i, d]
    lib.oracle_attn_bwd_window.restype = i
    lib.oracle_attn_fwd_decode.argtypes = [dp, dp, dp, dp, dp, i, i, i, i, i, i, i, d]
    lib.oracle_attn_fwd_decode.restype = i
    u8p = ctypes.POINTER(ctypes.c_ubyte)
    fp = ctypes.POINTER(ctypes.c_float)
    ll = ctypes.c_longlong
    lib.oracle_e4m3_encode.argtypes = [ctypes.c_float]
    lib.oracle_e4m3_encode.restype = ctypes.c_ubyte
    lib.oracle_e4m3_decode.argtypes = [ctypes.c_ubyte]
    lib.oracle_e4m3_decode.restype = ctypes.c_double
    lib.oracle_fp8_quant_block.argtypes = [fp, i, i, ll, u8p, ll, u8p, ll, fp]
    lib.oracle_fp8_quant_block.restype = i
    lib.oracle_hadamard_rotate.argtypes = [dp, i, i, ctypes.POINTER(ctypes.c_byte), dp]
    lib.oracle_hadamard_rotate.restype = i
    return lib


def load(mutant: int = 0) -> ctypes.CDLL:
    with _lock:
        if mutant not in _libs:
            _libs[mutant] = _bind(ctypes.CDLL(build(mutant)))
        return _libs[mutant]


def _ptr(a: np.ndarray | None):
    if a is None:
        return None
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _shape(q: np.ndarray, k: np.ndarray):
    B, H, N, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if (Bk, Nk, dk) != (B, N, d):
        raise ValueError(f"q {q.shape} and k {k.shape} disagree")
    return B, H, Hkv, N, d


def _check(rc: int, what: str):
    if rc != 0:
        raise RuntimeError(f"{what} failed with code {rc}")


def num_threads(mutant: int = 0) -> int:
    return int(load(mutant).oracle_num_threads())


def attn_fwd(q, k, v, causal: bool, scale: float, rows=None, return_p: bool = False,
             mutant: int = 0):
    """Standard attention.  q [B,H,N,d], k/v [B,Hkv,N,d].

    rows=None: returns (O [B,H,N,d], LSE [B,H,N]) (+ P [B,H,N,N] if return_p).
    rows=array of flat row ids (b*H + h)*N + i: returns (O [R,d], LSE [R]).
    """
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, N, d = _shape(q, k)
    lib = load(mutant)
    if rows is None:
        o = np.empty_like(q)
        lse = np.empty((B, H, N))
        p = np.empty((B, H, N, N)) if return_p else None
        rc = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), _ptr(p),
                                 B, H, Hkv, N, d, int(causal), float(scale), None, 0)
        _check(rc, "oracle_attn_fwd")
        return (o, lse, p) if return_p else (o, lse)
    if return_p:
        raise ValueError("return_p needs rows=None")
    r = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    o = np.empty((r.size, d))
    lse = np.empty(r.size)
    rc = lib.oracle_attn_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse), None,
                             B, H, Hkv, N, d, int(causal), float(scale),
                             r.ctypes.data_as(ctypes.POINTER(ctypes.c_longlong)), r.size)
    _check(rc, "oracle_attn_fwd(rows)")
    return o, lse


def attn_fwd_online(q, k, v, causal: bool, scale: float, block: int = 1,
                    deferred: bool = False, mutant: int = 0):
    """One-pass online-softmax attention; returns (O, LSE)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, N, d = _shape(q, k)
    o = np.empty_like(q)
    lse = np.empty((B, H, N))
    rc = load(mutant).oracle_attn_fwd_online(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             B, H, Hkv, N, d, int(causal), float(scale),
                                             int(block), int(deferred))
    _check(rc, "oracle_attn_fwd_online")
    return o, lse


def attn_fwd_window(q, k, v, window: int, scale: float, mutant: int = 0):
    """Causal sliding-window attention: query i sees keys i - window < j <= i.
    Returns (O, LSE)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Hkv, N, d = _shape(q, k)
    o = np.empty_like(q)
    lse = np.empty((B, H, N))
    rc = load(mutant).oracle_attn_fwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             B, H, Hkv, N, d, int(window), float(scale))
    _check(rc, "oracle_attn_fwd_window")
    return o, lse


def attn_bwd_window(q, k, v, dout, window: int, scale: float, mutant: int = 0):
    """Analytic backward of attn_fwd_window; returns (dQ, dK, dV, D)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Hkv, N, d = _shape(q, k)
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    D = np.empty((B, H, N))
    rc = load(mutant).oracle_attn_bwd_window(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq),
                                             _ptr(dk), _ptr(dv), _ptr(D), B, H, Hkv, N, d,
                                             int(window), float(scale))
    _check(rc, "oracle_attn_bwd_window")
    return dq, dk, dv, D


def attn_fwd_decode(q, k, v, causal: bool, scale: float, mutant: int = 0):
    """Fewer queries than keys: q [B,H,Nq,d], k/v [B,Hkv,Nk,d], Nq <= Nk; the
    queries are the last Nq positions (causal: query r sees keys
    j <= r + Nk - Nq).  Returns (O [B,H,Nq,d], LSE [B,H,Nq])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, Nq, d = q.shape
    Hkv, Nk = k.shape[1], k.shape[2]
    if k.shape[0] != B or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("q, k, v shapes disagree")
    o = np.empty_like(q)
    lse = np.empty((B, H, Nq))
    rc = load(mutant).oracle_attn_fwd_decode(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                                             B, H, Hkv, Nq, Nk, d, int(causal), float(scale))
    _check(rc, "oracle_attn_fwd_decode")
    return o, lse


def attn_bwd(q, k, v, dout, causal: bool, scale: float, mutant: int = 0):
    """Analytic backward; returns (dQ, dK, dV, D)."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    B, H, Hkv, N, d = _shape(q, k)
    if dout.shape != q.shape:
        raise ValueError("dout must have q's shape")
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    D = np.empty((B, H, N))
    rc = load(mutant).oracle_attn_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), _ptr(dq),
                                      _ptr(dk), _ptr(dv), _ptr(D), B, H, Hkv, N, d,
                                      int(causal), float(scale))
    _check(rc, "oracle_attn_bwd")
    return dq, dk, dv, D


# ------------------------------------------------------------------ varlen
# Packed variable-length batches (FlashAttention-2 review thread, the
# authors' answer "FA2 with variable sequence lengths": sequences concatenated
# without padding, their lengths in an array).  Layout q [H][T][d], k, v
# [Hkv][T][d]; sequence b is rows cu[b] .. cu[b+1] - 1.  Each sequence is an
# independent attention problem, so it is cut out and handed to attn_fwd /
# attn_bwd.  Mutant 17 (a planted mistake for the pins) lets each sequence
# run one row into the next.

def _varlen_spans(cu, T, mutant):
    cu = [int(x) for x in np.asarray(cu).ravel()]
    if cu[0] != 0 or cu[-1] != T or any(b < a for a, b in zip(cu, cu[1:])):
        raise ValueError("cu_seqlens must rise from 0 to the packed row count")
    for a, e in zip(cu, cu[1:]):
        if e > a:
            yield a, (min(e + 1, T) if mutant == 17 else e), e


def attn_fwd_varlen(q, k, v, cu_seqlens, causal: bool, scale: float, mutant: int = 0):
    """Returns (O [H][T][d], LSE [H][T])."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    H, T, d = q.shape
    o = np.zeros_like(q)
    lse = np.zeros((H, T))
    for a, e, keep in _varlen_spans(cu_seqlens, T, mutant):
        ob, lb = attn_fwd(q[None, :, a:e], k[None, :, a:e], v[None, :, a:e], causal, scale,
                          mutant=mutant)
        o[:, a:keep] = ob[0, :, :keep - a]
        lse[:, a:keep] = lb[0, :, :keep - a]
    return o, lse


def attn_bwd_varlen(q, k, v, dout, cu_seqlens, causal: bool, scale: float, mutant: int = 0):
    """Returns (dQ, dK, dV, D) in the packed layout."""
    q, k, v, dout = _f64(q), _f64(k), _f64(v), _f64(dout)
    H, T, d = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    D = np.zeros((H, T))
    for a, e, keep in _varlen_spans(cu_seqlens, T, mutant):
        g = attn_bwd(q[None, :, a:e], k[None, :, a:e], v[None, :, a:e], dout[None, :, a:e],
                     causal, scale, mutant=mutant)
        for dst, src in zip((dq, dk, dv, D), g):
            dst[:, a:keep] = src[0, :, :keep - a]
    return dq, dk, dv, D


# --------------------------------------------------------------------- FP8
FP8_BLOCK = 128


def e4m3_encode(x: float, mutant: int = 0) -> int:
    return int(load(mutant).oracle_e4m3_encode(ctypes.c_float(float(x))))


def e4m3_decode(code: int, mutant: int = 0) -> float:
    return float(load(mutant).oracle_e4m3_decode(ctypes.c_ubyte(int(code))))


def e4m3_decode_table(mutant: int = 0) -> np.ndarray:
    """Values of all 256 codes (NaN for the two NaN codes)."""
    return np.array([e4m3_decode(c, mutant) for c in range(256)])


def _quant_blocks(x: np.ndarray, transpose: bool, mutant: int):
    """x: [G][N][d] float32.  Returns (codes, scales): codes [G][Np][d] (or
    [G][d][Np] when transpose), scales [G][Np / 128] float32."""
    G, N, d = x.shape
    Np = (N + FP8_BLOCK - 1) // FP8_BLOCK * FP8_BLOCK
    nblk = Np // FP8_BLOCK
    out = np.zeros((G, d, Np) if transpose else (G, Np, d), dtype=np.uint8)
    scales = np.zeros((G, nblk), dtype=np.float32)
    lib = load(mutant)
    u8p = ctypes.POINTER(ctypes.c_ubyte)
    fp = ctypes.POINTER(ctypes.c_float)
    x = np.ascontiguousarray(x, dtype=np.float32)
    sc = ctypes.c_float()
    for g in range(G):
        for b in range(nblk):
            r0 = b * FP8_BLOCK
            rows = min(FP8_BLOCK, N - r0)
            src = x[g, r0:r0 + rows]
            if transpose:
                dst = out[g]
                rc = lib.oracle_fp8_quant_block(
                    src.ctypes.data_as(fp), rows, d, d, None, 0,
                    ctypes.cast(dst.ctypes.data + r0, u8p), Np, ctypes.byref(sc))
            else:
                dst = out[g, r0:r0 + rows]
                rc = lib.oracle_fp8_quant_block(
                    src.ctypes.data_as(fp), rows, d, d, dst.ctypes.data_as(u8p), d,
                    None, 0, ctypes.byref(sc))
            _check(rc, "oracle_fp8_quant_block")
            scales[g, b] = sc.value
    return out, scales


def fp8_quantize(q, k, v, mutant: int = 0) -> dict:
    """Block quantisation of bf16 Q [B,H,N,d], K and V [B,Hkv,N,d] (given as
    float32 or float64 arrays holding the bf16 values).  Returns
    q8 [B*H][Np][d], k8 [B*Hkv][Np][d], v8t [B*Hkv][d][Np] (uint8 codes, zero
    on padded rows), sq [B*H][nblk], sk, sv [B*Hkv][nblk] (float32 scales) and
    svmax [B*Hkv] (the largest V scale of each head)."""
    q = np.asarray(q, dtype=np.float32)
    k = np.asarray(k, dtype=np.float32)
    v = np.asarray(v, dtype=np.float32)
    B, H, N, d = q.shape
    Hkv = k.shape[1]
    q8, sq = _quant_blocks(q.reshape(B * H, N, d), False, mutant)
    k8, sk = _quant_blocks(k.reshape(B * Hkv, N, d), False, mutant)
    v8t, sv = _quant_blocks(v.reshape(B * Hkv, N, d), True, mutant)
    return {"q8": q8, "k8": k8, "v8t": v8t, "sq": sq, "sk": sk, "sv": sv,
            "svmax": sv.max(axis=1).astype(np.float32)}


def fp8_quantize_v(v, mutant: int = 0) -> dict:
    """Block quantisation of bf16 V [B,Hkv,N,d] alone (the operand the FP8
    forward takes in e4m3): v8t [B*Hkv][d][Np], sv [B*Hkv][nblk], svmax."""
    v = np.asarray(v, dtype=np.float32)
    B, Hkv, N, d = v.shape
    v8t, sv = _quant_blocks(v.reshape(B * Hkv, N, d), True, mutant)
    return {"v8t": v8t, "sv": sv, "svmax": sv.max(axis=1).astype(np.float32)}


def fp8_dequantize_v(qd: dict, B: int, Hkv: int, N: int, d: int) -> np.ndarray:
    """The values V's codes stand for (codes times block scales), float64
    [B,Hkv,N,d]."""
    vals = np.swapaxes(e4m3_decode_table()[qd["v8t"]], 1, 2)
    s = np.repeat(qd["sv"].astype(np.float64), FP8_BLOCK, axis=1)[:, :, None]
    return (vals * s)[:, :N, :].reshape(B, Hkv, N, d)


def incoherent_rotate(x, signs, mutant: int = 0) -> np.ndarray:
    """x [..., d] times M = diag(signs) Hd / sqrt(d) (incoherent processing of
    Q and K: scores unchanged, large entries spread over the channels); d a
    power of two, signs a sequence of d values +-1."""
    x = _f64(x)
    d = x.shape[-1]
    sg = np.ascontiguousarray(np.asarray(signs, dtype=np.int8))
    if sg.shape != (d,) or not np.all(np.abs(sg) == 1):
        raise ValueError("signs must be d values of +-1")
    flat = np.ascontiguousarray(x.reshape(-1, d))
    out = np.empty_like(flat)
    _check(load(mutant).oracle_hadamard_rotate(
        _ptr(flat), flat.shape[0], d, sg.ctypes.data_as(ctypes.POINTER(ctypes.c_byte)),
        _ptr(out)), "oracle_hadamard_rotate")
    return out.reshape(x.shape)


def fp8_dequantize(qd: dict, B: int, H: int, Hkv: int, N: int, d: int):
    """The values the quantised tensors stand for (codes times block scales),
    float64, in the [B,H,N,d] / [B,Hkv,N,d] layouts."""
    table = e4m3_decode_table()
    nb = FP8_BLOCK

    def expand(codes, scales, G, transpose):
        vals = table[codes]
        if transpose:
            vals = np.swapaxes(vals, 1, 2)
        s = np.repeat(scales.astype(np.float64), nb, axis=1)[:, :, None]
        return (vals * s)[:, :N, :]
    return (expand(qd["q8"], qd["sq"], B * H, False).reshape(B, H, N, d),
            expand(qd["k8"], qd["sk"], B * Hkv, False).reshape(B, Hkv, N, d),
            expand(qd["v8t"], qd["sv"], B * Hkv, True).reshape(B, Hkv, N, d))
