"""Build and load libfa.so, the sm_103a CUDA library behind the C ABI in
include/fa.h.  The library is built in-tree (``_lib/libfa.so``) with nvcc;
nothing here falls back to any other implementation: if the library is missing
or cannot be loaded, ``lib()`` raises."""
from __future__ import annotations

import concurrent.futures as cf
import ctypes
import os
import shutil
import subprocess
import threading

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
INCLUDE = os.path.join(ROOT, "include")
OUT_DIR = os.path.join(PKG, "_lib")
OBJ_DIR = os.path.join(PKG, "_build")
LIB_PATH = os.path.join(OUT_DIR, "libfa.so")

SOURCES = ["api.cu", "fa_fwd.cu", "fa_bwd.cu", "fa_noalloc.cu", "fa_fp8.cu", "fa_decode.cu",
           "fa_diag.cu"]
HEADERS = ["sm103_ptx.cuh", "fa_internal.h", "exp2_poly.h"]
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]
NVCC_FLAGS = ARCH + ["-O3", "-std=c++17", "-lineinfo", "-Xcompiler", "-fPIC",
                     "-Xcompiler", "-fvisibility=hidden", "-I", INCLUDE, "-I", CSRC]

_lock = threading.Lock()
_lib = None


def nvcc() -> str:
    for cand in (shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and os.path.exists(cand):
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is needed to build libfa.so")


def _stale(target: str, deps: list[str]) -> bool:
    if not os.path.exists(target):
        return True
    t = os.path.getmtime(target)
    return any(os.path.getmtime(d) > t for d in deps)


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every .cu for sm_103a (in parallel) and link libfa.so."""
    os.makedirs(OUT_DIR, exist_ok=True)
    os.makedirs(OBJ_DIR, exist_ok=True)
    hdrs = [os.path.join(CSRC, h) for h in HEADERS] + [os.path.join(INCLUDE, "fa.h")]
    cc = nvcc()
    jobs = []
    objs = []
    for src in SOURCES:
        sp = os.path.join(CSRC, src)
        op = os.path.join(OBJ_DIR, src.replace(".cu", ".o"))
        objs.append(op)
        if force or _stale(op, [sp] + hdrs):
            jobs.append([cc] + NVCC_FLAGS + ["-c", sp, "-o", op])

    def run(cmd):
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0:
            raise RuntimeError(f"nvcc failed:\n{' '.join(cmd)}\n{r.stdout}\n{r.stderr}")
        if verbose:
            print(r.stdout + r.stderr)

    with cf.ThreadPoolExecutor(max_workers=len(jobs) or 1) as ex:
        list(ex.map(run, jobs))
    if force or jobs or _stale(LIB_PATH, objs):
        tmp = f"{LIB_PATH}.{os.getpid()}.tmp"
        run([cc] + ARCH + ["-shared", "-o", tmp] + objs)
        os.replace(tmp, LIB_PATH)
    return LIB_PATH


def _bind(L: ctypes.CDLL) -> ctypes.CDLL:
    vp, i, f, sz = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_size_t
    L.fa_fwd.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.fa_fwd.restype = i
    L.fa_fwd_precise.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.fa_fwd_precise.restype = i
    L.fa_fwd_window.argtypes = [vp, vp, vp, vp, vp, i, i, i, i, i, i, f, vp]
    L.fa_fwd_window.restype = i
    L.fa_bwd_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f,
                                vp]
    L.fa_bwd_window.restype = i
    L.fa_fwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, i, f, vp]
    L.fa_fwd_varlen.restype = i
    L.fa_bwd_varlen_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_bwd_varlen_workspace_size.restype = sz
    L.fa_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, vp, i, i, i, i, i, i,
                                i, f, vp]
    L.fa_bwd_varlen.restype = i
    L.fa_bwd_workspace_size.argtypes = [i, i, i, i, i]
    L.fa_bwd_workspace_size.restype = sz
    L.fa_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_bwd.restype = i
    L.fa_bwd_precise.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f,
                                 vp]
    L.fa_bwd_precise.restype = i
    # training pair: forward that prepares the backward's workspace, and that backward
    L.fa_fwd_train.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_fwd_train.restype = i
    L.fa_fwd_train_precise.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_fwd_train_precise.restype = i
    L.fa_bwd_train.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_bwd_train.restype = i
    L.fa_fwd_window_train.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_fwd_window_train.restype = i
    L.fa_bwd_window_train.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i,
                                      f, vp]
    L.fa_bwd_window_train.restype = i
    L.fa_bwd_train_precise.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i,
                                       f, vp]
    L.fa_bwd_train_precise.restype = i
    L.fa_exp2_check.argtypes = [vp, vp, vp, i, vp]
    L.fa_exp2_check.restype = i
    L.fa_ex2_rate.argtypes = [vp, i, i, vp]
    L.fa_ex2_rate.restype = i
    L.fa_bwd_preprocess_train.argtypes = [vp, vp, vp, sz, i, i, i, i, i, vp]
    L.fa_bwd_preprocess_train.restype = i
    L.fa_bwd_preprocess_train_precise.argtypes = [vp, vp, vp, sz, i, i, i, i, i, vp]
    L.fa_bwd_preprocess_train_precise.restype = i
    L.fa_bwd_preprocess.argtypes = [vp, vp, vp, vp, sz, i, i, i, i, i, vp]
    L.fa_bwd_preprocess.restype = i
    L.fa_bwd_preprocess_precise.argtypes = [vp, vp, vp, vp, sz, i, i, i, i, i, vp]
    L.fa_bwd_preprocess_precise.restype = i
    L.fa_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_bwd_dkdv.restype = i
    L.fa_bwd_dkdv_window.argtypes = [vp, vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, f, vp]
    L.fa_bwd_dkdv_window.restype = i
    L.fa_bwd_dq_convert.argtypes = [vp, sz, vp, i, i, i, i, i, f, vp]
    L.fa_bwd_dq_convert.restype = i
    L.fa_bwd_static_scratch.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, i, i, i, i, i, i, f,
                                        vp]
    L.fa_bwd_static_scratch.restype = i
    L.fa_device_status.argtypes = [vp]
    L.fa_device_status.restype = i
    L.fa_device_status_detail.argtypes = [ctypes.POINTER(i), ctypes.POINTER(i)]
    L.fa_device_status_detail.restype = None
    L.fa_status_string.argtypes = [i]
    L.fa_status_string.restype = ctypes.c_char_p
    L.fa_kernel_launches.argtypes = []
    L.fa_kernel_launches.restype = ctypes.c_longlong
    L.fa_watchdog_selftest.argtypes = [ctypes.c_longlong, vp]
    L.fa_watchdog_selftest.restype = i
    L.fa_fp8_buffer_size.argtypes = [i, i, i, i, i]
    L.fa_fp8_buffer_size.restype = sz
    L.fa_fp8_quantize.argtypes = [vp, vp, sz, i, i, i, i, i, vp]
    L.fa_fp8_quantize.restype = i
    L.fa_fwd_fp8.argtypes = [vp, vp, vp, sz, vp, vp, i, i, i, i, i, i, f, vp]
    L.fa_fwd_fp8.restype = i
    L.fa_fwd_decode_workspace_size.argtypes = [i, i, i, i, i, i]
    L.fa_fwd_decode_workspace_size.restype = sz
    L.fa_fwd_decode.argtypes = [vp, vp, vp, vp, vp, vp, sz, i, i, i, i, i, i, i, f, vp]
    L.fa_fwd_decode.restype = i
    return L


def lib() -> ctypes.CDLL:
    """The loaded libfa.so.  Raises if it was not built (call build())."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise RuntimeError(
                    f"{LIB_PATH} is missing: build it with "
                    "exact_attention_online_gb300.build() (nvcc, sm_103a)")
            _lib = _bind(ctypes.CDLL(LIB_PATH))
        return _lib


# Every symbol include/fa.h declares.
EXPORTS = ["fa_fwd", "fa_fwd_precise", "fa_bwd_workspace_size", "fa_bwd", "fa_bwd_precise",
           "fa_bwd_preprocess", "fa_bwd_preprocess_precise", "fa_bwd_dkdv", "fa_bwd_dq_convert",
           "fa_bwd_static_scratch", "fa_device_status", "fa_device_status_detail",
           "fa_status_string", "fa_kernel_launches", "fa_watchdog_selftest",
           "fa_fp8_buffer_size", "fa_fp8_quantize", "fa_fwd_fp8",
           "fa_fwd_decode_workspace_size", "fa_fwd_decode", "fa_fwd_window", "fa_bwd_window",
           "fa_bwd_dkdv_window", "fa_fwd_varlen", "fa_bwd_varlen_workspace_size",
           "fa_bwd_varlen", "fa_fwd_train", "fa_fwd_train_precise", "fa_bwd_train",
           "fa_bwd_train_precise", "fa_bwd_preprocess_train", "fa_bwd_preprocess_train_precise", "fa_exp2_check",
           "fa_ex2_rate",
           "fa_fwd_window_train", "fa_bwd_window_train"]
