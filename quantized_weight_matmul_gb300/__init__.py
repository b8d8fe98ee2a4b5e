"""GB300-native quantized-weight matmul: Q4_K / Q6_K super-blocks x q8_1.

    out[t][r] = sum_k W[r][k] * x[t][k]

This package is the Python binding of the C-ABI library ``libqmm.so`` (see
``include/qmm.h``).  The ``qmm_*`` functions below have the same names and
arguments as the C entry points and only marshal arguments: pointers are
plain integers (``tensor.data_ptr()``), the stream is a ``cudaStream_t`` as an
integer.  Every step of the computation runs in the library's CUDA kernels;
there is no CPU or library-GEMM fallback.  If the library is missing or fails
to load, every call raises.

The tensor helpers at the bottom (``quantize_q8_1``, ``gemv``, ``gemm``,
``matmul``, ``block_dots``) wrap the same calls for torch CUDA tensors on the
current stream.
"""
from __future__ import annotations

import ctypes
import os
import re
import threading

from . import synth  # noqa: F401  (seeded input generators)
from .build import INCLUDE, LIB, build as build_library  # noqa: F401

Q4_K = 12
Q6_K = 14

QMM_OK = 0
QMM_EINVAL_QTYPE = -1
QMM_EINVAL_SHAPE = -2
QMM_EALIGN = -3
QMM_ENULL = -4
QMM_EWORKSPACE = -5
QMM_ESMEM = -6
QMM_ELAUNCH = -7
QMM_ETIMEOUT = -8
QMM_EDEVICE = -9

QMM_FLAG_STATIC_WEIGHTS = 1
QMM_BUILTIN_WORKSPACE_BYTES = 8 << 20

QMM_PATH_FUSED_MMVQ = 1
QMM_PATH_MMVQ = 2
QMM_PATH_MMQ = 3
# kernels one qmm_matmul call launches on each route
PATH_LAUNCHES = {QMM_PATH_FUSED_MMVQ: 1, QMM_PATH_MMVQ: 2, QMM_PATH_MMQ: 2}

_lock = threading.Lock()
_lib = None


class QmmError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        super().__init__(f"{what}: {qmm_strerror(status)} (status {status})")


_SIGS = {
    "qmm_weight_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64]),
    "qmm_q8_1_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "qmm_xq_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "qmm_xds_bytes": (ctypes.c_size_t, [ctypes.c_int64, ctypes.c_int64]),
    "qmm_gemm_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                   ctypes.c_int64]),
    "qmm_matmul_workspace_bytes": (ctypes.c_size_t, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64,
                                                     ctypes.c_int64]),
    "qmm_matmul_path": (ctypes.c_int, [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64]),
    "qmm_gemv_max_nt": (ctypes.c_int, []),
    "qmm_quantize_q8_1": (ctypes.c_int, [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_void_p,
                                         ctypes.c_void_p, ctypes.c_void_p]),
    "qmm_gemv": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_void_p]),
    "qmm_gemm": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "qmm_gemm_builtin_workspace": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                                  ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                                  ctypes.c_void_p]),
    "qmm_matmul": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p,
                                  ctypes.c_void_p, ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                  ctypes.c_int64, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_uint,
                                  ctypes.c_void_p]),
    "qmm_debug_block_dots": (ctypes.c_int, [ctypes.c_int, ctypes.c_void_p, ctypes.c_void_p,
                                            ctypes.c_void_p, ctypes.c_int64, ctypes.c_int64,
                                            ctypes.c_int64, ctypes.c_void_p, ctypes.c_int,
                                            ctypes.c_void_p, ctypes.c_size_t, ctypes.c_void_p]),
    "qmm_sync_status": (ctypes.c_int, [ctypes.c_void_p]),
    "qmm_debug_inject_stall": (ctypes.c_int, [ctypes.c_int, ctypes.c_int]),
    "qmm_strerror": (ctypes.c_char_p, [ctypes.c_int]),
}


def header_functions() -> list[str]:
    """Names of the functions declared in include/*.h."""
    names = []
    for fn in sorted(os.listdir(INCLUDE)):
        if fn.endswith(".h"):
            with open(os.path.join(INCLUDE, fn)) as f:
                text = f.read()
            names += re.findall(r"^[A-Za-z_][\w \*]*?\b(qmm_\w+)\s*\(", text, flags=re.M)
    return names


def load(path: str | None = None, build_if_missing: bool = True):
    """Load libqmm.so (building it with nvcc first if it is missing)."""
    global _lib
    with _lock:
        if _lib is not None and path is None:
            return _lib
        p = path or LIB
        if not os.path.exists(p):
            if not build_if_missing:
                raise RuntimeError(f"{p} is not built; run quantized_weight_matmul_gb300.build_library()")
            p = build_library()
        lib = ctypes.CDLL(p)
        for name, (res, args) in _SIGS.items():
            f = getattr(lib, name)
            f.restype = res
            f.argtypes = args
        if path is None:
            _lib = lib
        return lib


def _call(name, *args):
    return getattr(load(), name)(*args)


# ------------------------------------------------ C-ABI, same names -------
def qmm_weight_bytes(qtype, od, K): return _call("qmm_weight_bytes", qtype, od, K)
def qmm_q8_1_bytes(nt, K): return _call("qmm_q8_1_bytes", nt, K)
def qmm_xq_bytes(nt, K): return _call("qmm_xq_bytes", nt, K)
def qmm_xds_bytes(nt, K): return _call("qmm_xds_bytes", nt, K)
def qmm_gemm_workspace_bytes(qtype, od, K, nt): return _call("qmm_gemm_workspace_bytes", qtype, od, K, nt)
def qmm_matmul_workspace_bytes(qtype, od, K, nt): return _call("qmm_matmul_workspace_bytes", qtype, od, K, nt)
def qmm_matmul_path(qtype, od, K, nt): return _call("qmm_matmul_path", qtype, od, K, nt)
def qmm_gemv_max_nt(): return _call("qmm_gemv_max_nt")
def qmm_quantize_q8_1(x, nt, K, xq, xds, stream): return _call("qmm_quantize_q8_1", x, nt, K, xq, xds, stream)
def qmm_gemv(qtype, W, xq, xds, out, od, K, nt, stream):
    return _call("qmm_gemv", qtype, W, xq, xds, out, od, K, nt, stream)
def qmm_gemm(qtype, W, xq, xds, out, od, K, nt, workspace, ws_bytes, stream):
    return _call("qmm_gemm", qtype, W, xq, xds, out, od, K, nt, workspace, ws_bytes, stream)
def qmm_gemm_builtin_workspace(qtype, W, xq, xds, out, od, K, nt, stream):
    return _call("qmm_gemm_builtin_workspace", qtype, W, xq, xds, out, od, K, nt, stream)
def qmm_matmul(qtype, W, x, xq, xds, out, od, K, nt, workspace, ws_bytes, flags, stream):
    return _call("qmm_matmul", qtype, W, x, xq, xds, out, od, K, nt, workspace, ws_bytes, flags, stream)
def qmm_debug_block_dots(qtype, W, xq, xds, od, K, nt, dots, path, workspace, ws_bytes, stream):
    return _call("qmm_debug_block_dots", qtype, W, xq, xds, od, K, nt, dots, path, workspace, ws_bytes, stream)
def qmm_sync_status(stream): return _call("qmm_sync_status", stream)
def qmm_debug_inject_stall(on, ms): return _call("qmm_debug_inject_stall", on, ms)
def qmm_strerror(status):
    try:
        return _call("qmm_strerror", status).decode()
    except Exception:  # the library may be what failed to load
        return "unknown status"


# ------------------------------------------------- torch tensor helpers ---
def _torch():
    import torch
    return torch


def _stream():
    return _torch().cuda.current_stream().cuda_stream


def _check(rc, what):
    if rc != QMM_OK:
        raise QmmError(rc, what)


def _ptr(t):
    return 0 if t is None else t.data_ptr()


def quantize_q8_1(x):
    """x [nt][K] f32 CUDA tensor -> (xq int8 [nt][K], xds f32 [nt][K/32][2])."""
    torch = _torch()
    nt, K = x.shape
    xq = torch.empty((nt, K), dtype=torch.int8, device=x.device)
    xds = torch.empty((nt, K // 32, 2), dtype=torch.float32, device=x.device)
    _check(qmm_quantize_q8_1(_ptr(x), nt, K, _ptr(xq), _ptr(xds), _stream()), "qmm_quantize_q8_1")
    return xq, xds


def gemv(qtype, W, xq, xds, od):
    torch = _torch()
    nt, K = xq.shape
    out = torch.empty((nt, od), dtype=torch.float32, device=xq.device)
    _check(qmm_gemv(qtype, _ptr(W), _ptr(xq), _ptr(xds), _ptr(out), od, K, nt, _stream()), "qmm_gemv")
    return out


def workspace(nbytes, device):
    torch = _torch()
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


def gemm(qtype, W, xq, xds, od, ws=None):
    torch = _torch()
    nt, K = xq.shape
    need = qmm_gemm_workspace_bytes(qtype, od, K, nt)
    if ws is None:
        ws = workspace(need, xq.device)
    out = torch.empty((nt, od), dtype=torch.float32, device=xq.device)
    _check(qmm_gemm(qtype, _ptr(W), _ptr(xq), _ptr(xds), _ptr(out), od, K, nt, _ptr(ws), ws.numel(),
                    _stream()), "qmm_gemm")
    return out


def matmul(qtype, W, x, od, ws=None, flags=0, return_q8=False):
    """The whole method from f32 activations: quantize, then MMVQ or MMQ."""
    torch = _torch()
    nt, K = x.shape
    xq = torch.empty((nt, K), dtype=torch.int8, device=x.device)
    xds = torch.empty((nt, K // 32, 2), dtype=torch.float32, device=x.device)
    out = torch.empty((nt, od), dtype=torch.float32, device=x.device)
    need = qmm_matmul_workspace_bytes(qtype, od, K, nt)
    if ws is None and need:
        ws = workspace(need, x.device)
    _check(qmm_matmul(qtype, _ptr(W), _ptr(x), _ptr(xq), _ptr(xds), _ptr(out), od, K, nt, _ptr(ws),
                      0 if ws is None else ws.numel(), flags, _stream()), "qmm_matmul")
    return (out, xq, xds) if return_q8 else out


def block_dots(qtype, W, xq, xds, od, path):
    torch = _torch()
    nt, K = xq.shape
    ng = K // (32 if qtype == Q4_K or path == 1 else 16)
    dots = torch.empty((nt, od, ng), dtype=torch.int32, device=xq.device)
    ws = None
    if path == 1:
        ws = workspace(qmm_gemm_workspace_bytes(qtype, od, K, nt), xq.device)
    _check(qmm_debug_block_dots(qtype, _ptr(W), _ptr(xq), _ptr(xds), od, K, nt, _ptr(dots), path, _ptr(ws),
                                0 if ws is None else ws.numel(), _stream()), "qmm_debug_block_dots")
    return dots
