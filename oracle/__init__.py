"""CPU oracle for the quantized-weight matmul (test infrastructure only).

The oracle is a plain scalar C implementation (``qmm_oracle.c``) of what the
method computes: Q4_K / Q6_K super-block decode, q8_1 activation quantization,
exact int32 block dots, and the f64-accumulated output.  It shares no code with
the CUDA library.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package; the product path never
does.

``build()`` compiles the shared library with gcc (``-O2``, no fast-math, no FMA
contraction) into ``oracle/_build/``; the wrappers below take and return numpy
arrays.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

Q4_K = 12
Q6_K = 14
BLOCK_BYTES = {Q4_K: 144, Q6_K: 210}

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "qmm_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libqmm_oracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c11", "-fPIC", "-shared", "-pthread", "-ffp-contract=off",
          "-fno-fast-math", "-Wall"]


def build(force: bool = False) -> str:
    """Compile the oracle library if it is missing or older than its source."""
    os.makedirs(_BUILD, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".{os.getpid()}.tmp"
    subprocess.run(["gcc", *CFLAGS, _SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def compile_variant(src_text: str, out_path: str) -> str:
    """Compile a modified copy of the oracle source (used by mutation tests)."""
    src_path = out_path + ".c"
    with open(src_path, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", *CFLAGS, src_path, "-o", out_path, "-lm"], check=True)
    return out_path


def source_text() -> str:
    with open(_SRC) as f:
        return f.read()


def _bind(lib):
    i64, i32 = ctypes.c_int64, ctypes.c_int
    vp = ctypes.c_void_p
    lib.oracle_weight_bytes.restype = i64
    lib.oracle_weight_bytes.argtypes = [i32, i64, i64]
    lib.oracle_dequantize.restype = i32
    lib.oracle_dequantize.argtypes = [i32, vp, i64, i64, vp]
    lib.oracle_quantize_q8_1.restype = i32
    lib.oracle_quantize_q8_1.argtypes = [vp, i64, i64, vp, vp]
    lib.oracle_block_dots.restype = i32
    lib.oracle_block_dots.argtypes = [i32, vp, vp, i64, i64, i64, vp]
    lib.oracle_matmul_q8_1.restype = i32
    lib.oracle_matmul_q8_1.argtypes = [i32, vp, vp, vp, i64, i64, i64, vp, i32]
    lib.oracle_matmul.restype = i32
    lib.oracle_matmul.argtypes = [i32, vp, vp, i64, i64, i64, vp, i32]
    return lib


def load(path: str | None = None):
    """Load the oracle library (building it first when needed)."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    with _lock:
        if _lib is None:
            _lib = _bind(ctypes.CDLL(build()))
    return _lib


class Oracle:
    """numpy front end over one compiled oracle library (default or a variant)."""

    def __init__(self, lib=None):
        self.lib = lib if lib is not None else load()

    @staticmethod
    def _ptr(a: np.ndarray):
        assert a.flags["C_CONTIGUOUS"]
        return a.ctypes.data_as(ctypes.c_void_p)

    @staticmethod
    def _check(rc: int, what: str):
        if rc != 0:
            raise ValueError(f"oracle {what} failed with status {rc}")

    def weight_bytes(self, qtype: int, od: int, K: int) -> int:
        return int(self.lib.oracle_weight_bytes(qtype, od, K))

    def dequantize(self, qtype: int, W: np.ndarray, od: int, K: int) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        out = np.empty((od, K), dtype=np.float64)
        self._check(self.lib.oracle_dequantize(qtype, self._ptr(W), od, K, self._ptr(out)),
                    "dequantize")
        return out

    def quantize_q8_1(self, x: np.ndarray):
        x = np.ascontiguousarray(x, dtype=np.float32)
        nt, K = x.shape
        xq = np.empty((nt, K), dtype=np.int8)
        xds = np.empty((nt, K // 32, 2), dtype=np.float32)
        self._check(self.lib.oracle_quantize_q8_1(self._ptr(x), nt, K, self._ptr(xq),
                                                  self._ptr(xds)), "quantize")
        return xq, xds

    def block_dots(self, qtype: int, W: np.ndarray, xq: np.ndarray, od: int) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        nt, K = xq.shape
        ng = K // (32 if qtype == Q4_K else 16)
        dots = np.empty((nt, od, ng), dtype=np.int32)
        self._check(self.lib.oracle_block_dots(qtype, self._ptr(W), self._ptr(xq), od, K, nt,
                                               self._ptr(dots)), "block_dots")
        return dots

    def matmul_q8_1(self, qtype: int, W: np.ndarray, xq: np.ndarray, xds: np.ndarray, od: int,
                    nthreads: int = 1) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        xq = np.ascontiguousarray(xq, dtype=np.int8)
        xds = np.ascontiguousarray(xds, dtype=np.float32)
        nt, K = xq.shape
        out = np.empty((nt, od), dtype=np.float32)
        self._check(self.lib.oracle_matmul_q8_1(qtype, self._ptr(W), self._ptr(xq),
                                                self._ptr(xds), od, K, nt, self._ptr(out),
                                                nthreads), "matmul_q8_1")
        return out

    def matmul(self, qtype: int, W: np.ndarray, x: np.ndarray, od: int,
               nthreads: int = 1) -> np.ndarray:
        W = np.ascontiguousarray(W, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float32)
        nt, K = x.shape
        out = np.empty((nt, od), dtype=np.float32)
        self._check(self.lib.oracle_matmul(qtype, self._ptr(W), self._ptr(x), od, K, nt,
                                           self._ptr(out), nthreads), "matmul")
        return out


def default_threads() -> int:
    return max(1, len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
               else (os.cpu_count() or 1))
