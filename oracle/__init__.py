"""CPU oracle for the PN weight formats (test infrastructure).

Only the tests, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The CUDA library never loads it, and the
two share no code.  The arithmetic lives in ``pn_oracle.c`` (plain C, fp64
accumulation); this module compiles it with gcc and wraps it with ctypes over
numpy arrays.

Source: tensorless docs, "Why a P100-native weight format" (block layout,
half-word packing, exact decode, mid-tread codes with a signed scale; the
runtime Hadamard rotation of the activations, section "How Qwen3.8-27B-PN3
uses it"); tensorless docs, "What the fork adds", and the v100-skinny README,
"How QPN works" (prefill: weights rebuilt transiently, then a GEMM).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

PN3T = 124
PN4T = 125

_HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(_HERE, "pn_oracle.c")
LIBRARY = os.path.join(_HERE, "libpn_oracle.so")
CFLAGS = ["-O2", "-std=c11", "-fno-fast-math", "-ffp-contract=off", "-Wall", "-Wextra",
          "-shared", "-fPIC"]

_lock = threading.Lock()
_lib = None


def compile_oracle(source: str = SOURCE, output: str = LIBRARY, extra=()) -> str:
    """Compile an oracle source file into a shared library with gcc."""
    cmd = ["gcc", *CFLAGS, *extra, source, "-o", output, "-lm"]
    subprocess.run(cmd, check=True, capture_output=True, text=True)
    return output


def load(path: str | None = None) -> ctypes.CDLL:
    """Load (building first if needed) the oracle library and declare its symbols."""
    global _lib
    if path is None:
        with _lock:
            if _lib is not None:
                return _lib
            if (not os.path.exists(LIBRARY)
                    or os.path.getmtime(LIBRARY) < os.path.getmtime(SOURCE)):
                compile_oracle()
            _lib = _declare(ctypes.CDLL(LIBRARY))
            return _lib
    return _declare(ctypes.CDLL(path))


def _declare(lib: ctypes.CDLL) -> ctypes.CDLL:
    c_void_p, i64 = ctypes.c_void_p, ctypes.c_int64
    lib.oracle_row_bytes.restype = ctypes.c_size_t
    lib.oracle_row_bytes.argtypes = [ctypes.c_int, i64]
    lib.oracle_pack.restype = ctypes.c_int
    lib.oracle_pack.argtypes = [ctypes.c_int, c_void_p, i64, i64, c_void_p]
    lib.oracle_unpack.restype = ctypes.c_int
    lib.oracle_unpack.argtypes = [ctypes.c_int, c_void_p, i64, i64, c_void_p]
    lib.oracle_gemv.restype = ctypes.c_int
    lib.oracle_gemv.argtypes = [ctypes.c_int, c_void_p, i64, i64, c_void_p, ctypes.c_int,
                                c_void_p, c_void_p]
    lib.oracle_half_to_float.restype = ctypes.c_float
    lib.oracle_half_to_float.argtypes = [ctypes.c_uint16]
    lib.oracle_float_to_half.restype = ctypes.c_uint16
    lib.oracle_float_to_half.argtypes = [ctypes.c_float]
    lib.oracle_hadamard.restype = ctypes.c_int
    lib.oracle_hadamard.argtypes = [c_void_p, ctypes.c_int, i64, ctypes.c_int, c_void_p, c_void_p]
    lib.oracle_unpack_f16.restype = ctypes.c_int
    lib.oracle_unpack_f16.argtypes = [ctypes.c_int, c_void_p, i64, i64, c_void_p]
    lib.oracle_gemm_f16.restype = ctypes.c_int
    lib.oracle_gemm_f16.argtypes = [c_void_p, i64, i64, c_void_p, ctypes.c_int, c_void_p, c_void_p]
    if hasattr(lib, "oracle_gptq"):
        lib.oracle_gptq.restype = ctypes.c_int
        lib.oracle_gptq.argtypes = [ctypes.c_int, c_void_p, i64, i64, c_void_p, i64, ctypes.c_double, c_void_p]
    return lib


class Oracle:
    """numpy-facing wrapper around one compiled oracle library."""

    def __init__(self, lib: ctypes.CDLL | None = None):
        self.lib = lib if lib is not None else load()

    def row_bytes(self, pn_type: int, K: int) -> int:
        return int(self.lib.oracle_row_bytes(pn_type, K))

    def pack(self, pn_type: int, w: np.ndarray) -> np.ndarray:
        """fp32 weights [N][K] -> PN bytes [N][row_bytes] (uint8)."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        N, K = w.shape
        rb = self.row_bytes(pn_type, K)
        if rb == 0:
            raise ValueError(f"K={K} is not a whole number of blocks")
        out = np.zeros((N, rb), dtype=np.uint8)
        rc = self.lib.oracle_pack(pn_type, w.ctypes.data, N, K, out.ctypes.data)
        if rc:
            raise ValueError(f"oracle_pack failed ({rc})")
        return out

    def unpack(self, pn_type: int, W: np.ndarray, K: int) -> np.ndarray:
        """PN bytes [N][row_bytes] -> fp32 weights [N][K]."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        N = W.shape[0]
        if W.shape[1] != self.row_bytes(pn_type, K):
            raise ValueError("row size does not match K")
        w = np.empty((N, K), dtype=np.float32)
        rc = self.lib.oracle_unpack(pn_type, W.ctypes.data, N, K, w.ctypes.data)
        if rc:
            raise ValueError(f"oracle_unpack failed ({rc})")
        return w

    def gemv(self, pn_type: int, W: np.ndarray, K: int, x: np.ndarray,
             want_abs: bool = True):
        """y[M][N] = W x^T in fp64, rounded to fp32; also sum |w x| if asked."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float16)
        if x.ndim == 1:
            x = x[None, :]
        M = x.shape[0]
        N = W.shape[0]
        if x.shape[1] != K or W.shape[1] != self.row_bytes(pn_type, K):
            raise ValueError("shape mismatch")
        y = np.empty((M, N), dtype=np.float32)
        a = np.empty((M, N), dtype=np.float64) if want_abs else None
        rc = self.lib.oracle_gemv(pn_type, W.ctypes.data, N, K, x.view(np.uint16).ctypes.data,
                                  M, y.ctypes.data, a.ctypes.data if want_abs else None)
        if rc:
            raise ValueError(f"oracle_gemv failed ({rc})")
        return (y, a) if want_abs else y

    def gemv_threads(self, pn_type: int, W: np.ndarray, K: int, x: np.ndarray,
                     threads: int):
        """Same GEMV with the rows split over ``threads`` OS threads.

        ctypes releases the GIL for the duration of each C call, so the row
        ranges run in parallel; each row is still computed by the plain loop.
        """
        W = np.ascontiguousarray(W, dtype=np.uint8)
        x = np.ascontiguousarray(x, dtype=np.float16)
        if x.ndim == 1:
            x = x[None, :]
        M, N = x.shape[0], W.shape[0]
        y = np.empty((M, N), dtype=np.float32)
        bounds = np.linspace(0, N, threads + 1).astype(np.int64)
        parts = [None] * threads

        def run(i):
            lo, hi = bounds[i], bounds[i + 1]
            if hi > lo:
                parts[i] = self.gemv(pn_type, W[lo:hi], K, x, want_abs=False)

        ts = [threading.Thread(target=run, args=(i,)) for i in range(threads)]
        for t in ts:
            t.start()
        for t in ts:
            t.join()
        for i in range(threads):
            lo, hi = bounds[i], bounds[i + 1]
            if hi > lo:
                y[:, lo:hi] = parts[i]
        return y

    def hadamard(self, x: np.ndarray, block: int, want_f32: bool = False):
        """Block Hadamard rotation of fp16 activations [M][K] (reading R10):
        returns fp16 [M][K] and, if asked, the fp32 values before rounding."""
        x = np.ascontiguousarray(x, dtype=np.float16)
        if x.ndim == 1:
            x = x[None, :]
        M, K = x.shape
        out = np.empty((M, K), dtype=np.float16)
        o32 = np.empty((M, K), dtype=np.float32) if want_f32 else None
        rc = self.lib.oracle_hadamard(x.view(np.uint16).ctypes.data, M, K, block,
                                      out.view(np.uint16).ctypes.data,
                                      o32.ctypes.data if want_f32 else None)
        if rc:
            raise ValueError(f"oracle_hadamard failed ({rc})")
        return (out, o32) if want_f32 else out

    def unpack_f16(self, pn_type: int, W: np.ndarray, K: int) -> np.ndarray:
        """PN bytes [N][row_bytes] -> fp16 weights [N][K], each the exact
        decode rounded once to fp16 (reading R11, prefill reconstruction)."""
        W = np.ascontiguousarray(W, dtype=np.uint8)
        N = W.shape[0]
        if W.shape[1] != self.row_bytes(pn_type, K):
            raise ValueError("row size does not match K")
        w16 = np.empty((N, K), dtype=np.float16)
        rc = self.lib.oracle_unpack_f16(pn_type, W.ctypes.data, N, K, w16.view(np.uint16).ctypes.data)
        if rc:
            raise ValueError(f"oracle_unpack_f16 failed ({rc})")
        return w16

    def gemm_f16(self, w16: np.ndarray, x: np.ndarray, want_abs: bool = True):
        """y[M][N] = x w16^T in fp64, rounded to fp32; also sum |w x| if asked."""
        w16 = np.ascontiguousarray(w16, dtype=np.float16)
        x = np.ascontiguousarray(x, dtype=np.float16)
        if x.ndim == 1:
            x = x[None, :]
        (N, K), M = w16.shape, x.shape[0]
        if x.shape[1] != K:
            raise ValueError("shape mismatch")
        y = np.empty((M, N), dtype=np.float32)
        a = np.empty((M, N), dtype=np.float64) if want_abs else None
        rc = self.lib.oracle_gemm_f16(w16.view(np.uint16).ctypes.data, N, K, x.view(np.uint16).ctypes.data,
                                      M, y.ctypes.data, a.ctypes.data if want_abs else None)
        if rc:
            raise ValueError(f"oracle_gemm_f16 failed ({rc})")
        return (y, a) if want_abs else y

    def gptq(self, pn_type: int, w: np.ndarray, X: np.ndarray, damp: float = 0.01) -> np.ndarray:
        """GPTQ-style quantisation (reading R12) of fp32 weights [N][K] with
        calibration inputs X [n][K]: PN bytes [N][row_bytes]."""
        w = np.ascontiguousarray(w, dtype=np.float32)
        X = np.ascontiguousarray(X, dtype=np.float32)
        N, K = w.shape
        if X.ndim != 2 or X.shape[1] != K:
            raise ValueError("calibration inputs must be [n][K]")
        out = np.zeros((N, self.row_bytes(pn_type, K)), dtype=np.uint8)
        rc = self.lib.oracle_gptq(pn_type, w.ctypes.data, N, K, X.ctypes.data, X.shape[0], float(damp),
                                  out.ctypes.data)
        if rc:
            raise ValueError(f"oracle_gptq failed ({rc})")
        return out

    def half_to_float(self, h: int) -> float:
        return float(self.lib.oracle_half_to_float(h))

    def float_to_half(self, f: float) -> int:
        return int(self.lib.oracle_float_to_half(f))


def default() -> Oracle:
    return Oracle()
