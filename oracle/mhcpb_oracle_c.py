"""ctypes front of the C oracle (oracle/mhcpb_oracle_c.c) -- TEST
INFRASTRUCTURE ONLY (tests, smoke and bench.py's CPU-baseline leg).

Same definition and rounding as ``oracle.mhcpb_oracle.mhc_proj_rms_backward``
(without the addend), in plain C loops over FP64 with OpenMP over rows: the
CPU baseline that bench.py times.  tests/test_oracle_c.py pins it to the numpy
oracle bit for bit."""
from __future__ import annotations

import ctypes
import os

import numpy as np

from .build_c import LIB, build

_lib = None


def load():
    global _lib
    if _lib is None:
        if not os.path.exists(LIB):
            build()
        lib = ctypes.CDLL(LIB)
        P = ctypes.c_void_p
        lib.mhcpb_oracle_backward.argtypes = [ctypes.c_int64, ctypes.c_int64, P, P, P, P, P, P, P,
                                              ctypes.c_int]
        lib.mhcpb_oracle_backward.restype = None
        _lib = lib
    return _lib


def mhc_proj_rms_backward(x_bits, w, grad_proj, grad_r, r, nthreads: int = 0):
    """(dx_bits uint16 [T, K], dw float32 [24, K]); nthreads 0: OpenMP's default."""
    x = np.ascontiguousarray(x_bits, dtype=np.uint16)
    T, K = x.shape
    w = np.ascontiguousarray(w, dtype=np.float32)
    gp = np.ascontiguousarray(grad_proj, dtype=np.float32)
    gr = np.ascontiguousarray(grad_r, dtype=np.float32)
    rr = np.ascontiguousarray(r, dtype=np.float32)
    dx = np.empty((T, K), dtype=np.uint16)
    dw = np.empty((24, K), dtype=np.float32)
    ptr = lambda a: a.ctypes.data_as(ctypes.c_void_p)  # noqa: E731
    load().mhcpb_oracle_backward(T, K, ptr(x), ptr(w), ptr(gp), ptr(gr), ptr(rr), ptr(dx), ptr(dw),
                                 int(nthreads))
    return dx, dw
