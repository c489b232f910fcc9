"""A multi-token AVX2 CPU expert kernel (moe_avx2.c): a timed CPU baseline
beside the oracle, the kind of kernel the pages' CPU tier runs.  Only tests/
and bench.py's CPU legs use it; the product never does.  This module only
builds the library and marshals numpy arrays through ctypes."""
import ctypes
import os
import subprocess

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SRC = os.path.join(HERE, "moe_avx2.c")
LIB = os.path.join(HERE, "libmoe_avx2.so")
CFLAGS = ["-O3", "-std=c11", "-fPIC", "-shared", "-pthread", "-mavx2", "-mfma", "-mf16c", "-Wall", "-Wextra",
          "-Wno-unused-parameter"]

_lib = None


def build(force: bool = False) -> str:
    """Build the library if it is missing or older than its source; return its path."""
    if not force and os.path.exists(LIB) and os.path.getmtime(LIB) >= os.path.getmtime(SRC):
        return LIB
    tmp = LIB + ".tmp%d" % os.getpid()
    subprocess.run(["gcc", *CFLAGS, SRC, "-o", tmp, "-lm"], check=True)
    os.replace(tmp, LIB)
    return LIB


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        L = ctypes.CDLL(build())
        p, i32, i64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64
        L.cpu_moe_window.argtypes = [i32, i32, i32, i32, i64, p, p, p, p, i32, p]
        L.cpu_moe_window.restype = i32
        _lib = L
    return _lib


def moe_window(H, E, FF, k, x_bf16, ids, w, blobs, threads=1):
    """y fp32 [T][H] = sum of w[t][r] * FFN_{ids[t][r]}(x_t) over the window.

    x_bf16: uint16 [T][H]; ids: int32 [T][k]; w: float [T][k]; blobs: list of E
    uint8 arrays (Q4_K expert blobs) or None for experts no token selects."""
    x = np.ascontiguousarray(x_bf16, dtype=np.uint16)
    T = x.shape[0]
    ids = np.ascontiguousarray(ids, dtype=np.int32).reshape(T, k)
    w = np.ascontiguousarray(w, dtype=np.float32).reshape(T, k)
    keep = [np.ascontiguousarray(b, dtype=np.uint8) if b is not None else None for b in blobs]
    table = (ctypes.c_void_p * E)(*[b.ctypes.data if b is not None else None for b in keep])
    y = np.zeros((T, H), np.float32)
    rc = lib().cpu_moe_window(H, E, FF, k, T, x.ctypes.data, ids.ctypes.data, w.ctypes.data,
                              ctypes.cast(table, ctypes.c_void_p), int(threads), y.ctypes.data)
    if rc != 0:
        raise RuntimeError("cpu_moe_window: bad arguments or no AVX2/FMA on this CPU (%d)" % rc)
    return y
