"""CPU oracle for the sparse MoE layer over Q4_K experts -- TEST INFRASTRUCTURE.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product (the CUDA library and its
binding) never does, and this package imports nothing from the product.

The arithmetic lives in ``moe_oracle.c`` (plain C, fp64 FFN, fp32 IEEE
quantiser); this module only marshals numpy arrays through ctypes.  The
readings the oracle takes where the pages are silent are listed in the header
of ``moe_oracle.c`` (R1-R8).
"""
import ctypes
import os
from typing import Optional, Sequence, Tuple

import numpy as np

from . import build as _build

QK_K = 256
Q4K_BYTES = 144
Q5K_BYTES = 176
CODEC_Q4K = 0
CODEC_Q5K = 1
QK8 = 32
Q8_BYTES = 34
SCORE_SOFTMAX = 0
SCORE_SIGMOID_BIAS = 1

_lib = None
_p = ctypes.c_void_p
_i64 = ctypes.c_int64
_i32 = ctypes.c_int


def lib() -> ctypes.CDLL:
    """Load (building on first use) the oracle library."""
    global _lib
    if _lib is None:
        path = _build.build()
        L = ctypes.CDLL(path)
        L.orc_f32_to_f16.argtypes = [ctypes.c_float]
        L.orc_f32_to_f16.restype = ctypes.c_uint16
        L.orc_f16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_f16_to_f32.restype = ctypes.c_float
        L.orc_f64_to_f16.argtypes = [ctypes.c_double]
        L.orc_f64_to_f16.restype = ctypes.c_uint16
        for name in ("orc_q4k_dequantize_f16", "orc_q8_0_dequantize_f16"):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = None
        L.orc_bf16_to_f32.argtypes = [ctypes.c_uint16]
        L.orc_bf16_to_f32.restype = ctypes.c_float
        for name in ("orc_q4k_quantize", "orc_q8_0_quantize"):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = _i32
        for name in ("orc_q4k_dequantize", "orc_q8_0_dequantize"):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = None
        L.orc_route.argtypes = [_p, _p, _p, _i64, _i32, _i32, _i32, _i32, _p, _p, _p, _p, _p]
        L.orc_route.restype = _i32
        L.orc_bucket.argtypes = [_p, _i64, _i32, _i32, _p, _p, _p]
        L.orc_bucket.restype = _i32
        L.orc_moe_forward.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                      _p, _p, _p, _p, _p, _i64, _p, _p]
        L.orc_moe_forward.restype = _i32
        for name in ("orc_q5k_quantize",):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = _i32
        for name in ("orc_q5k_dequantize", "orc_q5k_dequantize_f16"):
            getattr(L, name).argtypes = [_p, _i64, _i64, _p]
            getattr(L, name).restype = None
        L.orc_moe_forward_codec.argtypes = [_i32, _i32, _i32, _i32, _i32, _i32, _i32,
                                            _p, _p, _p, _p, _p, _i64, _p, _i32, _p]
        L.orc_moe_forward_codec.restype = _i32
        L.orc_set_threads.argtypes = [_i32]
        L.orc_set_threads.restype = _i32
        _lib = L
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _c(a, dtype) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=dtype)


def set_threads(n: int = 0) -> int:
    """Set the OpenMP thread count (n <= 0 keeps the default); return the count in use."""
    return int(lib().orc_set_threads(int(n)))


# ---------------------------------------------------------------- scalars

def f32_to_f16_bits(v: float) -> int:
    return int(lib().orc_f32_to_f16(float(v)))


def f64_to_f16_bits(v: float) -> int:
    return int(lib().orc_f64_to_f16(float(v)))


def f16_bits_to_f32(b: int) -> float:
    return float(lib().orc_f16_to_f32(int(b)))


# ---------------------------------------------------------------- codecs

def q4k_quantize(w: np.ndarray) -> np.ndarray:
    """[rows, cols] fp32 -> [rows, cols/256*144] uint8 (raises on non-finite input)."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    out = np.zeros((rows, cols // QK_K * Q4K_BYTES), np.uint8)
    if lib().orc_q4k_quantize(_ptr(w), rows, cols, _ptr(out)) != 0:
        raise ValueError("q4k_quantize: bad shape or non-finite / out-of-range input")
    return out


def q4k_dequantize(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    blob = _c(blob, np.uint8)
    assert blob.size == rows * (cols // QK_K) * Q4K_BYTES
    out = np.empty((rows, cols), np.float32)
    lib().orc_q4k_dequantize(_ptr(blob), rows, cols, _ptr(out))
    return out


def q4k_dequantize_f16(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """The fp16 operand rounding of the Q4_K weights (R9): uint16 bit patterns [rows, cols]."""
    blob = _c(blob, np.uint8)
    assert blob.size == rows * (cols // QK_K) * Q4K_BYTES
    out = np.empty((rows, cols), np.uint16)
    lib().orc_q4k_dequantize_f16(_ptr(blob), rows, cols, _ptr(out))
    return out


def q8_0_dequantize_f16(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """fp16(d*q) of the Q8_0 weights (R9): uint16 bit patterns [rows, cols]."""
    blob = _c(blob, np.uint8)
    assert blob.size == rows * (cols // QK8) * Q8_BYTES
    out = np.empty((rows, cols), np.uint16)
    lib().orc_q8_0_dequantize_f16(_ptr(blob), rows, cols, _ptr(out))
    return out


def q5k_quantize(w: np.ndarray) -> np.ndarray:
    """[rows, cols] fp32 -> [rows, cols/256*176] uint8 Q5_K blocks (R10, R11)."""
    w = _c(w, np.float32)
    rows, cols = w.shape
    out = np.zeros((rows, cols // QK_K * Q5K_BYTES), np.uint8)
    if lib().orc_q5k_quantize(_ptr(w), rows, cols, _ptr(out)) != 0:
        raise ValueError("q5k_quantize: bad shape or non-finite / out-of-range input")
    return out


def q5k_dequantize(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    blob = _c(blob, np.uint8)
    assert blob.size == rows * (cols // QK_K) * Q5K_BYTES
    out = np.empty((rows, cols), np.float32)
    lib().orc_q5k_dequantize(_ptr(blob), rows, cols, _ptr(out))
    return out


def q5k_dequantize_f16(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    """The fp16 operand rounding (R9) of the Q5_K weights: uint16 bit patterns [rows, cols]."""
    blob = _c(blob, np.uint8)
    assert blob.size == rows * (cols // QK_K) * Q5K_BYTES
    out = np.empty((rows, cols), np.uint16)
    lib().orc_q5k_dequantize_f16(_ptr(blob), rows, cols, _ptr(out))
    return out


def q8_0_quantize(w: np.ndarray) -> np.ndarray:
    w = _c(w, np.float32)
    rows, cols = w.shape
    out = np.zeros((rows, cols // QK8 * Q8_BYTES), np.uint8)
    if lib().orc_q8_0_quantize(_ptr(w), rows, cols, _ptr(out)) != 0:
        raise ValueError("q8_0_quantize: bad shape or non-finite / out-of-range input")
    return out


def q8_0_dequantize(blob: np.ndarray, rows: int, cols: int) -> np.ndarray:
    blob = _c(blob, np.uint8)
    assert blob.size == rows * (cols // QK8) * Q8_BYTES
    out = np.empty((rows, cols), np.float32)
    lib().orc_q8_0_dequantize(_ptr(blob), rows, cols, _ptr(out))
    return out


def pack_expert_q4k(w3: np.ndarray) -> np.ndarray:
    """[3, FF, H] fp32 (gate, up, down stored [FF][H]) -> flat expert blob."""
    return np.concatenate([q4k_quantize(w3[m]).reshape(-1) for m in range(3)])


def pack_expert_q5k(w3: np.ndarray) -> np.ndarray:
    """[3, FF, H] fp32 -> flat Q5_K expert blob (same matrix order as Q4_K)."""
    return np.concatenate([q5k_quantize(w3[m]).reshape(-1) for m in range(3)])


def pack_expert(w3: np.ndarray, codec: int = CODEC_Q4K) -> np.ndarray:
    return pack_expert_q5k(w3) if codec == CODEC_Q5K else pack_expert_q4k(w3)


def pack_shared_q8_0(w3: np.ndarray) -> np.ndarray:
    return np.concatenate([q8_0_quantize(w3[m]).reshape(-1) for m in range(3)])


# ---------------------------------------------------------------- router

def route(x_bf16: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray], k: int,
          score_fn: int, forced_ids: Optional[np.ndarray] = None
          ) -> Tuple[np.ndarray, np.ndarray, np.ndarray, np.ndarray]:
    """Route tokens.  Returns (ids [T,k] int32, w [T,k] f64, kth_key [T], next_key [T])."""
    x = _c(x_bf16, np.uint16)
    wr = _c(wr, np.float32)
    T, H = x.shape
    E = wr.shape[0]
    b = None if bias is None else _c(bias, np.float32)
    f = None if forced_ids is None else _c(forced_ids, np.int32)
    ids = np.zeros((T, k), np.int32)
    w = np.zeros((T, k), np.float64)
    kth = np.zeros(T, np.float64)
    nxt = np.zeros(T, np.float64)
    rc = lib().orc_route(_ptr(x), _ptr(wr), _ptr(b), T, H, E, k, score_fn, _ptr(f),
                         _ptr(ids), _ptr(w), _ptr(kth), _ptr(nxt))
    if rc != 0:
        raise ValueError("route: bad arguments")
    return ids, w, kth, nxt


def bucket(ids: np.ndarray, n_experts: int) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Stable counting sort of the assignments.  Returns (counts, offsets, assign)."""
    ids = _c(ids, np.int32)
    T, k = ids.shape
    counts = np.zeros(n_experts, np.int32)
    offsets = np.zeros(n_experts + 1, np.int32)
    assign = np.zeros(T * k, np.int32)
    if lib().orc_bucket(_ptr(ids), T, k, n_experts, _ptr(counts), _ptr(offsets), _ptr(assign)) != 0:
        raise ValueError("bucket: id out of range")
    return counts, offsets, assign


# ---------------------------------------------------------------- layer

def moe_forward(hidden: int, n_experts: int, ff: int, top_k: int, score_fn: int,
                x_bf16: np.ndarray, wr: np.ndarray, bias: Optional[np.ndarray],
                blobs: Sequence[Optional[np.ndarray]], shared_ff: int = 0,
                shared_blob: Optional[np.ndarray] = None,
                forced_ids: Optional[np.ndarray] = None, codec: int = CODEC_Q4K) -> np.ndarray:
    """The whole layer in fp64.  ``blobs[e]`` is expert e's blob (or None if unused),
    Q4_K or (codec = CODEC_Q5K) Q5_K."""
    L = lib()
    x = _c(x_bf16, np.uint16)
    wr = _c(wr, np.float32)
    T = x.shape[0]
    assert x.shape[1] == hidden and wr.shape == (n_experts, hidden)
    b = None if bias is None else _c(bias, np.float32)
    keep = [None if bl is None else _c(bl, np.uint8) for bl in blobs]
    table = (ctypes.c_void_p * n_experts)(*[None if bl is None else bl.ctypes.data for bl in keep])
    sb = None if shared_blob is None else _c(shared_blob, np.uint8)
    f = None if forced_ids is None else _c(forced_ids, np.int32)
    y = np.zeros((T, hidden), np.float64)
    rc = L.orc_moe_forward_codec(hidden, n_experts, ff, top_k, score_fn, int(sb is not None), shared_ff,
                                 _ptr(x), _ptr(wr), _ptr(b), ctypes.cast(table, ctypes.c_void_p),
                                 _ptr(sb), T, _ptr(f), int(codec), _ptr(y))
    if rc != 0:
        raise ValueError("moe_forward failed (%d)" % rc)
    return y
