"""Python binding of libmoe.so -- argument marshalling only.

Every entry point here has the name of the C function it calls (include/moe.h)
and takes torch tensors that live on the GPU; the work itself runs in the
library's CUDA kernels.  PyTorch provides device memory and streams, nothing
else.  If the library has not been built the first call raises: there is no
fallback.
"""
import ctypes
import os
from typing import Optional

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libmoe.so")

MOE_OK = 0
MOE_ERR_INVALID_ARG = 1
MOE_ERR_UNSUPPORTED_SHAPE = 2
MOE_ERR_MISALIGNED = 3
MOE_ERR_WORKSPACE_TOO_SMALL = 4
MOE_ERR_CUDA = 5
MOE_ERR_TIMEOUT = 6
MOE_ERR_DEVICE_FAULT = 7

MOE_SCORE_SOFTMAX = 0
MOE_SCORE_SIGMOID_BIAS = 1

MOE_CODEC_Q4K = 0
MOE_CODEC_Q5K = 1

MOE_FLAG_DETERMINISTIC = 1
MOE_FLAG_FORCE_GEMV = 2
MOE_FLAG_FORCE_GEMM = 4
MOE_FLAG_STATIC_WEIGHTS = 8
MOE_FLAG_RESIDUAL = 16

EXPORTS = (
    "moe_q4k_bytes", "moe_q5k_bytes", "moe_q8_0_bytes", "moe_expert_bytes", "moe_shared_bytes",
    "moe_pack_q4k", "moe_pack_q5k", "moe_pack_q8_0", "moe_dequant_q4k", "moe_dequant_q8_0",
    "moe_workspace_bytes", "moe_workspace_init", "moe_route", "moe_forward",
    "moe_workspace_routing", "moe_last_device_status", "moe_status_string",
    "moe_profile_enable", "moe_profile_read", "moe_forward_static_ws",
    "moe_dequant_q4k_f16", "moe_dequant_q8_0_f16", "moe_debug_set",
    "moe_dequant_q5k", "moe_dequant_q5k_f16", "moe_forward_stack",
    "moe_cache_create", "moe_cache_destroy", "moe_cache_plan", "moe_cache_issue", "moe_cache_poll",
    "moe_cache_stats", "moe_host_address",
)

MOE_DEBUG_WAIT_CYCLES = 1
MOE_DEBUG_SKIP_COPY = 2
MOE_DEBUG_SKIP_ROUTER = 3

MOE_STATIC_WS_BYTES = 4 << 20


class moe_profile_entry(ctypes.Structure):
    _fields_ = [("name", ctypes.c_char_p), ("launches", ctypes.c_int64), ("timed", ctypes.c_int64),
                ("total_ms", ctypes.c_double)]


class MoeError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__("%s: %s (status %d)" % (where, status_string(status), status))


class moe_config(ctypes.Structure):
    _fields_ = [("hidden", ctypes.c_int32), ("n_experts", ctypes.c_int32), ("ff", ctypes.c_int32),
                ("top_k", ctypes.c_int32), ("score_fn", ctypes.c_int32), ("shared_ff", ctypes.c_int32),
                ("flags", ctypes.c_int32), ("codec", ctypes.c_int32)]


def make_config(hidden, n_experts, ff, top_k, score_fn=MOE_SCORE_SOFTMAX, shared_ff=0, flags=0,
                codec=MOE_CODEC_Q4K) -> moe_config:
    return moe_config(hidden, n_experts, ff, top_k, score_fn, shared_ff, flags, codec)


def config_for(wl, flags: int = 0) -> moe_config:
    """moe_config of a synthetic workload (quantized_moe_expert_04_b300.synth.Workload)."""
    return make_config(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, wl.shared_ff, flags, wl.codec)


_lib = None
_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_SZ = ctypes.c_size_t
_CFG = ctypes.POINTER(moe_config)


def lib() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libmoe.so is not built (%s); run: python -m quantized_moe_expert_04_b300.build"
                               % LIB_PATH)
        L = ctypes.CDLL(LIB_PATH)
        sig = {
            "moe_q4k_bytes": (_SZ, [_I64, _I64]),
            "moe_q5k_bytes": (_SZ, [_I64, _I64]),
            "moe_q8_0_bytes": (_SZ, [_I64, _I64]),
            "moe_expert_bytes": (_SZ, [_CFG]),
            "moe_shared_bytes": (_SZ, [_CFG]),
            "moe_pack_q4k": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
            "moe_pack_q5k": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
            "moe_pack_q8_0": (ctypes.c_int, [_P, _I64, _I64, _P, _P, _P]),
            "moe_dequant_q4k": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
            "moe_dequant_q8_0": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
            "moe_dequant_q4k_f16": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
            "moe_dequant_q5k": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
            "moe_forward_stack": (ctypes.c_int, [_CFG, _I32, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
            "moe_dequant_q5k_f16": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
            "moe_dequant_q8_0_f16": (ctypes.c_int, [_P, _I64, _I64, _P, _P]),
            "moe_workspace_bytes": (_SZ, [_CFG, _I32]),
            "moe_workspace_init": (ctypes.c_int, [_P, _SZ, _P]),
            "moe_route": (ctypes.c_int, [_CFG, _P, _P, _P, _I32, _P, _P, _P, _P, _P, _SZ, _P]),
            "moe_forward": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _SZ, _P]),
            "moe_workspace_routing": (ctypes.c_int, [_CFG, _I32, _P, _SZ, ctypes.POINTER(_P), ctypes.POINTER(_P),
                                                     ctypes.POINTER(_P), ctypes.POINTER(_P)]),
            "moe_last_device_status": (ctypes.c_int, [_P, _P]),
            "moe_status_string": (ctypes.c_char_p, [ctypes.c_int]),
            "moe_profile_enable": (ctypes.c_int, [_I32]),
            "moe_debug_set": (ctypes.c_int, [_I32, _I64]),
            "moe_forward_static_ws": (ctypes.c_int, [_CFG, _P, _P, _P, _P, _P, _I32, _P, _P, _P, _P]),
            "moe_profile_read": (_I32, [ctypes.POINTER(moe_profile_entry), _I32]),
            "moe_cache_create": (ctypes.c_int, [_I32, _I64, _P, _P, _I32, ctypes.POINTER(_P)]),
            "moe_cache_destroy": (None, [_P]),
            "moe_cache_plan": (ctypes.c_int, [_P, _P, _I32, _P, ctypes.POINTER(_I32)]),
            "moe_cache_issue": (ctypes.c_int, [_P, _P, _P]),
            "moe_cache_poll": (ctypes.c_int, [_P]),
            "moe_cache_stats": (ctypes.c_int, [_P, _P]),
            "moe_host_address": (ctypes.c_int, [_P, ctypes.POINTER(_P)]),
        }
        for name, (res, args) in sig.items():
            fn = getattr(L, name)
            fn.restype = res
            fn.argtypes = args
        _lib = L
    return _lib


def status_string(status: int) -> str:
    try:
        return lib().moe_status_string(int(status)).decode()
    except Exception:   # library missing: still describe the code
        return "status %d" % status


def _check(status: int, where: str):
    if status != MOE_OK:
        raise MoeError(status, where)


def _ptr(t: Optional[torch.Tensor]):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError("expected a contiguous tensor")
    return ctypes.c_void_p(t.data_ptr())


def _stream(stream: Optional[torch.cuda.Stream]):
    s = stream if stream is not None else torch.cuda.current_stream()
    return ctypes.c_void_p(s.cuda_stream)


def _bf16_bits(x: torch.Tensor) -> torch.Tensor:
    if x.dtype == torch.bfloat16:
        return x
    if x.dtype in (torch.int16, torch.uint16):
        return x
    raise ValueError("hidden states must be bf16")


# ---------------------------------------------------------------- sizes

def moe_q4k_bytes(rows: int, cols: int) -> int:
    return int(lib().moe_q4k_bytes(rows, cols))


def moe_q5k_bytes(rows: int, cols: int) -> int:
    return int(lib().moe_q5k_bytes(rows, cols))


def moe_q8_0_bytes(rows: int, cols: int) -> int:
    return int(lib().moe_q8_0_bytes(rows, cols))


def moe_expert_bytes(cfg: moe_config) -> int:
    return int(lib().moe_expert_bytes(ctypes.byref(cfg)))


def moe_shared_bytes(cfg: moe_config) -> int:
    return int(lib().moe_shared_bytes(ctypes.byref(cfg)))


def moe_workspace_bytes(cfg: moe_config, max_tokens: int) -> int:
    return int(lib().moe_workspace_bytes(ctypes.byref(cfg), max_tokens))


# ---------------------------------------------------------------- packing

def moe_pack_q4k(w: torch.Tensor, out: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    assert w.dtype == torch.float32 and w.dim() == 2 and out.dtype == torch.uint8
    _check(lib().moe_pack_q4k(_ptr(w), w.shape[0], w.shape[1], _ptr(out), _ptr(dev_status), _stream(stream)),
           "moe_pack_q4k")
    return out


def moe_pack_q5k(w: torch.Tensor, out: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                 stream=None) -> torch.Tensor:
    assert w.dtype == torch.float32 and w.dim() == 2 and out.dtype == torch.uint8
    _check(lib().moe_pack_q5k(_ptr(w), w.shape[0], w.shape[1], _ptr(out), _ptr(dev_status), _stream(stream)),
           "moe_pack_q5k")
    return out


def moe_pack_q8_0(w: torch.Tensor, out: torch.Tensor, dev_status: Optional[torch.Tensor] = None,
                  stream=None) -> torch.Tensor:
    assert w.dtype == torch.float32 and w.dim() == 2 and out.dtype == torch.uint8
    _check(lib().moe_pack_q8_0(_ptr(w), w.shape[0], w.shape[1], _ptr(out), _ptr(dev_status), _stream(stream)),
           "moe_pack_q8_0")
    return out


def moe_dequant_q4k(blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    assert out.dtype == torch.float32 and out.numel() == rows * cols
    _check(lib().moe_dequant_q4k(_ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "moe_dequant_q4k")
    return out


def moe_dequant_q5k(blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    assert out.dtype == torch.float32 and out.numel() == rows * cols
    _check(lib().moe_dequant_q5k(_ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "moe_dequant_q5k")
    return out


def moe_dequant_q5k_f16(blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """fp16 operand weights (bit patterns in an int16/uint16 tensor) of a Q5_K matrix."""
    assert out.element_size() == 2 and out.numel() == rows * cols
    _check(lib().moe_dequant_q5k_f16(_ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "moe_dequant_q5k_f16")
    return out


def moe_dequant_q8_0(blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    assert out.dtype == torch.float32 and out.numel() == rows * cols
    _check(lib().moe_dequant_q8_0(_ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "moe_dequant_q8_0")
    return out


def moe_dequant_q4k_f16(blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    """fp16 operand weights (bit patterns in an int16/uint16 tensor) of a Q4_K matrix."""
    assert out.element_size() == 2 and out.numel() == rows * cols
    _check(lib().moe_dequant_q4k_f16(_ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "moe_dequant_q4k_f16")
    return out


def moe_dequant_q8_0_f16(blocks: torch.Tensor, rows: int, cols: int, out: torch.Tensor, stream=None) -> torch.Tensor:
    assert out.element_size() == 2 and out.numel() == rows * cols
    _check(lib().moe_dequant_q8_0_f16(_ptr(blocks), rows, cols, _ptr(out), _stream(stream)), "moe_dequant_q8_0_f16")
    return out


# ---------------------------------------------------------------- layer

def moe_workspace_init(ws: torch.Tensor, stream=None):
    _check(lib().moe_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "moe_workspace_init")


def moe_route(cfg: moe_config, x: torch.Tensor, router_w: torch.Tensor, router_bias: Optional[torch.Tensor],
              T: int, topk_ids: torch.Tensor, topk_w: torch.Tensor, expert_offsets: torch.Tensor,
              assign: torch.Tensor, ws: torch.Tensor, stream=None):
    x = _bf16_bits(x)
    _check(lib().moe_route(ctypes.byref(cfg), _ptr(x), _ptr(router_w), _ptr(router_bias), T, _ptr(topk_ids),
                           _ptr(topk_w), _ptr(expert_offsets), _ptr(assign), _ptr(ws),
                           ws.numel() * ws.element_size(), _stream(stream)), "moe_route")


def moe_forward(cfg: moe_config, x: torch.Tensor, router_w: torch.Tensor, router_bias: Optional[torch.Tensor],
                expert_blobs: torch.Tensor, shared_blob: Optional[torch.Tensor], T: int, y: torch.Tensor,
                y_f32: Optional[torch.Tensor], ws: torch.Tensor, stream=None):
    """expert_blobs: int64 CUDA tensor [E] of device pointers to the expert blobs."""
    x = _bf16_bits(x)
    _check(lib().moe_forward(ctypes.byref(cfg), _ptr(x), _ptr(router_w), _ptr(router_bias), _ptr(expert_blobs),
                             _ptr(shared_blob), T, _ptr(y), _ptr(y_f32), _ptr(ws),
                             ws.numel() * ws.element_size(), _stream(stream)), "moe_forward")


def moe_forward_stack(cfg: moe_config, n_layers: int, x: torch.Tensor, router_w: torch.Tensor,
                      router_bias: Optional[torch.Tensor], expert_blobs: torch.Tensor,
                      shared_blobs: Optional[torch.Tensor], T: int, y: torch.Tensor, y_f32: Optional[torch.Tensor],
                      ws: torch.Tensor, stream=None):
    """A window through n_layers layers in one launch.  x, y: bf16 [L][T][H]
    (with MOE_FLAG_RESIDUAL x[1:] is written); router_w, router_bias,
    shared_blobs: int64 CUDA tensors [L] of device pointers; expert_blobs:
    int64 CUDA tensor [L * E] of blob pointers."""
    x = _bf16_bits(x)
    _check(lib().moe_forward_stack(ctypes.byref(cfg), n_layers, _ptr(x), _ptr(router_w), _ptr(router_bias),
                                   _ptr(expert_blobs), _ptr(shared_blobs), T, _ptr(y), _ptr(y_f32), _ptr(ws),
                                   ws.numel() * ws.element_size(), _stream(stream)), "moe_forward_stack")


def moe_forward_static_ws(cfg: moe_config, x: torch.Tensor, router_w: torch.Tensor,
                          router_bias: Optional[torch.Tensor], expert_blobs: torch.Tensor,
                          shared_blob: Optional[torch.Tensor], T: int, y: torch.Tensor,
                          y_f32: Optional[torch.Tensor] = None, dev_status: Optional[torch.Tensor] = None,
                          stream=None):
    """moe_forward without a workspace, for callers that cannot allocate device
    memory: the scratch is the library's own fixed array (MOE_STATIC_WS_BYTES).
    Calls sharing a device must not overlap on the GPU."""
    x = _bf16_bits(x)
    _check(lib().moe_forward_static_ws(ctypes.byref(cfg), _ptr(x), _ptr(router_w), _ptr(router_bias),
                                       _ptr(expert_blobs), _ptr(shared_blob), T, _ptr(y), _ptr(y_f32),
                                       _ptr(dev_status), _stream(stream)), "moe_forward_static_ws")


def moe_workspace_routing(cfg: moe_config, T: int, ws: torch.Tensor):
    """Device addresses (ints) of ids, w, offsets and assign inside ws."""
    outs = [ctypes.c_void_p() for _ in range(4)]
    _check(lib().moe_workspace_routing(ctypes.byref(cfg), T, _ptr(ws), ws.numel() * ws.element_size(),
                                       *[ctypes.byref(o) for o in outs]), "moe_workspace_routing")
    return [o.value for o in outs]


def moe_last_device_status(ws: torch.Tensor, stream=None) -> int:
    return int(lib().moe_last_device_status(_ptr(ws), _stream(stream)))


# ---------------------------------------------------------------- diagnostics

def moe_debug_set(what: int, value: int):
    """Test hooks of the bounded device waits (see include/moe.h)."""
    _check(lib().moe_debug_set(int(what), int(value)), "moe_debug_set")


def moe_profile_enable(on: bool = True):
    _check(lib().moe_profile_enable(1 if on else 0), "moe_profile_enable")


def moe_profile_read():
    """{kernel name: (launches, timed launches, total ms)} since the last reset."""
    buf = (moe_profile_entry * 64)()
    n = lib().moe_profile_read(buf, 64)
    return {buf[i].name.decode(): (buf[i].launches, buf[i].timed, buf[i].total_ms) for i in range(n)}


# ---------------------------------------------------------------- host tier of the experts

def moe_host_address(host: torch.Tensor) -> int:
    """Device-usable address (int) of a pinned, mapped host tensor's first byte."""
    d = ctypes.c_void_p()
    _check(lib().moe_host_address(ctypes.c_void_p(host.data_ptr()), ctypes.byref(d)), "moe_host_address")
    return d.value


class ExpertCache:
    """The C library's device cache of expert blobs over pinned host memory
    (moe_cache_* in include/moe.h): marshalling only.

    host_blobs: device-usable addresses (ints) of the pinned, mapped host copies;
    slot_memory: a device tensor of n_slots * blob_bytes bytes (kept alive here)."""

    def __init__(self, n_experts: int, blob_bytes: int, host_blobs, slot_memory, n_slots: int):
        self.n_experts = int(n_experts)
        self._host = (ctypes.c_void_p * self.n_experts)(*[int(p) for p in host_blobs])
        self._slots = slot_memory
        self._table = (ctypes.c_void_p * self.n_experts)()
        h = ctypes.c_void_p()
        _check(lib().moe_cache_create(self.n_experts, int(blob_bytes), ctypes.cast(self._host, _P),
                                      _ptr(slot_memory) if n_slots else None, int(n_slots), ctypes.byref(h)),
               "moe_cache_create")
        self._h = h

    def plan(self, ids):
        """Host array of the window's expert ids -> (table as a list of ints, fills planned)."""
        arr = (ctypes.c_int32 * len(ids))(*[int(i) for i in ids])
        n = ctypes.c_int32()
        _check(lib().moe_cache_plan(self._h, ctypes.cast(arr, _P), len(ids), ctypes.cast(self._table, _P),
                                    ctypes.byref(n)), "moe_cache_plan")
        return [self._table[i] or 0 for i in range(self.n_experts)], n.value

    def issue(self, compute_stream=None, copy_stream=None):
        _check(lib().moe_cache_issue(self._h, _stream(compute_stream), _stream(copy_stream)), "moe_cache_issue")

    def poll(self):
        _check(lib().moe_cache_poll(self._h), "moe_cache_poll")

    def stats(self):
        out = (ctypes.c_int64 * 4)()
        _check(lib().moe_cache_stats(self._h, ctypes.cast(out, _P)), "moe_cache_stats")
        return {"hits": out[0], "misses": out[1], "fills": out[2], "bytes": out[3]}

    def close(self):
        if getattr(self, "_h", None):
            lib().moe_cache_destroy(self._h)
            self._h = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass
