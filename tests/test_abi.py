"""The C-ABI library loads, exports every entry point include/moe.h declares,
and rejects bad arguments on the host (no GPU needed: these checks run before
any CUDA call)."""
import ctypes
import os
import re

import pytest

from quantized_moe_expert_04_b300 import moe

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _declared():
    names = set()
    for fn in os.listdir(os.path.join(ROOT, "include")):
        if fn.endswith(".h"):
            text = open(os.path.join(ROOT, "include", fn)).read()
            names |= set(re.findall(r"^MOE_API\s+[\w\s\*]*?\b(moe_\w+)\s*\(", text, re.M))
    return names


def test_library_exports_every_declared_symbol():
    declared = _declared()
    assert len(declared) >= 15
    L = moe.lib()
    for name in sorted(declared):
        assert hasattr(L, name), name
    assert declared == set(moe.EXPORTS)


def test_sizes():
    assert moe.moe_q4k_bytes(320, 2560) == 460800
    assert moe.moe_q4k_bytes(1, 255) == 0
    assert moe.moe_q8_0_bytes(2048, 4096) == 2048 * 128 * 34
    qwen = moe.make_config(2560, 512, 320, 10)
    assert moe.moe_expert_bytes(qwen) == 1382400          # the pages' per-expert blob
    ds = moe.make_config(4096, 256, 2048, 6, moe.MOE_SCORE_SIGMOID_BIAS, 2048)
    assert moe.moe_expert_bytes(ds) == 3 * 2048 * 16 * 144
    assert moe.moe_shared_bytes(ds) == 3 * 2048 * 128 * 34
    assert moe.moe_shared_bytes(qwen) == 0
    assert moe.moe_workspace_bytes(qwen, 5) > 0
    assert moe.moe_workspace_bytes(moe.make_config(2560, 512, 320, 10, 7), 5) == 0   # bad score_fn
    assert moe.moe_workspace_bytes(moe.make_config(2500, 512, 320, 10), 5) == 0     # H % 256
    assert moe.moe_workspace_bytes(moe.make_config(2560, 512, 300, 10), 5) == 0     # FF % 64
    assert moe.moe_workspace_bytes(moe.make_config(256, 4, 64, 5), 5) == 0          # k > E
    # Q5_K experts: 176 bytes a 256-weight block
    assert moe.moe_q5k_bytes(320, 2560) == 320 * 10 * 176
    assert moe.moe_q5k_bytes(1, 255) == 0
    qwen5 = moe.make_config(2560, 512, 320, 10, codec=moe.MOE_CODEC_Q5K)
    assert moe.moe_expert_bytes(qwen5) == 3 * 320 * 10 * 176
    assert moe.moe_expert_bytes(moe.make_config(2560, 512, 320, 10, codec=2)) == 0    # unknown codec
    assert moe.moe_workspace_bytes(moe.make_config(2560, 512, 320, 10, codec=-1), 5) == 0


def test_host_checks_reject_before_launch():
    L = moe.lib()
    p = ctypes.c_void_p(4096)           # never dereferenced: checks fail first
    assert L.moe_pack_q4k(p, 4, 100, p, None, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_pack_q4k(p, -1, 256, p, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_q4k(None, 4, 256, p, None, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_pack_q4k(ctypes.c_void_p(4100), 4, 256, p, None, None) == moe.MOE_ERR_MISALIGNED
    assert L.moe_pack_q8_0(p, 4, 48, p, None, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    cfg = moe.make_config(256, 16, 128, 2)
    need = moe.moe_workspace_bytes(cfg, 4)
    args = (ctypes.byref(cfg), p, p, None, 4, p, p, p, p, p)
    assert L.moe_route(*args, need - 1, None) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert L.moe_route(ctypes.byref(cfg), p, p, None, -1, p, p, p, p, p, need, None) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward(ctypes.byref(cfg), ctypes.c_void_p(4098), p, None, p, None, 4, p, None, p, need,
                         None) == moe.MOE_ERR_MISALIGNED
    assert L.moe_forward(ctypes.byref(cfg), p, p, None, None, None, 4, p, None, p, need,
                         None) == moe.MOE_ERR_INVALID_ARG
    bad = moe.make_config(256, 16, 128, 2, 5)
    assert L.moe_forward(ctypes.byref(bad), p, p, None, p, None, 4, p, None, p, need, None) == moe.MOE_ERR_INVALID_ARG
    odd = moe.make_config(320, 16, 128, 2)
    assert L.moe_forward(ctypes.byref(odd), p, p, None, p, None, 4, p, None, p, need,
                         None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    ds = moe.make_config(256, 16, 128, 2, moe.MOE_SCORE_SIGMOID_BIAS, 64)
    need_ds = moe.moe_workspace_bytes(ds, 4)
    assert L.moe_forward(ctypes.byref(ds), p, p, None, p, None, 4, p, None, p, need_ds,
                         None) == moe.MOE_ERR_INVALID_ARG     # shared expert without its blob
    # unknown codec; Q5_K experts off the decode path (a window above 8 tokens, or
    # the tensor-core path forced)
    bad_codec = moe.make_config(256, 16, 128, 2, codec=3)
    assert L.moe_forward(ctypes.byref(bad_codec), p, p, None, p, None, 4, p, None, p, need,
                         None) == moe.MOE_ERR_INVALID_ARG
    q5 = moe.make_config(256, 16, 128, 2, codec=moe.MOE_CODEC_Q5K)
    need40 = moe.moe_workspace_bytes(q5, 40)
    assert L.moe_forward(ctypes.byref(q5), p, p, None, p, None, 40, p, None, p, need40,
                         None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    q5g = moe.make_config(256, 16, 128, 2, flags=moe.MOE_FLAG_FORCE_GEMM, codec=moe.MOE_CODEC_Q5K)
    assert L.moe_forward(ctypes.byref(q5g), p, p, None, p, None, 4, p, None, p, moe.moe_workspace_bytes(q5g, 4),
                         None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_pack_q5k(p, 4, 100, p, None, None) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    assert L.moe_pack_q5k(ctypes.c_void_p(4100), 4, 256, p, None, None) == moe.MOE_ERR_MISALIGNED
    # T = 0 is a no-op success
    assert L.moe_forward(ctypes.byref(cfg), None, None, None, None, None, 0, None, None, p, need, None) == 0


def test_status_strings():
    for code in range(8):
        assert moe.status_string(code) and moe.status_string(code) != "unknown status"


def test_static_ws_checks_arguments_before_any_cuda_call():
    """moe_forward_static_ws rejects bad arguments on the host before it
    looks up or clears its device array (no GPU in this process)."""
    L = moe.lib()
    p = ctypes.c_void_p(4096)
    cfg = moe.make_config(256, 16, 128, 2)
    args = lambda **kw: [ctypes.byref(kw.get("cfg", cfg)), kw.get("x", p), p, None, kw.get("table", p), None,
                         kw.get("T", 4), kw.get("y", p), None, kw.get("st", None), None]
    assert L.moe_forward_static_ws(*args(y=None)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_static_ws(*args(table=None)) == moe.MOE_ERR_INVALID_ARG
    assert L.moe_forward_static_ws(*args(x=ctypes.c_void_p(4098))) == moe.MOE_ERR_MISALIGNED
    assert L.moe_forward_static_ws(*args(y=ctypes.c_void_p(4100))) == moe.MOE_ERR_MISALIGNED
    assert L.moe_forward_static_ws(*args(st=ctypes.c_void_p(4098))) == moe.MOE_ERR_MISALIGNED
    assert L.moe_forward_static_ws(*args(T=-1)) == moe.MOE_ERR_INVALID_ARG
    gemv = moe.make_config(256, 16, 128, 2, flags=moe.MOE_FLAG_FORCE_GEMV)
    assert L.moe_forward_static_ws(*args(cfg=gemv, T=9)) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    big = moe.make_config(2560, 512, 320, 10)
    assert L.moe_forward_static_ws(*args(cfg=big, T=4096)) == moe.MOE_ERR_WORKSPACE_TOO_SMALL


def test_stack_checks_arguments_before_any_cuda_call():
    """moe_forward_stack rejects bad arguments and unsupported shapes on the
    host (no GPU in this process)."""
    L = moe.lib()
    p = ctypes.c_void_p(4096)
    cfg = moe.make_config(256, 16, 128, 2)
    need = moe.moe_workspace_bytes(cfg, 4)

    def call(c=cfg, n=2, x=p, wr=p, blobs=p, shared=None, T=4, y=p, y32=None, ws=p, nbytes=need):
        return L.moe_forward_stack(ctypes.byref(c), n, x, wr, None, blobs, shared, T, y, y32, ws, nbytes, None)

    assert call(n=0) == moe.MOE_OK and call(T=0) == moe.MOE_OK            # no-ops
    assert call(n=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(T=-1) == moe.MOE_ERR_INVALID_ARG
    assert call(y=None) == moe.MOE_ERR_INVALID_ARG
    assert call(wr=None) == moe.MOE_ERR_INVALID_ARG
    assert call(x=ctypes.c_void_p(4098)) == moe.MOE_ERR_MISALIGNED
    assert call(wr=ctypes.c_void_p(4100)) == moe.MOE_ERR_MISALIGNED
    assert call(nbytes=need - 1) == moe.MOE_ERR_WORKSPACE_TOO_SMALL
    assert call(T=9, nbytes=moe.moe_workspace_bytes(cfg, 9)) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    for fl in (moe.MOE_FLAG_FORCE_GEMM, moe.MOE_FLAG_DETERMINISTIC):
        c = moe.make_config(256, 16, 128, 2, flags=fl)
        assert call(c=c, nbytes=moe.moe_workspace_bytes(c, 4)) == moe.MOE_ERR_UNSUPPORTED_SHAPE
    ds = moe.make_config(256, 16, 128, 2, moe.MOE_SCORE_SIGMOID_BIAS, 64)
    assert call(c=ds, nbytes=moe.moe_workspace_bytes(ds, 4)) == moe.MOE_ERR_INVALID_ARG   # no shared table


def test_debug_hooks_check_their_values_on_the_host():
    """moe_debug_set touches host state only: each skip hook takes -1 .. 2^20
    and rejects the rest; the wait limit takes any value >= 0."""
    for what in (moe.MOE_DEBUG_SKIP_COPY, moe.MOE_DEBUG_SKIP_ROUTER):
        for bad in (-2, (1 << 20) + 1):
            with pytest.raises(moe.MoeError):
                moe.moe_debug_set(what, bad)
        moe.moe_debug_set(what, 7)
        moe.moe_debug_set(what, -1)
    with pytest.raises(moe.MoeError):
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, -1)
    moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_debug_set(4, 0)
