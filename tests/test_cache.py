"""The expert cache's host-side bookkeeping (moe_cache_plan), on the CPU: no
CUDA call is made by create / plan / destroy.  Fake, aligned addresses stand
in for the pinned host copies and the device slots (nothing dereferences
them here)."""
import ctypes

import pytest

from quantized_moe_expert_04_b300 import moe

BLOB = 4096
HOST0, SLOT0 = 0x10000000, 0x80000000


def _make(E, n_slots, host=None):
    L = moe.lib()
    host = host or [HOST0 + e * BLOB for e in range(E)]
    arr = (ctypes.c_void_p * E)(*host)
    h = ctypes.c_void_p()
    st = L.moe_cache_create(E, BLOB, ctypes.cast(arr, ctypes.c_void_p), ctypes.c_void_p(SLOT0) if n_slots else None,
                            n_slots, ctypes.byref(h))
    return st, h


def _plan(h, E, ids):
    L = moe.lib()
    a = (ctypes.c_int32 * max(1, len(ids)))(*ids)
    t = (ctypes.c_void_p * E)()
    n = ctypes.c_int32(-1)
    st = L.moe_cache_plan(h, ctypes.cast(a, ctypes.c_void_p), len(ids), ctypes.cast(t, ctypes.c_void_p),
                          ctypes.byref(n))
    return st, [t[i] or 0 for i in range(E)], n.value


def _stats(h):
    out = (ctypes.c_int64 * 4)()
    assert moe.lib().moe_cache_stats(h, ctypes.cast(out, ctypes.c_void_p)) == moe.MOE_OK
    return list(out)


def test_create_checks_arguments():
    assert _make(4, 2, host=[HOST0, HOST0 + 8, HOST0 + 16, HOST0 + 32])[0] == moe.MOE_ERR_MISALIGNED
    assert _make(0, 2)[0] == moe.MOE_ERR_INVALID_ARG
    st, h = _make(4, 0)                 # no slots: everything stays in host memory
    assert st == moe.MOE_OK
    st, table, n = _plan(h, 4, [1, 3, 3])
    assert st == moe.MOE_OK and n == 0 and table == [HOST0 + e * BLOB for e in range(4)]
    assert _stats(h) == [0, 2, 0, 0]
    moe.lib().moe_cache_destroy(h)
    moe.lib().moe_cache_destroy(None)


def test_plan_assigns_slots_and_keeps_host_addresses_until_filled():
    E = 6
    st, h = _make(E, 2)
    assert st == moe.MOE_OK
    st, table, n = _plan(h, E, [4, 1, 4])          # two distinct misses, two free slots
    assert st == moe.MOE_OK and n == 2
    host = [HOST0 + e * BLOB for e in range(E)]
    # the missed experts point at the slots their fills will fill, the others at host memory
    assert table[4] == SLOT0 and table[1] == SLOT0 + BLOB
    assert [table[e] for e in (0, 2, 3, 5)] == [host[e] for e in (0, 2, 3, 5)]
    st, table2, n = _plan(h, E, [4, 1, 2])         # 4 and 1 keep their planned slots; 2 finds none
    assert n == 0 and table2[4] == SLOT0 and table2[1] == SLOT0 + BLOB and table2[2] == host[2]
    assert _stats(h)[:3] == [0, 5, 0]              # nothing issued: every selection is still a miss
    assert _plan(h, E, [6])[0] == moe.MOE_ERR_INVALID_ARG
    assert _plan(h, E, [-1])[0] == moe.MOE_ERR_INVALID_ARG
    moe.lib().moe_cache_destroy(h)
