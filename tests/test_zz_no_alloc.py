"""moe_forward_static_ws: the layer for callers that cannot allocate device
memory (its scratch is the library's fixed device array).  Checked through the
C ABI against the ordinary moe_forward, on two calls in a row.  This file is
collected last on purpose."""
import ctypes

import numpy as np
import pytest
import torch

from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import forward, pack_layer, workspace
from parity import check_close

pytestmark = pytest.mark.gpu

CASES = [
    (synth.WORKLOADS["tiny"], 4),
    (synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e64", n_experts=64), 5),
    (synth.small_variant(synth.WORKLOADS["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32,
                         ff=512, shared_ff=512), 8),
]


FLAGS = [0, moe.MOE_FLAG_STATIC_WEIGHTS, moe.MOE_FLAG_DETERMINISTIC]


@pytest.mark.parametrize("flags", FLAGS, ids=["default", "static_weights", "deterministic"])
@pytest.mark.parametrize("wl,T", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_static_workspace_matches_moe_forward_twice(wl, T, flags):
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl, flags)
    if moe.moe_workspace_bytes(cfg, T) > moe.MOE_STATIC_WS_BYTES:
        pytest.skip("this call needs more scratch than the fixed array holds")
    ws = workspace(cfg, T)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for call in range(2):            # two calls in a row share the array
        x = synth.hidden_states(wl, T, seed=call).cuda()
        ref32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
        ref = forward(pl, x, ws, y_f32=ref32, cfg=cfg)
        y = torch.full((T, wl.hidden), float("nan"), dtype=torch.bfloat16, device="cuda")
        y32 = torch.full((T, wl.hidden), float("nan"), dtype=torch.float32, device="cuda")
        st.fill_(-1)
        moe.moe_forward_static_ws(cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, T, y, y32, st)
        torch.cuda.synchronize()
        assert int(st.item()) == moe.MOE_OK
        check_close(y32.cpu().numpy(), ref32.cpu().numpy(), what="y_f32 call %d" % call)
        check_close(y.float().cpu().numpy(), ref.float().cpu().numpy(), what="y call %d" % call)


def test_static_workspace_rejects_calls_beyond_its_size():
    wl = synth.WORKLOADS["qwen_prefill"]
    cfg = moe.config_for(wl)
    assert moe.moe_workspace_bytes(cfg, 4096) > moe.MOE_STATIC_WS_BYTES
    x = torch.zeros(4096, wl.hidden, dtype=torch.bfloat16, device="cuda")
    y = torch.empty_like(x)
    wr = torch.zeros(wl.n_experts, wl.hidden, dtype=torch.float32, device="cuda")
    table = torch.zeros(wl.n_experts, dtype=torch.int64, device="cuda")
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward_static_ws(cfg, x, wr, None, table, None, 4096, y)
    assert err.value.status == moe.MOE_ERR_WORKSPACE_TOO_SMALL


def test_static_workspace_reports_device_faults():
    wl = synth.WORKLOADS["tiny"]
    pl = pack_layer(wl, gen_device="cpu")
    x = synth.hidden_states(wl, 4).cuda()
    x[1, 3] = float("nan")
    y = torch.empty(4, wl.hidden, dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_forward_static_ws(pl.cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, 4, y, None, st)
    assert int(st.item()) == moe.MOE_ERR_DEVICE_FAULT
    # the next call starts from a cleared status word
    x = synth.hidden_states(wl, 4).cuda()
    moe.moe_forward_static_ws(pl.cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, 4, y, None, st)
    assert int(st.item()) == moe.MOE_OK


def test_static_workspace_fits_decode_windows_with_default_flags():
    """4 MiB holds every decode window (T <= 8) of both full layer shapes with
    the default flags."""
    for wl in (synth.WORKLOADS["qwen_decode"], synth.WORKLOADS["deepseek_decode"]):
        for T in range(1, 9):
            assert moe.moe_workspace_bytes(moe.config_for(wl), T) <= moe.MOE_STATIC_WS_BYTES, (wl.name, T)


def test_static_workspace_status_word_rules():
    """T == 0 writes MOE_OK; a rejected call leaves the caller's status word as it was."""
    wl = synth.WORKLOADS["tiny"]
    pl = pack_layer(wl, gen_device="cpu")
    x = synth.hidden_states(wl, 4).cuda()
    x[1, 3] = float("nan")
    y = torch.empty(4, wl.hidden, dtype=torch.bfloat16, device="cuda")
    st = torch.full((1,), 99, dtype=torch.int32, device="cuda")
    moe.moe_forward_static_ws(pl.cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, 0, y, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == moe.MOE_OK
    moe.moe_forward_static_ws(pl.cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, 4, y, None, st)
    torch.cuda.synchronize()
    assert int(st.item()) == moe.MOE_ERR_DEVICE_FAULT
    cfg = pl.cfg
    rc = moe.lib().moe_forward_static_ws(ctypes.byref(cfg), x.data_ptr(), pl.router_w.data_ptr(), None, None, None,
                                         4, y.data_ptr(), None, st.data_ptr(), None)   # null expert table
    assert rc == moe.MOE_ERR_INVALID_ARG
    torch.cuda.synchronize()
    assert int(st.item()) == moe.MOE_ERR_DEVICE_FAULT     # still the earlier call's status
