"""A window through a stack of layers in one launch (moe_forward_stack).

Every layer must match the oracle on the input the kernel gave it.  With the
residual stream the kernel writes x[l + 1] = bf16(x[l] + y[l]) itself; that
sum is checked bit for bit here, and layer l + 1 is then checked against the
oracle on that x (so one layer's rounding never leaks into the next layer's
reference).  Without it every layer reads its own seeded input.  A grid
barrier that runs out must end the launch with MOE_ERR_TIMEOUT and leave the
context usable.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import LayerStack, pack_layer, routing_views, workspace
from parity import check_close, compare_ids, oracle_blobs, oracle_forward, oracle_inputs, selection_keys

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS
sv = synth.small_variant

QWEN_E64 = sv(W["qwen_decode"], name="qwen_e64", n_experts=64)
DS_SMALL = sv(W["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32, ff=512, shared_ff=512)


def _stack(wl, L, gen_device="cpu"):
    return LayerStack([pack_layer(wl, 0, l, gen_device=gen_device) for l in range(L)])


def _check_layer(wl, l, x_l, y32_l, gen_device="cpu"):
    """Layer l of the stack on input x_l (bf16 [T][H], CPU) against the oracle."""
    xb, wr, b = oracle_inputs(wl, x_l.shape[0], 0, l, gen_device=gen_device, x=x_l)
    oids, _, kth, nxt = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, sblob = oracle_blobs(wl, oids.reshape(-1), 0, l, gen_device=gen_device)
    ref = oracle_forward(wl, xb, wr, b, blobs, sblob)
    return check_close(y32_l.astype(np.float64), ref, what="layer %d" % l)


def _bf16_sum(a, b):
    """bf16(fp32(a) + fp32(b)): the residual stream's definition."""
    return (a.float() + b.float()).to(torch.bfloat16)


@pytest.mark.parametrize("wl,L,T", [(W["tiny"], 2, 4), (QWEN_E64, 3, 3), (QWEN_E64, 2, 1), (QWEN_E64, 2, 8),
                                    (DS_SMALL, 2, 4), (DS_SMALL, 3, 8),
                                    (sv(QWEN_E64, name="qwen_e64_q5k", codec=1), 2, 3),
                                    (sv(DS_SMALL, name="ds_small_q5k", codec=1), 2, 5)],
                         ids=lambda c: getattr(c, "name", str(c)))
def test_residual_stack_matches_the_oracle_layer_by_layer(wl, L, T):
    st = _stack(wl, L)
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    x = torch.zeros(L, T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    x[0] = synth.hidden_states(wl, T, 0, 0).cuda()
    y32 = torch.empty(L, T, wl.hidden, dtype=torch.float32, device="cuda")
    y = st.forward(x, ws, y_f32=y32, residual=True)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    xc, yc, y32c = x.cpu(), y.cpu(), y32.cpu().numpy()
    # y is the bf16 rounding of y_f32; the stream is bf16(x + y), bit for bit
    assert torch.equal(yc, torch.from_numpy(y32c).to(torch.bfloat16))
    for l in range(L - 1):
        assert torch.equal(xc[l + 1], _bf16_sum(xc[l], yc[l])), "residual stream differs after layer %d" % l
    for l in range(L):
        r = _check_layer(wl, l, xc[l], y32c[l])
        print("%s L=%d T=%d layer %d: rel-L2 %.2e" % (wl.name, L, T, l, r[0]))


@pytest.mark.parametrize("wl,L,T", [(QWEN_E64, 3, 5), (DS_SMALL, 2, 8)], ids=["qwen_e64", "ds_small"])
def test_independent_inputs_match_the_oracle(wl, L, T):
    st = _stack(wl, L)
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    xs = torch.stack([synth.hidden_states(wl, T, 0, l) for l in range(L)]).to(torch.bfloat16).cuda()
    x = xs.clone()
    y32 = torch.empty(L, T, wl.hidden, dtype=torch.float32, device="cuda")
    st.forward(x, ws, y_f32=y32, residual=False)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    assert torch.equal(x, xs)                       # inputs are not written without the residual flag
    for l in range(L):
        _check_layer(wl, l, xs[l].cpu(), y32[l].cpu().numpy())
    # the workspace's routing views hold the last layer's routing
    ids, _, _, _ = routing_views(cfg, T, ws)
    xb, wr, b = oracle_inputs(wl, T, 0, L - 1, x=xs[L - 1].cpu())
    oids, _, kth, nxt = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    compare_ids(ids.cpu().numpy(), oids, kth, nxt, keys_of=lambda t: selection_keys(xb[t], wr, b, wl.score_fn))


def test_full_size_residual_stack_qwen_decode():
    """The benchmark's launch configuration: qwen_decode, T = 3, 6 layers (the
    oracle checks the first two and the last one on the kernel's own inputs)."""
    wl, L, T = W["qwen_decode"], 6, 3
    st = _stack(wl, L, gen_device="cuda")
    ws = workspace(moe.config_for(wl), T)
    x = torch.zeros(L, T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    x[0] = synth.hidden_states(wl, T, 0, 0).cuda()
    y32 = torch.empty(L, T, wl.hidden, dtype=torch.float32, device="cuda")
    y = st.forward(x, ws, y_f32=y32, residual=True)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    xc, yc, y32c = x.cpu(), y.cpu(), y32.cpu().numpy()
    for l in range(L - 1):
        assert torch.equal(xc[l + 1], _bf16_sum(xc[l], yc[l]))
    for l in (0, 1, L - 1):
        _check_layer(wl, l, xc[l], y32c[l], gen_device="cuda")


def test_full_size_stack_deepseek_decode():
    wl, L, T = W["deepseek_decode"], 2, 8
    st = _stack(wl, L, gen_device="cuda")
    ws = workspace(moe.config_for(wl), T)
    x = torch.zeros(L, T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    x[0] = synth.hidden_states(wl, T, 0, 0).cuda()
    y32 = torch.empty(L, T, wl.hidden, dtype=torch.float32, device="cuda")
    st.forward(x, ws, y_f32=y32, residual=True)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    for l in range(L):
        _check_layer(wl, l, x[l].cpu(), y32[l].cpu().numpy(), gen_device="cuda")


@pytest.mark.parametrize("cta", [0, 5])
def test_grid_barrier_timeout_is_reported_and_the_context_survives(cta):
    """One CTA never arrives at the first grid barrier: every other CTA's wait
    runs out (bounded), the grid's abort word ends the rest, and the call
    reports MOE_ERR_TIMEOUT.  The next call, hooks cleared, is right."""
    wl, L, T = QWEN_E64, 2, 3
    st = _stack(wl, L)
    ws = workspace(moe.config_for(wl), T)
    x = torch.zeros(L, T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    x[0] = synth.hidden_states(wl, T, 0, 0).cuda()
    try:
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 1 << 22)      # ~2 ms
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, cta)
        st.forward(x, ws, residual=True)
        assert moe.moe_last_device_status(ws) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, -1)
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 0)
    y32 = torch.empty(L, T, wl.hidden, dtype=torch.float32, device="cuda")
    st.forward(x, ws, y_f32=y32, residual=True)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    _check_layer(wl, 0, x[0].cpu(), y32[0].cpu().numpy())
    _check_layer(wl, 1, x[1].cpu(), y32[1].cpu().numpy())
