"""Failure detection on the GPU without a fault: a bounded wait that runs out.

moe_debug_set shortens every device wait and makes one CTA of the decode
layer kernel arm its prologue barrier without issuing the copy it waits for,
so the wait gives up.  The call
must end (no hang), report MOE_ERR_TIMEOUT through the workspace status word,
and leave the context usable: the next call, with the hooks cleared, matches
the oracle.  Nothing here faults, traps or spins without a limit.
"""
import numpy as np
import pytest
import torch

from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import forward, pack_layer, workspace
from parity import check_close, oracle_blobs, oracle_forward, oracle_inputs

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("cta", [0, 1, 7])
def test_decode_wait_timeout_is_reported_and_the_context_survives(cta):
    wl = synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e64", n_experts=64)
    T = 3
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMV)
    ws = workspace(cfg, T)
    x = synth.hidden_states(wl, T).cuda()
    try:
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 1 << 22)      # ~2 ms
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, cta)
        forward(pl, x, ws, cfg=cfg)
        assert moe.moe_last_device_status(ws) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, -1)
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 0)
    # the skip is one-shot and the context is intact: the next call is right
    y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
    forward(pl, x, ws, y_f32=y32, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    xb, wr, b = oracle_inputs(wl, T, x=x.cpu())
    import oracle
    ids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, sblob = oracle_blobs(wl, ids.reshape(-1))
    check_close(y32.cpu().numpy(), oracle_forward(wl, xb, wr, b, blobs, sblob))


def test_debug_hook_rejects_bad_values():
    with pytest.raises(moe.MoeError):
        moe.moe_debug_set(99, 0)
    with pytest.raises(moe.MoeError):
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, -5)
    with pytest.raises(moe.MoeError):
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, -2)


@pytest.mark.parametrize("cta", [0, 3])
def test_gemm_wait_timeout_is_reported_and_the_context_survives(cta):
    """The tensor-core path: one CTA of the routed gate/up GEMM arms a token-row
    copy it never issues; its MMA warp's wait runs out, every role of the CTA
    leaves its loop on the abort flag, in-flight copies and MMAs drain, and the
    tensor memory is freed.  The call reports MOE_ERR_TIMEOUT; the next one is
    right."""
    wl = synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e64", n_experts=64)
    T = 40
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMM)
    ws = workspace(cfg, T)
    x = synth.hidden_states(wl, T).cuda()
    try:
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 1 << 22)      # ~2 ms
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, cta)
        forward(pl, x, ws, cfg=cfg)
        assert moe.moe_last_device_status(ws) == moe.MOE_ERR_TIMEOUT
    finally:
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_COPY, -1)
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 0)
    y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
    forward(pl, x, ws, y_f32=y32, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    xb, wr, b = oracle_inputs(wl, T, x=x.cpu())
    import oracle
    ids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, sblob = oracle_blobs(wl, ids.reshape(-1))
    check_close(y32.cpu().numpy(), oracle_forward(wl, xb, wr, b, blobs, sblob))


@pytest.mark.parametrize("E,tile,times_out", [(64, 0, True), (64, 2, True), (128, 4, True), (128, 1000, False)])
def test_router_wait_timeout_is_reported_and_the_context_survives(E, tile, times_out):
    """The tensor-core router (T = 300: three 128-token tiles, the last one
    ragged; E = 128 adds a second expert tile): one tile never issues its first
    stage's copies, its MMA warp's wait runs out, the epilogue leaves on the
    abort flag without writing that tile's logits, and the call reports
    MOE_ERR_TIMEOUT (the routing that follows reads whatever the logits buffer
    held: ids stay in range whatever it holds).  A tile past the grid skips
    nothing.  Either way the hook is spent and the next call is right."""
    wl = synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e%d" % E, n_experts=E)
    T = 300
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    x = synth.hidden_states(wl, T).cuda()
    try:
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 1 << 22)      # ~2 ms
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_ROUTER, tile)
        forward(pl, x, ws, cfg=cfg)
        assert moe.moe_last_device_status(ws) == (moe.MOE_ERR_TIMEOUT if times_out else moe.MOE_OK)
    finally:
        moe.moe_debug_set(moe.MOE_DEBUG_SKIP_ROUTER, -1)
        moe.moe_debug_set(moe.MOE_DEBUG_WAIT_CYCLES, 0)
    y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
    forward(pl, x, ws, y_f32=y32, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    xb, wr, b = oracle_inputs(wl, T, x=x.cpu())
    import oracle
    ids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, sblob = oracle_blobs(wl, ids.reshape(-1))
    check_close(y32.cpu().numpy(), oracle_forward(wl, xb, wr, b, blobs, sblob))
