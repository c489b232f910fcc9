"""Host tier of the experts on the GPU: every expert in pinned host memory, a
device cache of some of them (moe_cache_*).  Experts outside the cache are read
by the layer kernels straight from host memory; the window's missed experts are
copied into device slots for the windows that follow.  Every window must match
the oracle whatever the cache holds; a repeated window must hit."""
import pytest
import torch

from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import TieredLayer, pack_layer, workspace
from parity import check_close, oracle_blobs, oracle_forward, oracle_inputs

pytestmark = pytest.mark.gpu

QWEN_E64 = synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e64", n_experts=64)
DS_SMALL = synth.small_variant(synth.WORKLOADS["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32,
                               ff=256, top_k=4, shared_ff=512)


def _oracle_y(wl, T, x):
    import oracle
    xb, wr, b = oracle_inputs(wl, T, x=x)
    ids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, sblob = oracle_blobs(wl, ids.reshape(-1))
    return oracle_forward(wl, xb, wr, b, blobs, sblob)


QWEN_E64_Q5K = synth.small_variant(QWEN_E64, name="qwen_e64_q5k", codec=1)


@pytest.mark.parametrize("wl,T,n_slots", [(QWEN_E64, 3, 40), (QWEN_E64, 5, 0), (DS_SMALL, 4, 10),
                                          (QWEN_E64_Q5K, 3, 30)],
                         ids=["qwen_e64-slots40", "qwen_e64-host-only", "ds_small-slots10", "qwen_e64_q5k-slots30"])
def test_tiered_layer_matches_the_oracle_and_fills_its_cache(wl, T, n_slots):
    pl = pack_layer(wl, gen_device="cpu")
    tl = TieredLayer(pl, n_slots)
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    windows = [0, 1, 0, 2, 1]                 # repeated windows: their experts were filled
    for win in windows:
        x = synth.hidden_states(wl, T, 0, win)
        y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
        tl.forward(x.cuda(), ws, y_f32=y32)
        assert moe.moe_last_device_status(ws) == moe.MOE_OK
        check_close(y32.cpu().numpy(), _oracle_y(wl, T, x))
        tl.copy_stream.synchronize()          # the fills of this window land before the next plan
    st = tl.stats()
    if n_slots == 0:
        assert st["hits"] == 0 and st["fills"] == 0 and st["misses"] > 0
    else:
        assert st["fills"] > 0 and st["bytes"] == st["fills"] * wl.blob_bytes
        assert st["hits"] > 0
    tl.cache.close()


def test_host_address_rejects_pageable_memory():
    t = torch.empty(1024, dtype=torch.uint8)            # pageable
    with pytest.raises(moe.MoeError):
        moe.moe_host_address(t)
    p = torch.empty(1024, dtype=torch.uint8).pin_memory()
    assert moe.moe_host_address(p) != 0
