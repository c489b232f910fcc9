"""The whole layer on the GPU against the oracle.

Small shapes (oracle over every token, several warps/tiles and ragged tails)
and the full workload sizes in the benchmark's launch configuration: every
token of the 4096-token Qwen-shaped prefill, and for the skewed DeepSeek-shaped
prefill the tokens that sit at every tile of the grouped GEMM (the layer is
token-parallel, so checking a token checks every tile it passed through).
Ids must match up to reported near-ties; y within rel-L2 5e-3 and max-abs
2e-2 * max|ref|; for a near-tie token the oracle is rerun with the GPU's ids.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import forward, pack_layer, routing_views, workspace
from parity import check_close, compare_ids, oracle_blobs, oracle_forward, oracle_inputs, selection_keys

pytestmark = pytest.mark.gpu
W = synth.WORKLOADS
sv = synth.small_variant

SMALL = [
    (W["tiny"], 4),
    (W["tiny"], 1),
    (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 1),
    (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 3),
    (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 5),
    (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 8),
    (sv(W["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32, ff=512, shared_ff=512), 1),
    (sv(W["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32, ff=512, shared_ff=512), 8),
    (sv(W["deepseek_prefill_skewed"], name="ds_skew_small", hidden=1024, n_experts=32, ff=256, shared_ff=256), 77),
    (sv(W["qwen_prefill"], name="qwen_e64_prefill", n_experts=64), 200),
    # Q5_K routed experts (the decode path)
    (sv(W["qwen_decode"], name="qwen_e64_q5k", n_experts=64, codec=1), 1),
    (sv(W["qwen_decode"], name="qwen_e64_q5k", n_experts=64, codec=1), 3),
    (sv(W["qwen_decode"], name="qwen_e64_q5k", n_experts=64, codec=1), 8),
    (sv(W["qwen_decode"], name="qwen_e8_k4_q5k", n_experts=8, top_k=4, codec=1), 8),
    (sv(W["deepseek_decode"], name="ds_small_q5k", hidden=1024, n_experts=32, ff=512, shared_ff=512, codec=1), 1),
    (sv(W["deepseek_decode"], name="ds_small_q5k", hidden=1024, n_experts=32, ff=512, shared_ff=512, codec=1), 4),
    (sv(W["deepseek_decode"], name="ds_small_q5k", hidden=1024, n_experts=32, ff=512, shared_ff=512, codec=1), 8),
]


def tile_sample(offsets, assign, k, T, shared, tile=128):
    """Tokens that put the oracle on every tile of the grouped GEMM.

    The GEMM's work tiles run over bucket order: each expert's bucket is cut
    into token tiles of at most `tile` rows (equal sizes, multiples of 16), and
    every token of a tile meets all of its weight tiles and K splits.  So the
    first and last token of every token tile of every expert -- and of the
    shared expert's tiles over tokens 0..T-1 -- cover every (expert, weight
    tile, K split, token tile) position.  Bucket positions 16j and 16j - 1 are
    taken as well, so the sample does not depend on where exactly a tile ends."""
    toks = set()
    for e in range(len(offsets) - 1):
        b0, b1 = int(offsets[e]), int(offsets[e + 1])
        n = b1 - b0
        if n == 0:
            continue
        nt = (n + tile - 1) // tile
        tn = ((n + nt - 1) // nt + 15) // 16 * 16
        for p in list(range(0, n, tn)) + [min(j + tn, n) - 1 for j in range(0, n, tn)]:
            toks.add(int(assign[b0 + p]) // k)
        for p in range(0, n, 64):
            toks.add(int(assign[b0 + p]) // k)
        toks.add(int(assign[b1 - 1]) // k)
    if shared:
        nt = (T + tile - 1) // tile
        tn = ((T + nt - 1) // nt + 15) // 16 * 16
        for j in range(0, T, tn):
            toks.update((j, min(j + tn, T) - 1))
    return sorted(toks)


def _run(wl, T, gen_device, sample=None, flags=0, seed=0, layer=0):
    x = synth.hidden_states(wl, T, seed, layer)
    pl = pack_layer(wl, seed, layer, gen_device=gen_device)
    cfg = moe.config_for(wl, flags)
    ws = workspace(cfg, T)
    y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
    y = forward(pl, x.cuda(), ws, y_f32=y32, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    ids, w, offs, assign = routing_views(cfg, T, ws)
    if isinstance(sample, str) and sample == "tiles":
        sample = tile_sample(offs.cpu().numpy(), assign.cpu().numpy(), wl.top_k, T, wl.has_shared)
    toks = np.arange(T) if sample is None else np.asarray(sample)
    gids = ids.cpu().numpy()[toks]
    xb, wr, b = oracle_inputs(wl, T, seed, layer, gen_device=gen_device, x=x)
    xs = xb[toks]
    oids, ow, kth, nxt = oracle.route(xs, wr, b, wl.top_k, wl.score_fn)
    diff = compare_ids(gids, oids, kth, nxt, keys_of=lambda t: selection_keys(xs[t], wr, b, wl.score_fn))
    used = set(oids.reshape(-1).tolist()) | set(gids.reshape(-1).tolist())
    blobs, sblob = oracle_blobs(wl, used, seed, layer, gen_device=gen_device)
    forced = gids if diff else None
    ref = oracle_forward(wl, xs, wr, b, blobs, sblob, forced=forced)
    got32 = y32.cpu().numpy().astype(np.float64)[toks]
    got16 = y.float().cpu().numpy().astype(np.float64)[toks]
    r32 = check_close(got32, ref, what="y_f32")
    r16 = check_close(got16, ref, what="y")
    print("%s T=%d: rel-L2 %.2e (f32) %.2e (bf16), max-abs/max %.2e; near-ties %d" %
          (wl.name, T, r32[0], r16[0], r32[1], len(diff)))
    return y, y32, ws, pl


@pytest.mark.parametrize("wl,T", SMALL, ids=lambda c: getattr(c, "name", str(c)))
def test_small_shapes_match_oracle(wl, T):
    _run(wl, T, gen_device="cpu")


@pytest.mark.parametrize("wl,T", [(W["tiny"], 4), (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 8),
                                  (sv(W["qwen_decode"], name="qwen_e8_k4", n_experts=8, top_k=4), 8)],
                         ids=["tiny", "qwen_e64", "qwen_e8_k4"])
def test_forced_gemv_path(wl, T):
    """The decode path at its largest window; with 8 experts every expert
    serves several tokens (token pairs in the down projection)."""
    _run(wl, T, gen_device="cpu", flags=moe.MOE_FLAG_FORCE_GEMV)


def test_forced_gemv_rejects_windows_above_8():
    wl = sv(W["qwen_decode"], name="qwen_e64", n_experts=64)
    pl = pack_layer(wl, gen_device="cpu", experts=[])
    cfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMV)
    ws = workspace(cfg, 9)
    x = synth.hidden_states(wl, 9).cuda()
    y = torch.empty(9, wl.hidden, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(moe.MoeError) as err:
        moe.moe_forward(cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, 9, y, None, ws)
    assert err.value.status == moe.MOE_ERR_UNSUPPORTED_SHAPE


@pytest.mark.parametrize("T", [1, 3, 8])
def test_decode_deterministic_mode_matches_oracle(T):
    wl = sv(W["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32, ff=512, shared_ff=512)
    y, y32, ws, pl = _run(wl, T, gen_device="cpu", flags=moe.MOE_FLAG_DETERMINISTIC)
    cfg = moe.config_for(wl, moe.MOE_FLAG_DETERMINISTIC)
    x = synth.hidden_states(wl, T).cuda()
    assert torch.equal(forward(pl, x, ws, cfg=cfg), y)


def test_static_weights_flag_decode_path():
    """Decode windows chained with MOE_FLAG_STATIC_WEIGHTS (router rows and the
    expert table read before the previous call has finished), several calls
    back to back on one stream, each checked against the oracle."""
    wl = sv(W["qwen_decode"], name="qwen_e64", n_experts=64)
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl, moe.MOE_FLAG_STATIC_WEIGHTS | moe.MOE_FLAG_FORCE_GEMV)
    T = 5
    ws = workspace(cfg, T)
    xs = [synth.hidden_states(wl, T, seed=s).cuda() for s in range(4)]
    outs = [torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda") for _ in xs]
    for x, y32 in zip(xs, outs):
        forward(pl, x, ws, y_f32=y32, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    for s, (x, y32) in enumerate(zip(xs, outs)):
        xb, wr, b = oracle_inputs(wl, T, x=x.cpu())
        ids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
        blobs, sblob = oracle_blobs(wl, ids.reshape(-1))
        check_close(y32.cpu().numpy(), oracle_forward(wl, xb, wr, b, blobs, sblob), what="call %d" % s)


def test_static_weights_flag_matches():
    """Calls that may start reading the router early give the same result."""
    wl = sv(W["qwen_decode"], name="qwen_e64", n_experts=64)
    pl = pack_layer(wl, gen_device="cpu")
    x = synth.hidden_states(wl, 5).cuda()
    cfg0 = moe.config_for(wl, moe.MOE_FLAG_DETERMINISTIC)
    cfg1 = moe.config_for(wl, moe.MOE_FLAG_DETERMINISTIC | moe.MOE_FLAG_STATIC_WEIGHTS)
    ws = workspace(cfg0, 5)
    a = forward(pl, x, ws, cfg=cfg0).clone()
    outs = [forward(pl, x, ws, cfg=cfg1).clone() for _ in range(3)]
    for b in outs:
        assert torch.equal(a, b)


FULL = [
    (W["qwen_decode"], 1, None), (W["qwen_decode"], 3, None), (W["qwen_decode"], 5, None),
    (W["deepseek_decode"], 1, None), (W["deepseek_decode"], 4, None), (W["deepseek_decode"], 8, None),
    (W["qwen_prefill"], 4096, None),                    # every token (the oracle takes ~15 s)
    (W["deepseek_prefill_skewed"], 4096, "tiles"),      # every GEMM tile position
    (sv(W["qwen_decode"], name="qwen_decode_q5k", codec=1), 3, None),
    (sv(W["deepseek_decode"], name="deepseek_decode_q5k", codec=1), 8, None),
]


@pytest.mark.parametrize("wl,T,sample", FULL, ids=lambda c: getattr(c, "name", str(c)))
def test_full_size_sampled(wl, T, sample):
    _run(wl, T, gen_device="cuda", sample=sample)


def test_deterministic_reruns_bit_identical():
    wl = sv(W["qwen_decode"], name="qwen_e64", n_experts=64)
    x = synth.hidden_states(wl, 5).cuda()
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl, moe.MOE_FLAG_DETERMINISTIC)
    ws = workspace(cfg, 5)
    a = forward(pl, x, ws, cfg=cfg).clone()
    b = forward(pl, x, ws, cfg=cfg).clone()
    assert torch.equal(a, b)


def test_device_faults_are_reported():
    wl = W["tiny"]
    pl = pack_layer(wl, gen_device="cpu")
    cfg = pl.cfg
    ws = workspace(cfg, 4)
    x = synth.hidden_states(wl, 4).cuda()
    x[2, 7] = float("nan")
    forward(pl, x, ws)
    assert moe.moe_last_device_status(ws) == moe.MOE_ERR_DEVICE_FAULT
    assert moe.moe_last_device_status(ws) == moe.MOE_OK          # read clears it
    # a selected expert without a blob
    x = synth.hidden_states(wl, 4).cuda()
    forward(pl, x, ws)
    ids, _, _, _ = routing_views(cfg, 4, ws)
    e = int(ids[0, 0].item())
    table = pl.table.clone()
    table[e] = 0
    y = torch.empty(4, wl.hidden, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, x, pl.router_w, pl.router_bias, table, pl.shared, 4, y, None, ws)
    assert moe.moe_last_device_status(ws) == moe.MOE_ERR_DEVICE_FAULT


def test_missing_expert_blob_on_tensor_cores_is_reported():
    """The tensor-core path: the work tiles of a selected expert whose blob
    pointer is null are flagged when the tiles are planned, every role of both
    GEMMs skips them, and the call reports MOE_ERR_DEVICE_FAULT; the next call
    with the full table is right."""
    wl = sv(W["qwen_decode"], name="qwen_e16", n_experts=16)
    T = 40
    pl = pack_layer(wl, gen_device="cpu")
    cfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMM)
    ws = workspace(cfg, T)
    x = synth.hidden_states(wl, T).cuda()
    forward(pl, x, ws, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    ids, _, _, _ = routing_views(cfg, T, ws)
    table = pl.table.clone()
    table[int(ids[0, 0].item())] = 0
    y = torch.empty(T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, x, pl.router_w, pl.router_bias, table, pl.shared, T, y, None, ws)
    assert moe.moe_last_device_status(ws) == moe.MOE_ERR_DEVICE_FAULT
    y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
    forward(pl, x, ws, y_f32=y32, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    xb, wr, b = oracle_inputs(wl, T, x=x.cpu())
    oids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, sblob = oracle_blobs(wl, oids.reshape(-1))
    check_close(y32.cpu().numpy(), oracle_forward(wl, xb, wr, b, blobs, sblob))


GEMM_SMALL = [
    (W["tiny"], 4),
    (W["tiny"], 1),
    (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 5),
    (sv(W["deepseek_decode"], name="ds_small", hidden=1024, n_experts=32, ff=512, shared_ff=512), 8),
    (sv(W["qwen_decode"], name="qwen_e8_skew", n_experts=8, top_k=2), 700),   # buckets > 256: several N tiles
]


@pytest.mark.parametrize("wl,T", GEMM_SMALL, ids=lambda c: getattr(c, "name", str(c)))
def test_forced_gemm_path_matches_oracle(wl, T):
    """The tensor-core path at decode-sized and ragged buckets."""
    _run(wl, T, gen_device="cpu", flags=moe.MOE_FLAG_FORCE_GEMM)


@pytest.mark.parametrize("wl,T", [(sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 37),
                                  (sv(W["deepseek_prefill_skewed"], name="ds_skew_small", hidden=1024,
                                      n_experts=32, ff=256, shared_ff=256), 77)],
                         ids=["qwen_e64", "ds_skew_small"])
def test_gemm_deterministic_mode(wl, T):
    flags = moe.MOE_FLAG_FORCE_GEMM | moe.MOE_FLAG_DETERMINISTIC
    y, y32, ws, pl = _run(wl, T, gen_device="cpu", flags=flags)
    cfg = moe.config_for(wl, flags)
    x = synth.hidden_states(wl, T).cuda()
    y2 = forward(pl, x, ws, cfg=cfg)
    assert torch.equal(y, y2)


FULL_GEMM = [(W["qwen_decode"], 1), (W["qwen_decode"], 3), (W["deepseek_decode"], 1), (W["deepseek_decode"], 8)]


@pytest.mark.parametrize("wl,T", FULL_GEMM, ids=lambda c: getattr(c, "name", str(c)))
def test_full_size_decode_on_tensor_cores(wl, T):
    """Decode windows through the tensor-core path (K split across CTAs)."""
    _run(wl, T, gen_device="cuda", flags=moe.MOE_FLAG_FORCE_GEMM)


def test_prefill_activation_beyond_fp16_is_reported():
    """The tensor-core path multiplies fp16 activations: |SiLU(g) u| > 65504
    must raise MOE_ERR_DEVICE_FAULT instead of an infinite y."""
    wl = sv(W["qwen_decode"], name="qwen_e16", n_experts=16)
    T = 40
    pl = pack_layer(wl, gen_device="cpu", experts=[])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for e in range(wl.n_experts):
        w = synth.expert_weight(wl, e).clone()
        w[:2] *= 1000.0                                  # gate and up: |g|, |u| ~ 1e3, a ~ 1e6
        moe.moe_pack_q4k(w.reshape(3 * wl.ff, wl.hidden).cuda(), pl.blobs[e], st)
    assert int(st.item()) == 0
    cfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMM)
    ws = workspace(cfg, T)
    forward(pl, synth.hidden_states(wl, T).cuda(), ws, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_ERR_DEVICE_FAULT
    # the same layer at the normal scale is fine
    pl2 = pack_layer(wl, gen_device="cpu")
    forward(pl2, synth.hidden_states(wl, T).cuda(), ws, cfg=cfg)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK


@pytest.mark.parametrize("flags,T", [(moe.MOE_FLAG_FORCE_GEMM, 40), (moe.MOE_FLAG_FORCE_GEMV, 3)], ids=["gemm", "decode"])
def test_input_beyond_fp16_is_reported_on_both_paths(flags, T):
    """Both paths multiply fp16 copies of x: an element whose magnitude is not
    below 65504 -- for a bf16 value, 65536 and up (the bf16 number below it,
    65280, is an fp16 number), infinities and NaN too -- raises
    MOE_ERR_DEVICE_FAULT; 65280 itself passes.  The experts are scaled down
    (x 1e-3) so that the large element leaves the activations inside the fp16
    range."""
    wl = sv(W["qwen_decode"], name="qwen_e16", n_experts=16)
    pl = pack_layer(wl, gen_device="cpu", experts=[])
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    for e in range(wl.n_experts):
        w = synth.expert_weight(wl, e) * 1e-3
        moe.moe_pack_q4k(w.reshape(3 * wl.ff, wl.hidden).cuda(), pl.blobs[e], st)
    assert int(st.item()) == 0
    cfg = moe.config_for(wl, flags)
    ws = workspace(cfg, T)
    x0 = synth.hidden_states(wl, T)
    for v, ok in [(65280.0, True), (-65280.0, True), (65536.0, False), (-65536.0, False),
                  (float("inf"), False), (float("nan"), False)]:
        x = x0.clone()
        x[T - 1, 7] = v
        y = forward(pl, x.cuda(), ws, cfg=cfg)
        status = moe.moe_last_device_status(ws)
        assert status == (moe.MOE_OK if ok else moe.MOE_ERR_DEVICE_FAULT), (v, status)
        if ok:
            assert bool(torch.isfinite(y.float()).all())
