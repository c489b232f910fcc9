"""GPU router / top-k / bucketing against the oracle (ids and buckets bit-exact
up to reported near-ties; weights close)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import workspace
from parity import compare_ids, oracle_inputs, selection_keys

sv = synth.small_variant

pytestmark = pytest.mark.gpu

W = synth.WORKLOADS
CASES = [
    (W["tiny"], 4), (W["tiny"], 0), (W["tiny"], 1000),
    (W["qwen_decode"], 1), (W["qwen_decode"], 5), (W["qwen_decode"], 8), (W["qwen_decode"], 333),
    (W["qwen_prefill"], 4096),
    (W["deepseek_decode"], 1), (W["deepseek_decode"], 8),
    (W["deepseek_prefill_skewed"], 4096),
]


def _route(wl, T, seed=0):
    x = synth.hidden_states(wl, max(T, 1), seed)[:T]
    xb, wr, b = oracle_inputs(wl, T, seed, x=x)
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    dev = "cuda"
    ids = torch.zeros(max(T, 1), wl.top_k, dtype=torch.int32, device=dev)
    w = torch.zeros(max(T, 1), wl.top_k, dtype=torch.float32, device=dev)
    offs = torch.full((wl.n_experts + 1,), -7, dtype=torch.int32, device=dev)
    assign = torch.zeros(max(T * wl.top_k, 1), dtype=torch.int32, device=dev)
    bias = None if b is None else torch.from_numpy(b).to(dev)
    moe.moe_route(cfg, x.to(dev).contiguous(), torch.from_numpy(wr).to(dev), bias, T, ids, w, offs, assign, ws)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    return xb, wr, b, ids[:T].cpu().numpy(), w[:T].cpu().numpy(), offs.cpu().numpy(), assign[:T * wl.top_k].cpu().numpy()


@pytest.mark.parametrize("wl,T", CASES, ids=lambda c: getattr(c, "name", str(c)))
def test_route_matches_oracle(wl, T):
    xb, wr, b, ids, w, offs, assign = _route(wl, T)
    if T == 0:
        assert (offs == 0).all()
        return
    oids, ow, kth, nxt = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    diff = compare_ids(ids, oids, kth, nxt, keys_of=lambda t: selection_keys(xb[t], wr, b, wl.score_fn))
    if diff:
        print("near-ties (reported): %d token(s): %s" % (len(diff), diff[:10]))
    same = [t for t in range(T) if t not in set(diff)]
    np.testing.assert_allclose(w[same], ow[same], rtol=2e-5, atol=1e-7)
    np.testing.assert_allclose(w.sum(1), 1.0, atol=1e-5)
    # buckets are a function of the ids: compare against the oracle's sort of the GPU ids
    counts, ooffs, oassign = oracle.bucket(ids, wl.n_experts)
    assert np.array_equal(offs, ooffs)
    assert np.array_equal(assign, oassign)
    assert counts.sum() == T * wl.top_k


def test_skewed_bias_concentrates_tokens():
    """ln(Zipf(1.2)) bias: hot experts get > 10x the mean token count."""
    wl = W["deepseek_prefill_skewed"]
    _, _, _, ids, _, offs, _ = _route(wl, 4096)
    counts = np.diff(offs)
    assert counts.max() > 10 * counts.mean()
    print("skewed routing: %d active experts, max/mean %.1f" % ((counts > 0).sum(), counts.max() / counts.mean()))


# ---------------------------------------------------------------- exact ties

TIE_GROUPS = [(2, 5, 11), (7, 8)]     # experts sharing one router row (and bias)


def _tied(wl, T, seed=0):
    x = synth.hidden_states(wl, T, seed)
    xb, wr, b = oracle_inputs(wl, T, seed, x=x)
    wr = wr.copy()
    b = None if b is None else b.copy()
    for grp in TIE_GROUPS:
        for e in grp[1:]:
            wr[e] = wr[grp[0]]
            if b is not None:
                b[e] = b[grp[0]]
    return x, xb, wr, b


def _assert_lower_id_wins(ids):
    """Experts with equal scores: a higher id is selected only after every lower one of its group."""
    hits = 0
    for t in range(ids.shape[0]):
        pos = {int(e): r for r, e in enumerate(ids[t])}
        for grp in TIE_GROUPS:
            for lo, hi in zip(grp, grp[1:]):
                if hi in pos:
                    assert lo in pos and pos[lo] < pos[hi], "token %d: ids %s break the lower-id rule" % (
                        t, ids[t].tolist())
                    hits += 1
    return hits


@pytest.mark.parametrize("wl,T", [(W["tiny"], 300), (sv(W["qwen_decode"], name="qwen_e64", n_experts=64), 300),
                                  (sv(W["deepseek_decode"], name="ds_e32", hidden=1024, n_experts=32, ff=512,
                                      shared_ff=0), 300)],
                         ids=["tiny", "qwen_e64", "ds_e32"])
def test_exact_ties_prefill_router(wl, T):
    """moe_route at T > 8 (tensor-core logits, warp top-k): equal scores go to the lower id."""
    x, xb, wr, b = _tied(wl, T)
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    ids = torch.zeros(T, wl.top_k, dtype=torch.int32, device="cuda")
    w = torch.zeros(T, wl.top_k, dtype=torch.float32, device="cuda")
    offs = torch.zeros(wl.n_experts + 1, dtype=torch.int32, device="cuda")
    assign = torch.zeros(T * wl.top_k, dtype=torch.int32, device="cuda")
    bias = None if b is None else torch.from_numpy(b).cuda()
    moe.moe_route(cfg, x.cuda(), torch.from_numpy(wr).cuda(), bias, T, ids, w, offs, assign, ws)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    gids = ids.cpu().numpy()
    oids, ow, kth, nxt = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    assert _assert_lower_id_wins(oids) > 0          # the case occurs
    hits = _assert_lower_id_wins(gids)
    assert hits > 0
    compare_ids(gids, oids, kth, nxt, keys_of=lambda t: selection_keys(xb[t], wr, b, wl.score_fn))


@pytest.mark.parametrize("T", [1, 5, 8])
@pytest.mark.parametrize("wl", [W["tiny"], sv(W["qwen_decode"], name="qwen_e64", n_experts=64),
                                sv(W["deepseek_decode"], name="ds_e32", hidden=1024, n_experts=32, ff=512,
                                   shared_ff=512)], ids=["tiny", "qwen_e64", "ds_e32"])
def test_exact_ties_decode_path(wl, T):
    """moe_forward on a decode window: the window's routing (read back through
    moe_workspace_routing) follows the lower-id rule for equal scores, and y
    matches the oracle."""
    from quantized_moe_expert_04_b300.layer import pack_layer, routing_views
    from parity import check_close, oracle_blobs, oracle_forward
    x, xb, wr, b = _tied(wl, 64)
    x, xb = x[:T], xb[:T]
    pl = pack_layer(wl, gen_device="cpu")
    pl.router_w.copy_(torch.from_numpy(wr))
    if b is not None:
        pl.router_bias.copy_(torch.from_numpy(b))
    cfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMV)
    ws = workspace(cfg, T)
    y32 = torch.empty(T, wl.hidden, dtype=torch.float32, device="cuda")
    y = torch.empty(T, wl.hidden, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg, x.cuda(), pl.router_w, pl.router_bias, pl.table, pl.shared, T, y, y32, ws)
    assert moe.moe_last_device_status(ws) == moe.MOE_OK
    ids, _, _, _ = routing_views(cfg, T, ws)
    gids = ids.cpu().numpy()
    oids, ow, kth, nxt = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    _assert_lower_id_wins(gids)
    diff = compare_ids(gids, oids, kth, nxt, keys_of=lambda t: selection_keys(xb[t], wr, b, wl.score_fn))
    blobs, sblob = oracle_blobs(wl, set(gids.reshape(-1).tolist()) | set(oids.reshape(-1).tolist()))
    ref = oracle_forward(wl, xb, wr, b, blobs, sblob, forced=gids if diff else None)
    check_close(y32.cpu().numpy(), ref, what="y_f32")


def test_exact_ties_occur_in_decode_windows():
    """The tied groups are selected inside decode windows of the cases above
    (so the decode tests exercise the rule, not just pass vacuously)."""
    wl = sv(W["qwen_decode"], name="qwen_e64", n_experts=64)
    _, xb, wr, b = _tied(wl, 64)
    oids, _, _, _ = oracle.route(xb[:8], wr, b, wl.top_k, wl.score_fn)
    assert _assert_lower_id_wins(oids) > 0
