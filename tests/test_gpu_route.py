"""GPU router / top-k / bucketing against the oracle (ids and buckets bit-exact
up to reported near-ties; weights close)."""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import moe, synth
from quantized_moe_expert_04_b300.layer import workspace
from parity import compare_ids, oracle_inputs, selection_keys

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
