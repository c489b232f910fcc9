"""Pins for the oracle's router, top-k selection, weights and bucketing (CPU).

External pins: numpy fp64 matmul/exp for the scores (library routines), Python's
stable sorted() for the selection order and for the bucketing (textbook
routines), and the invariants weights-sum-to-one and counts-sum-to-T*k.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import synth


def _inputs(T, H, E, seed, bias=False):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(T, H, generator=g).to(torch.bfloat16)
    wr = (torch.randn(E, H, generator=g) / np.sqrt(H)).float().numpy()
    b = (0.1 * torch.randn(E, generator=g)).float().numpy() if bias else None
    return synth.bf16_bits(x), x.float().numpy().astype(np.float64), wr, b


def _brute_force(xf, wr, b, k, score_fn):
    logits = xf @ wr.astype(np.float64).T
    if score_fn == oracle.SCORE_SOFTMAX:
        z = np.exp(logits - logits.max(1, keepdims=True))
        score = z / z.sum(1, keepdims=True)
        key = score
    else:
        score = 1.0 / (1.0 + np.exp(-logits))
        key = score + (b.astype(np.float64) if b is not None else 0.0)
    ids, ws, kth, nxt = [], [], [], []
    for t in range(xf.shape[0]):
        order = sorted(range(wr.shape[0]), key=lambda e: (-key[t, e], e))
        sel = order[:k]
        ids.append(sel)
        ws.append(score[t, sel] / score[t, sel].sum())
        kth.append(key[t, sel[-1]])
        nxt.append(key[t, order[k]] if len(order) > k else -np.inf)
    return np.array(ids), np.array(ws), np.array(kth), np.array(nxt)


@pytest.mark.parametrize("T,H,E,k", [(5, 256, 16, 2), (7, 512, 64, 10), (3, 256, 33, 6), (4, 256, 8, 8)])
def test_softmax_route_matches_brute_force(T, H, E, k):
    xb, xf, wr, _ = _inputs(T, H, E, seed=T * 100 + E)
    ids, w, kth, nxt = oracle.route(xb, wr, None, k, oracle.SCORE_SOFTMAX)
    rids, rw, rkth, rnxt = _brute_force(xf, wr, None, k, oracle.SCORE_SOFTMAX)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=1e-12, atol=1e-15)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(kth, rkth, rtol=1e-12)
    np.testing.assert_allclose(nxt, rnxt, rtol=1e-12)


@pytest.mark.parametrize("T,H,E,k", [(6, 256, 32, 6), (3, 512, 256, 6)])
def test_sigmoid_bias_route_matches_brute_force(T, H, E, k):
    xb, xf, wr, b = _inputs(T, H, E, seed=7 + E, bias=True)
    ids, w, kth, nxt = oracle.route(xb, wr, b, k, oracle.SCORE_SIGMOID_BIAS)
    rids, rw, rkth, rnxt = _brute_force(xf, wr, b, k, oracle.SCORE_SIGMOID_BIAS)
    assert np.array_equal(ids, rids)
    np.testing.assert_allclose(w, rw, rtol=1e-12)
    np.testing.assert_allclose(w.sum(1), 1.0, rtol=0, atol=1e-12)
    np.testing.assert_allclose(kth, rkth, rtol=1e-12)


def test_bias_changes_selection_not_weights():
    """A large bias on one expert forces it into the top-k; its weight stays s_e / sum s."""
    xb, xf, wr, _ = _inputs(4, 256, 16, seed=5)
    b = np.zeros(16, np.float32)
    b[11] = 100.0
    ids, w, _, _ = oracle.route(xb, wr, b, 3, oracle.SCORE_SIGMOID_BIAS)
    assert (ids[:, 0] == 11).all()
    s = 1.0 / (1.0 + np.exp(-(xf @ wr.astype(np.float64).T)))
    for t in range(4):
        np.testing.assert_allclose(w[t], s[t, ids[t]] / s[t, ids[t]].sum(), rtol=1e-12)


def test_exact_ties_go_to_the_lower_id():
    xb, _, wr, _ = _inputs(3, 256, 8, seed=9)
    wr[5] = wr[2]          # experts 2, 5 and 6 score identically for every token
    wr[6] = wr[2]
    ids, _, _, _ = oracle.route(xb, wr, None, 8, oracle.SCORE_SOFTMAX)
    for t in range(3):
        pos = {e: list(ids[t]).index(e) for e in (2, 5, 6)}
        assert pos[2] < pos[5] < pos[6]
        assert pos[6] - pos[2] == 2      # equal scores sit next to each other
    # with k = 1 and the tied trio on top, the lowest id wins
    wr[2] = np.where(xb[0].view(np.int16) < 0, -5.0, 5.0).astype(np.float32)
    wr[5] = wr[2]
    wr[6] = wr[2]
    ids1, _, _, _ = oracle.route(xb[:1], wr, None, 1, oracle.SCORE_SOFTMAX)
    assert ids1[0, 0] == 2


def test_forced_ids_give_forced_selection_and_renormalised_weights():
    xb, xf, wr, _ = _inputs(4, 256, 16, seed=21)
    forced = np.array([[3, 1], [0, 15], [7, 8], [2, 2 + 1]], np.int32)
    ids, w, _, _ = oracle.route(xb, wr, None, 2, oracle.SCORE_SOFTMAX, forced_ids=forced)
    assert np.array_equal(ids, forced)
    logits = xf @ wr.astype(np.float64).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    for t in range(4):
        np.testing.assert_allclose(w[t], p[t, forced[t]] / p[t, forced[t]].sum(), rtol=1e-12)


@pytest.mark.parametrize("T,k,E", [(1, 1, 4), (9, 3, 16), (64, 10, 512), (40, 6, 8), (0, 2, 4)])
def test_bucket_is_a_stable_counting_sort(T, k, E):
    rng = np.random.default_rng(T + k + E)
    ids = np.stack([rng.choice(E, k, replace=False) for _ in range(T)]) if T else np.zeros((0, k), np.int64)
    counts, offsets, assign = oracle.bucket(ids.astype(np.int32), E)
    flat = ids.reshape(-1)
    assert counts.sum() == T * k
    assert offsets[0] == 0 and offsets[-1] == T * k
    assert (np.diff(offsets) == counts).all()
    ref = sorted(range(T * k), key=lambda a: (flat[a], a))
    assert list(assign) == ref
    for e in range(E):
        seg = assign[offsets[e]:offsets[e + 1]]
        assert (flat[seg] == e).all()
        assert (np.diff(seg // k) > 0).all()     # token-ascending, one entry per token


def test_bucket_rejects_out_of_range_ids():
    with pytest.raises(ValueError):
        oracle.bucket(np.array([[0, 4]], np.int32), 4)
