"""Pins for the oracle's whole layer (CPU only).

Strict top-k routing is the dense evaluation of every expert masked to the
selected k (the correctness baseline of the "Gap" post, item 6, turns off
every shortcut that would change which experts run).  The brute force here
evaluates all E experts for every token with numpy fp64 matmuls and masks the
result; the oracle's sparse, bucketed, expert-major loop must agree with it.
"""
import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import synth


def _make(wl, T, seed=0, zero_routed=False):
    x = synth.hidden_states(wl, T, seed)
    wr = synth.router_weight(wl, seed).numpy()
    b = synth.router_bias(wl, seed)
    b = None if b is None else b.numpy()
    w32 = [synth.expert_weight(wl, e, seed).numpy() for e in range(wl.n_experts)]
    if zero_routed:
        w32 = [np.zeros_like(w) for w in w32]
    blobs = [oracle.pack_expert_q4k(w) for w in w32]
    sw = synth.shared_weight(wl, seed)
    sblob = None if sw is None else oracle.pack_shared_q8_0(sw.numpy())
    return synth.bf16_bits(x), x.float().numpy().astype(np.float64), wr, b, blobs, sblob


def _dense_masked(wl, xf, wr, b, blobs, sblob):
    """All experts for every token, then the top-k mask (numpy fp64)."""
    T, H, FF = xf.shape[0], wl.hidden, wl.ff
    logits = xf @ wr.astype(np.float64).T
    if wl.score_fn == synth.SOFTMAX:
        p = np.exp(logits - logits.max(1, keepdims=True))
        score = p / p.sum(1, keepdims=True)
        key = score
    else:
        score = 1.0 / (1.0 + np.exp(-logits))
        key = score + b.astype(np.float64)
    mask = np.zeros_like(score)
    for t in range(T):
        sel = sorted(range(wl.n_experts), key=lambda e: (-key[t, e], e))[:wl.top_k]
        mask[t, sel] = score[t, sel] / score[t, sel].sum()
    y = np.zeros((T, H))
    nbytes = FF * (H // 256) * 144
    for e in range(wl.n_experts):
        W = [oracle.q4k_dequantize(blobs[e][m * nbytes:(m + 1) * nbytes], FF, H).astype(np.float64)
             for m in range(3)]
        g = xf @ W[0].T
        u = xf @ W[1].T
        a = g / (1.0 + np.exp(-g)) * u
        y += mask[:, e:e + 1] * (a @ W[2])
    if sblob is not None:
        SF = wl.shared_ff
        sbytes = SF * (H // 32) * 34
        S = [oracle.q8_0_dequantize(sblob[m * sbytes:(m + 1) * sbytes], SF, H).astype(np.float64)
             for m in range(3)]
        g = xf @ S[0].T
        u = xf @ S[1].T
        y += (g / (1.0 + np.exp(-g)) * u) @ S[2]
    return y


def _oracle(wl, xb, wr, b, blobs, sblob, forced=None):
    return oracle.moe_forward(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, xb, wr, b,
                              blobs, wl.shared_ff, sblob, forced_ids=forced)


SHAPES = [
    synth.WORKLOADS["tiny"],
    synth.small_variant(synth.WORKLOADS["tiny"], name="t2", n_experts=8, ff=64, top_k=3, tokens=(9,)),
    synth.small_variant(synth.WORKLOADS["deepseek_decode"], name="t3", hidden=256, n_experts=12, ff=64,
                        top_k=4, shared_ff=96, tokens=(5,)),
    synth.small_variant(synth.WORKLOADS["deepseek_prefill_skewed"], name="t4", hidden=512, n_experts=16,
                        ff=32, top_k=2, shared_ff=64, tokens=(11,)),
]


@pytest.mark.parametrize("wl", SHAPES, ids=lambda w: w.name)
def test_sparse_equals_dense_masked(wl):
    T = wl.tokens[0]
    xb, xf, wr, b, blobs, sblob = _make(wl, T, seed=1)
    y = _oracle(wl, xb, wr, b, blobs, sblob)
    ref = _dense_masked(wl, xf, wr, b, blobs, sblob)
    np.testing.assert_allclose(y, ref, rtol=1e-10, atol=1e-13 * np.abs(ref).max())


def test_unused_experts_need_no_blob_and_forced_ids_reproduce():
    wl = SHAPES[1]
    xb, xf, wr, b, blobs, _ = _make(wl, 9, seed=2)
    ids, _, _, _ = oracle.route(xb, wr, None, wl.top_k, wl.score_fn)
    used = set(ids.reshape(-1).tolist())
    sparse_blobs = [blobs[e] if e in used else None for e in range(wl.n_experts)]
    y = _oracle(wl, xb, wr, None, sparse_blobs, None)
    y2 = _oracle(wl, xb, wr, None, blobs, None, forced=ids)
    assert np.array_equal(y, y2)
    missing = list(sparse_blobs)
    missing[ids[0, 0]] = None
    with pytest.raises(ValueError):
        _oracle(wl, xb, wr, None, missing, None)


def test_shared_expert_alone():
    """All routed experts zero: the layer is the shared Q8_0 FFN."""
    wl = SHAPES[2]
    xb, xf, wr, b, blobs, sblob = _make(wl, 5, seed=3, zero_routed=True)
    y = _oracle(wl, xb, wr, b, blobs, sblob)
    H, SF = wl.hidden, wl.shared_ff
    sbytes = SF * (H // 32) * 34
    S = [oracle.q8_0_dequantize(sblob[m * sbytes:(m + 1) * sbytes], SF, H).astype(np.float64) for m in range(3)]
    g, u = xf @ S[0].T, xf @ S[1].T
    ref = (g * u / (1.0 + np.exp(-g))) @ S[2]
    np.testing.assert_allclose(y, ref, rtol=1e-11, atol=1e-14)


def test_single_expert_closed_form():
    """E = k = 1, one token, weights a constant per matrix: every dot product has
    a closed form, so y = c_d * FF * SiLU(c_g * S) * (c_u * S) with S = sum_h x_h."""
    wl = synth.Workload("one", 256, 1, 64, 1, synth.SOFTMAX, 0, "none", 1, (1,))
    w3 = np.stack([np.full((64, 256), c, np.float32) for c in (0.25, -0.5, 0.125)])
    blob = oracle.pack_expert_q4k(w3)
    consts = []
    for m in range(3):   # a constant matrix packs to a constant (rounded) matrix
        W = oracle.q4k_dequantize(blob[m * 64 * 144:(m + 1) * 64 * 144], 64, 256)
        assert (W == W[0, 0]).all() and abs(W[0, 0] - w3[m, 0, 0]) < 0.01
        consts.append(float(W[0, 0]))
    cg, cu, cd = consts
    x = torch.linspace(-1, 1, 256).to(torch.bfloat16)[None, :]
    xb = synth.bf16_bits(x)
    S = x.float().double().sum().item()
    y = _oracle(wl, xb, np.ones((1, 256), np.float32), None, [blob], None)
    g, u = cg * S, cu * S
    expect = cd * 64 * (g / (1 + np.exp(-g))) * u
    np.testing.assert_allclose(y, np.full((1, 256), expect), rtol=1e-13)


def test_token_permutation_equivariance():
    wl = SHAPES[3]
    xb, xf, wr, b, blobs, sblob = _make(wl, 11, seed=4)
    y = _oracle(wl, xb, wr, b, blobs, sblob)
    perm = np.random.default_rng(0).permutation(11)
    yp = _oracle(wl, xb[perm], wr, b, blobs, sblob)
    np.testing.assert_allclose(yp, y[perm], rtol=1e-12, atol=1e-15)


def test_zero_tokens():
    wl = SHAPES[0]
    xb, xf, wr, b, blobs, sblob = _make(wl, 1, seed=5)
    y = _oracle(wl, xb[:0], wr, b, blobs, sblob)
    assert y.shape == (0, wl.hidden)
