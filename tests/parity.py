"""Shared helpers of the parity tests: tolerances, id comparison, oracle runs.

Tolerances (the layer's stated bar): expert ids bit-exact except where the
oracle's k-th and (k+1)-th selection keys lie within 1e-6 of each other
(reported); outputs within relative L2 <= 5e-3 and max-abs <= 2e-2 * max|ref|.
"""
import numpy as np
import torch

import oracle
from quantized_moe_expert_04_b300 import synth

REL_L2 = 5e-3
MAX_ABS_FRAC = 2e-2
NEAR_TIE = 1e-6


def check_close(got, ref, rel_l2=REL_L2, max_abs_frac=MAX_ABS_FRAC, what="y"):
    got = np.asarray(got, np.float64)
    ref = np.asarray(ref, np.float64)
    assert got.shape == ref.shape, (got.shape, ref.shape)
    if ref.size == 0:
        return 0.0, 0.0
    assert np.isfinite(got).all(), "%s: non-finite output" % what
    den = np.linalg.norm(ref)
    rl = np.linalg.norm(got - ref) / den if den > 0 else np.linalg.norm(got)
    scale = np.abs(ref).max()
    ma = np.abs(got - ref).max() / scale if scale > 0 else np.abs(got).max()
    assert rl <= rel_l2, "%s: rel-L2 %.3e > %.1e" % (what, rl, rel_l2)
    assert ma <= max_abs_frac, "%s: max-abs %.3e * max|ref| > %.1e" % (what, ma, max_abs_frac)
    return rl, ma


def selection_keys(xb_row, wr, bias, score_fn):
    """fp64 selection keys of one token (the logit, or sigmoid + bias), used only
    to check that ids the GPU orders differently are near-ties."""
    x = (np.asarray(xb_row, np.uint16).astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    l = np.asarray(wr, np.float64) @ x
    if score_fn == 0:
        return l
    return 1.0 / (1.0 + np.exp(-l)) + (0.0 if bias is None else np.asarray(bias, np.float64))


def compare_ids(gpu_ids, orc_ids, kth_key, next_key, keys_of=None):
    """Tokens whose selected id lists differ from the oracle's; every one must be a near-tie.

    A different selected set is allowed only where the oracle's k-th and
    (k+1)-th keys are within NEAR_TIE.  A different order of the same experts
    is allowed only where the swapped experts' oracle keys are within
    NEAR_TIE (keys_of(t) gives token t's fp64 key vector); without keys_of an
    order difference fails.  Returns the differing tokens (reported by the
    caller)."""
    gpu_ids = np.asarray(gpu_ids)
    orc_ids = np.asarray(orc_ids)
    diff = [t for t in range(orc_ids.shape[0]) if not np.array_equal(gpu_ids[t], orc_ids[t])]
    for t in diff:
        if set(gpu_ids[t].tolist()) != set(orc_ids[t].tolist()):
            gap = kth_key[t] - next_key[t]
            assert gap <= NEAR_TIE, "token %d: ids differ (gpu %s, oracle %s) with key gap %.3e > %.0e" % (
                t, gpu_ids[t].tolist(), orc_ids[t].tolist(), gap, NEAR_TIE)
        if keys_of is not None:
            key = keys_of(t)
            g = gpu_ids[t]
            for r in range(len(g) - 1):
                assert key[g[r]] >= key[g[r + 1]] - NEAR_TIE, (
                    "token %d: gpu order %s puts key %.9f before %.9f" % (t, g.tolist(), key[g[r]], key[g[r + 1]]))
        else:
            assert set(gpu_ids[t].tolist()) != set(orc_ids[t].tolist()), (
                "token %d: same experts in another order (gpu %s, oracle %s)" % (
                    t, gpu_ids[t].tolist(), orc_ids[t].tolist()))
    return diff


def oracle_inputs(wl, T, seed=0, layer=0, gen_device="cpu", experts=None, x=None):
    """Oracle-side inputs drawn from the same generators as the GPU side."""
    if x is None:
        x = synth.hidden_states(wl, T, seed, layer)
    xb = synth.bf16_bits(x)
    wr = synth.router_weight(wl, seed, layer, device=gen_device).cpu().numpy()
    b = synth.router_bias(wl, seed, layer, device=gen_device)
    b = None if b is None else b.cpu().numpy()
    return xb, wr, b


def oracle_blobs(wl, expert_ids, seed=0, layer=0, gen_device="cpu"):
    """The oracle's own blobs (its quantiser, the workload's codec) for the listed
    experts; None elsewhere."""
    blobs = [None] * wl.n_experts
    for e in sorted(set(int(i) for i in expert_ids)):
        w = synth.expert_weight(wl, e, seed, layer, device=gen_device).cpu().numpy()
        blobs[e] = oracle.pack_expert(w, wl.codec)
    sblob = None
    if wl.has_shared:
        sblob = oracle.pack_shared_q8_0(synth.shared_weight(wl, seed, layer, device=gen_device).cpu().numpy())
    return blobs, sblob


def oracle_forward(wl, xb, wr, b, blobs, sblob, forced=None):
    return oracle.moe_forward(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, xb, wr, b, blobs,
                              wl.shared_ff, sblob, forced_ids=forced, codec=wl.codec)
