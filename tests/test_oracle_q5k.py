"""Pins for the oracle's Q5_K codec (readings R10, R11 in oracle/moe_oracle.c), CPU only.

  * with every fifth bit zero, a Q5_K block is a Q4_K block with 32 extra
    bytes: it must decode exactly as the Q4_K block it was transcoded from (the
    Q4_K codec is pinned by its hand-made golden block);
  * the fifth bit of element 64c + 32h + l is bit 2c + h of qh[l]: a block with
    d = 1, dmin = 0, every scale 1 and one qh bit set decodes to a single 16;
  * the quantiser: every weight within half a step of its sub-block's grid
    (31 steps), never worse than Q4_K's 15-step grid on the same data;
  * the fp16 operand rounding (R9 on Q5_K): the nearest fp16 of q*S + NZ;
  * the layer with Q5_K experts equals the dense all-experts evaluation masked
    to the top-k, with the Q5_K weights.
"""
from fractions import Fraction

import numpy as np
import pytest

import oracle
from quantized_moe_expert_04_b300 import synth


def _transcode_q4k_to_q5k(b4):
    b4 = b4.reshape(-1, 144)
    out = np.zeros((b4.shape[0], 176), np.uint8)
    out[:, :16] = b4[:, :16]          # d, dmin, scales
    out[:, 48:] = b4[:, 16:]          # low four bits; qh stays zero
    return out.reshape(-1)


def test_q5k_without_fifth_bits_decodes_as_q4k():
    rng = np.random.default_rng(3)
    w = (rng.standard_normal((6, 512)) * 0.02).astype(np.float32)
    b4 = oracle.q4k_quantize(w)
    b5 = _transcode_q4k_to_q5k(b4)
    assert np.array_equal(oracle.q5k_dequantize(b5, 6, 512), oracle.q4k_dequantize(b4, 6, 512))


def _unit_block():
    blk = np.zeros(176, np.uint8)
    blk[0:2] = np.frombuffer(np.float16(1.0).tobytes(), np.uint8)     # d = 1, dmin = 0
    s = blk[4:16]
    for j in range(4):
        s[j] = 1                       # sc_j = 1, m_j = 0 (j < 4)
        s[j + 8] = 1                   # sc_{j+4} = 1 (low nibble), m_{j+4} = 0
    return blk


@pytest.mark.parametrize("c", range(4))
@pytest.mark.parametrize("h", range(2))
def test_q5k_fifth_bit_position(c, h):
    for l in (0, 7, 31):
        blk = _unit_block()
        blk[16 + l] = 1 << (2 * c + h)
        y = oracle.q5k_dequantize(blk, 1, 256)[0]
        expect = np.zeros(256, np.float32)
        expect[64 * c + 32 * h + l] = 16.0
        assert np.array_equal(y, expect), (c, h, l)


def test_q5k_quantiser_error_bound_and_no_worse_than_q4k():
    rng = np.random.default_rng(11)
    w = (rng.standard_normal((8, 1024)) * 0.02 * 10.0 ** rng.integers(-2, 2, (8, 1))).astype(np.float32)
    b5 = oracle.q5k_quantize(w).reshape(-1, 176)
    y5 = oracle.q5k_dequantize(b5, 8, 1024).reshape(-1, 8, 32)
    y4 = oracle.q4k_dequantize(oracle.q4k_quantize(w), 8, 1024).reshape(-1, 8, 32)
    x = w.reshape(-1, 8, 32)
    for bi in range(b5.shape[0]):
        d = float(np.frombuffer(b5[bi, 0:2].tobytes(), np.float16)[0])
        dm = float(np.frombuffer(b5[bi, 2:4].tobytes(), np.float16)[0])
        s = b5[bi, 4:16]
        for j in range(8):
            sc = (s[j] & 63) if j < 4 else ((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4))
            m = (s[j + 4] & 63) if j < 4 else ((s[j + 4] >> 4) | ((s[j] >> 6) << 4))
            step, z = d * sc, dm * m
            mn = min(0.0, float(x[bi, j].min()))
            mx = float(x[bi, j].max())
            scale, nmin = (mx - mn) / 31, -mn
            err = np.abs(y5[bi, j] - x[bi, j])
            # the grid -z + q * step (q = 0..31) against [mn, mx] = [-nmin, -nmin + 31 scale]:
            # half a step inside it, plus how far its ends miss the range
            bound = 0.5 * step + 31 * abs(scale - step) + abs(nmin - z) + 1e-7
            assert err.max() <= bound, (bi, j, err.max(), bound)
    assert np.abs(y5 - x).mean() < np.abs(y4 - x).mean()


def test_q5k_f16_operand_rounding_is_the_nearest_fp16():
    rng = np.random.default_rng(2)
    w = (rng.standard_normal((2, 256)) * 0.03).astype(np.float32)
    blk = oracle.q5k_quantize(w).reshape(-1, 176)
    got = oracle.q5k_dequantize_f16(blk, 2, 256).reshape(-1, 256)
    for b in range(2):
        d = Fraction(float(np.frombuffer(blk[b, 0:2].tobytes(), np.float16)[0]))
        dm = Fraction(float(np.frombuffer(blk[b, 2:4].tobytes(), np.float16)[0]))
        s, qh, qs = blk[b, 4:16], blk[b, 16:48], blk[b, 48:]
        for j in range(8):
            sc = (s[j] & 63) if j < 4 else ((s[j + 4] & 15) | ((s[j - 4] >> 6) << 4))
            m = (s[j + 4] & 63) if j < 4 else ((s[j + 4] >> 4) | ((s[j] >> 6) << 4))
            S = Fraction(float(np.float16(float(d * sc))))
            NZ = Fraction(float(np.float16(float(-(dm * m)))))
            c, h = j // 2, j % 2
            for l in range(0, 32, 5):
                q = ((qs[32 * c + l] >> (4 * h)) & 15) | (((qh[l] >> (2 * c + h)) & 1) << 4)
                exact = q * S + NZ
                want = np.float16(float(exact))          # one rounding of a value exact in float64
                assert int(got[b, 64 * c + 32 * h + l]) == int(want.view(np.uint16)), (b, j, l)


def test_layer_with_q5k_experts_is_the_dense_masked_evaluation():
    wl = synth.small_variant(synth.WORKLOADS["tiny"], name="tiny_q5k", n_experts=8, ff=64, top_k=3)
    T = 5
    x = synth.hidden_states(wl, T)
    xf = x.float().numpy().astype(np.float64)
    wr = synth.router_weight(wl).numpy()
    blobs = [oracle.pack_expert_q5k(synth.expert_weight(wl, e).numpy()) for e in range(wl.n_experts)]
    y = oracle.moe_forward(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, synth.bf16_bits(x), wr, None,
                           blobs, codec=oracle.CODEC_Q5K)
    H, FF = wl.hidden, wl.ff
    logits = xf @ wr.astype(np.float64).T
    p = np.exp(logits - logits.max(1, keepdims=True))
    p /= p.sum(1, keepdims=True)
    ref = np.zeros((T, H))
    nbytes = FF * (H // 256) * 176
    for t in range(T):
        sel = sorted(range(wl.n_experts), key=lambda e: (-p[t, e], e))[:wl.top_k]
        for e in sel:
            W = [oracle.q5k_dequantize(blobs[e][m * nbytes:(m + 1) * nbytes], FF, H).astype(np.float64)
                 for m in range(3)]
            g, u = W[0] @ xf[t], W[1] @ xf[t]
            a = g / (1.0 + np.exp(-g)) * u
            ref[t] += p[t, e] / p[t, sel].sum() * (a @ W[2])
    assert np.allclose(y, ref, rtol=1e-9, atol=1e-12)
