"""Pins for the oracle's fp16 operand rounding of the dequantised weights (CPU only).

The GPU's tensor-core paths multiply fp16 weights: S_j = fp16(d*sc_j),
NZ_j = fp16(-(dmin*m_j)), w = fp16(q*S_j + NZ_j) with one rounding (Q4_K) and
w = fp16(d*q) (Q8_0).  The oracle writes that rounding out (its reading R9);
here it is pinned to things other than itself:
  * numpy's float64 -> float16 conversion (a library routine) for the
    double-to-half rounding the recipe ends with, including exact ties;
  * the hand-packed golden blocks, whose weights are exact fp16 values, so the
    rounded weights must equal the exact dequantised ones;
  * brute force: every result is the nearest fp16 (ties to even) of the
    exact rational q*S + NZ, found by scanning the fp16 grid;
  * the error bound against the exact (fp32) dequantisation.
"""
import os
from fractions import Fraction

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _fixture(name):
    fields = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if line and not line.startswith("#"):
                key, *vals = line.split()
                fields.setdefault(key, []).extend(vals)
    return fields


# every finite non-negative fp16 value, as exact fractions, for brute-force rounding
_F16_POS = np.arange(0, 0x7c00, dtype=np.uint16)
_F16_VALS = _F16_POS.view(np.float16).astype(np.float64)


def _nearest_f16_bits(v: Fraction) -> int:
    """Nearest binary16 to the exact rational v, ties to the even pattern (brute force)."""
    a = abs(v)
    i = int(np.searchsorted(_F16_VALS, float(a)))
    best = None
    for j in range(max(0, i - 2), min(len(_F16_VALS), i + 3)):
        cand = Fraction(float(_F16_VALS[j]))
        key = (abs(cand - a), int(_F16_POS[j]) & 1)
        if best is None or key < best[0]:
            best = (key, int(_F16_POS[j]))
    if a > Fraction(65504) + Fraction(16):          # beyond the rounding range of the largest finite
        bits = 0x7c00
    else:
        bits = best[1]
    return bits | (0x8000 if v < 0 else 0)


def test_f64_to_f16_matches_numpy():
    rng = np.random.default_rng(5)
    v = rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000)
    # values no fp32 holds (fp16 ties +- a double ulp), exact ties, range edges
    f16 = np.arange(1, 0x7bff, 5, dtype=np.uint16).view(np.float16).astype(np.float64)
    nxt = (np.arange(1, 0x7bff, 5, dtype=np.uint16) + 1).view(np.float16).astype(np.float64)
    mid = (f16 + nxt) / 2
    edges = np.array([65504.0, 65519.999999, 65520.0, 1e6, 2.0 ** -24, 2.0 ** -25, 2.0 ** -25 + 2.0 ** -60,
                      3 * 2.0 ** -26, 2.0 ** -14, 0.0, -0.0, 1 + 2.0 ** -11 + 2.0 ** -40])
    allv = np.concatenate([v, mid, np.nextafter(mid, np.inf), np.nextafter(mid, -np.inf), edges])
    allv = np.concatenate([allv, -allv])
    with np.errstate(over="ignore"):
        ref = allv.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f64_to_f16_bits(float(x)) for x in allv], np.uint16)
    bad = np.nonzero(got != ref)[0]
    assert bad.size == 0, [(allv[i], got[i], ref[i]) for i in bad[:5]]


def _handmade_q4k_bytes():
    f = _fixture("q4k_handmade_block.txt")
    return np.frombuffer(bytes(int(b, 16) for b in f["bytes"]), np.uint8)


def test_q4k_f16_handmade_block_is_exact():
    """d = 1/64, dmin = 1/128: every scale, min and weight is an exact fp16
    value, so the operand rounding changes nothing."""
    blk = _handmade_q4k_bytes()
    exact = oracle.q4k_dequantize(blk, 1, 256)[0]
    assert np.array_equal(exact.astype(np.float16).astype(np.float32), exact)
    got = oracle.q4k_dequantize_f16(blk, 1, 256)[0]
    assert np.array_equal(got, exact.astype(np.float16).view(np.uint16))


def test_q8_0_f16_handmade_block_is_exact():
    f = _fixture("q8_0_handmade_block.txt")
    blk = np.frombuffer(bytes(int(b, 16) for b in f["bytes"]), np.uint8)
    exact = oracle.q8_0_dequantize(blk, 1, 32)[0]
    got = oracle.q8_0_dequantize_f16(blk, 1, 32)[0]
    assert np.array_equal(got, exact.astype(np.float16).view(np.uint16))


def _q4k_fields(blk):
    d = Fraction(float(np.frombuffer(blk[0:2].tobytes(), np.float16)[0]))
    dmin = Fraction(float(np.frombuffer(blk[2:4].tobytes(), np.float16)[0]))
    sc8 = blk[4:16]
    out = []
    for j in range(8):
        if j < 4:
            sc, m = sc8[j] & 63, sc8[j + 4] & 63
        else:
            sc = (sc8[j + 4] & 15) | ((sc8[j - 4] >> 6) << 4)
            m = (sc8[j + 4] >> 4) | ((sc8[j] >> 6) << 4)
        out.append((int(sc), int(m)))
    return d, dmin, out


@pytest.mark.parametrize("seed", [0, 1])
def test_q4k_f16_is_nearest_fp16_of_the_rounded_terms(seed):
    """Brute force on random blocks: S and NZ are the nearest fp16 to the exact
    products, and each weight the nearest fp16 to q*S + NZ (one rounding)."""
    rng = np.random.default_rng(seed)
    w = (rng.standard_normal((2, 512)) * 0.02 * 10.0 ** rng.integers(-2, 3, (2, 1))).astype(np.float32)
    blob = oracle.q4k_quantize(w)
    got = oracle.q4k_dequantize_f16(blob, 2, 512).reshape(-1, 256)
    blocks = blob.reshape(-1, 144)
    for b in range(blocks.shape[0]):
        blk = blocks[b]
        d, dmin, sm = _q4k_fields(blk)
        qs = blk[16:]
        for j, (sc, m) in enumerate(sm):
            S = Fraction(float(np.uint16(_nearest_f16_bits(d * sc)).view(np.float16)))
            NZ = Fraction(float(np.uint16(_nearest_f16_bits(-(dmin * m))).view(np.float16)))
            c, half = j // 2, j % 2
            for l in range(0, 32, 3):
                byte = int(qs[32 * c + l])
                q = (byte >> 4) if half else (byte & 15)
                assert int(got[b, 32 * j + l]) == _nearest_f16_bits(q * S + NZ), (b, j, l)


def test_q4k_f16_error_bound_against_exact_dequant():
    rng = np.random.default_rng(9)
    w = (rng.standard_normal((16, 2560)) * 0.02).astype(np.float32)
    blob = oracle.q4k_quantize(w)
    exact = oracle.q4k_dequantize(blob, 16, 2560).astype(np.float64)
    f16 = oracle.q4k_dequantize_f16(blob, 16, 2560).view(np.float16).astype(np.float64)
    blocks = blob.reshape(-1, 144)
    err = np.abs(f16 - exact).reshape(-1, 8, 32)
    for b in range(blocks.shape[0]):
        d, dmin, sm = _q4k_fields(blocks[b])
        for j, (sc, m) in enumerate(sm):
            s, z = float(d * sc), float(dmin * m)
            # |S - s| <= ulp(s)/2, |NZ + z| <= ulp(z)/2, then one rounding of a value <= 15 s + z
            u = lambda v: 2.0 ** (np.floor(np.log2(max(v, 2.0 ** -14))) - 10)
            bound = 15 * u(s) / 2 + u(z) / 2 + u(15 * s + z) / 2
            assert err[b, j].max() <= bound * (1 + 1e-9)


def test_q8_0_f16_is_nearest_fp16_of_d_times_q():
    rng = np.random.default_rng(4)
    w = (rng.standard_normal((4, 256)) * 0.02).astype(np.float32)
    blob = oracle.q8_0_quantize(w).reshape(-1, 34)
    got = oracle.q8_0_dequantize_f16(blob, 4, 256).reshape(-1, 32)
    for b in range(blob.shape[0]):
        d = Fraction(float(np.frombuffer(blob[b, :2].tobytes(), np.float16)[0]))
        q = blob[b, 2:].view(np.int8)
        for i in range(0, 32, 5):
            assert int(got[b, i]) == _nearest_f16_bits(d * int(q[i]))
