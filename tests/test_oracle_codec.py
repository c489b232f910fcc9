"""Pins for the oracle's fp16 conversion and its Q4_K / Q8_0 codecs (CPU only).

External pins: numpy's IEEE binary16 conversion (a library routine) for every
fp16 value and for rounding ties; hand-packed blocks under tests/golden/ whose
bytes follow from the format reading by hand; error bounds of the quantisers.
"""
import os

import numpy as np
import pytest

import oracle

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _read_fixture(name):
    fields = {}
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            fields.setdefault(key, []).extend(vals)
    return fields


# ---------------------------------------------------------------- fp16

def test_f16_decode_matches_numpy_for_every_pattern():
    bits = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = bits.view(np.float16).astype(np.float32)
    got = np.array([oracle.f16_bits_to_f32(int(b)) for b in bits], np.float32)
    nan = np.isnan(ref)
    assert np.array_equal(np.isnan(got), nan)
    assert np.array_equal(got[~nan].view(np.uint32), ref[~nan].view(np.uint32))


def test_f16_roundtrip_every_non_nan_pattern():
    for b in range(65536):
        v = np.uint16(b).view(np.float16)
        if np.isnan(v):
            continue
        assert oracle.f32_to_f16_bits(float(np.float32(v))) == b


def test_f16_encode_matches_numpy_rne():
    rng = np.random.default_rng(1)
    # random magnitudes over the whole fp16 range and beyond, plus exact ties
    # (halfway between neighbouring fp16 values) and subnormal / overflow edges
    vals = [rng.standard_normal(4000).astype(np.float32) * np.float32(10.0) ** rng.integers(-9, 6, 4000)]
    f16 = np.arange(0, 0x7bff, 7, dtype=np.uint16).view(np.float16).astype(np.float64)
    ties = ((f16[:-1] + np.arange(0, 0x7bff, 7, dtype=np.uint16)[1:].view(np.float16).astype(np.float64)) / 2)
    vals.append(ties.astype(np.float32))
    vals.append(np.array([65504, 65519, 65520, 65536, 2.0 ** -24, 2.0 ** -25, 3 * 2.0 ** -26,
                          2.0 ** -14, 1 + 2.0 ** -11, 1 + 3 * 2.0 ** -11, 0.0, -0.0], np.float32))
    v = np.concatenate(vals)
    v = np.concatenate([v, -v])
    with np.errstate(over="ignore"):
        ref = v.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_bits(float(x)) for x in v], np.uint16)
    assert np.array_equal(got, ref)


# ---------------------------------------------------------------- Q4_K

def _handmade_q4k():
    f = _read_fixture("q4k_handmade_block.txt")
    sc = [int(s) for s in f["sc"]]
    m = [int(s) for s in f["m"]]
    expect = bytes(int(b, 16) for b in f["bytes"])
    assert len(expect) == 144
    x = np.zeros(256, np.float32)
    for j in range(8):
        for i in range(32):
            q = (i + j) % 16
            x[32 * j + i] = (2 * sc[j] * q - m[j]) / 128.0
    return x, expect


def test_q4k_handmade_block_packs_to_hand_bytes():
    x, expect = _handmade_q4k()
    got = oracle.q4k_quantize(x[None, :]).tobytes()
    assert got == expect


def test_q4k_handmade_block_dequantises_exactly():
    x, expect = _handmade_q4k()
    y = oracle.q4k_dequantize(np.frombuffer(expect, np.uint8), 1, 256)[0]
    assert np.array_equal(y.view(np.uint32), x.view(np.uint32))


def _decode_sub_scales(blk):
    """Per-sub-block step s_j and offset z_j of one block (test-side decode)."""
    d = np.frombuffer(blk[0:2], np.float16)[0].astype(np.float32)
    dmin = np.frombuffer(blk[2:4], np.float16)[0].astype(np.float32)
    scales = blk[4:16]
    s, z = [], []
    for j in range(8):
        if j < 4:
            sc, m = scales[j] & 63, scales[j + 4] & 63
        else:
            sc = (scales[j + 4] & 15) | ((scales[j - 4] >> 6) << 4)
            m = (scales[j + 4] >> 4) | ((scales[j] >> 6) << 4)
        s.append(np.float32(d * np.float32(sc)))
        z.append(np.float32(dmin * np.float32(m)))
    return np.array(s), np.array(z)


@pytest.mark.parametrize("dist", ["normal", "positive", "negative", "wide"])
def test_q4k_roundtrip_error_bound(dist):
    rng = np.random.default_rng(7)
    rows, cols = 64, 1024
    w = rng.standard_normal((rows, cols)).astype(np.float32) * np.float32(0.02)
    if dist == "positive":
        w = np.abs(w) + np.float32(0.01)
    elif dist == "negative":
        w = -np.abs(w) - np.float32(0.01)
    elif dist == "wide":
        w *= np.float32(10.0) ** rng.integers(-3, 3, (rows, cols // 32, 1)).repeat(32, 2).reshape(rows, cols).astype(np.float32)
    blob = oracle.q4k_quantize(w)
    y = oracle.q4k_dequantize(blob, rows, cols)
    xb = w.reshape(-1, 8, 32)
    yb = y.reshape(-1, 8, 32)
    blocks = blob.reshape(-1, 144)
    for b in range(blocks.shape[0]):
        s, z = _decode_sub_scales(blocks[b].tobytes())
        for j in range(8):
            x = xb[b, j].astype(np.float64)
            mn, mx = min(0.0, x.min()), x.max()
            # inside the covered grid [-z, 15 s - z] the error is at most half a step;
            # outside it the clamp at q = 0 / 15 sets the error
            bound = max(s[j] / 2, mx + z[j] - 15 * s[j], -(mn + z[j]))
            err = np.abs(x - yb[b, j].astype(np.float64)).max()
            assert err <= bound * (1 + 1e-5) + 1e-6 * np.abs(x).max() + 1e-30
    # the grid is never much coarser than the data: step <= (max-min)/15 * (1 + 1/63)
    assert np.abs(w - y).max() <= 0.06 * np.abs(w).max()


def test_q4k_zero_block_and_rejects_non_finite():
    z = np.zeros((2, 256), np.float32)
    blob = oracle.q4k_quantize(z)
    assert not blob.any()
    assert not oracle.q4k_dequantize(blob, 2, 256).any()
    bad = np.zeros((1, 256), np.float32)
    bad[0, 17] = np.nan
    with pytest.raises(ValueError):
        oracle.q4k_quantize(bad)
    bad[0, 17] = np.inf
    with pytest.raises(ValueError):
        oracle.q4k_quantize(bad)
    with pytest.raises(ValueError):
        oracle.q4k_quantize(np.full((1, 256), 3e38, np.float32))


def test_q4k_block_order_and_row_layout():
    """Blocks run along the row (cols), rows one after another."""
    rng = np.random.default_rng(3)
    w = rng.standard_normal((3, 512)).astype(np.float32)
    blob = oracle.q4k_quantize(w)
    for r in range(3):
        for b in range(2):
            one = oracle.q4k_quantize(w[r:r + 1, 256 * b:256 * (b + 1)])
            assert np.array_equal(blob[r, 144 * b:144 * (b + 1)], one[0])


# ---------------------------------------------------------------- Q8_0

def test_q8_0_handmade_block():
    f = _read_fixture("q8_0_handmade_block.txt")
    q = np.array([int(v) for v in f["q"]], np.float32)
    expect = bytes(int(b, 16) for b in f["bytes"])
    x = (q / np.float32(32.0)).astype(np.float32)
    assert oracle.q8_0_quantize(x[None, :]).tobytes() == expect
    y = oracle.q8_0_dequantize(np.frombuffer(expect, np.uint8), 1, 32)[0]
    assert np.array_equal(y, x)


def test_q8_0_roundtrip_error_bound():
    rng = np.random.default_rng(11)
    w = rng.standard_normal((32, 512)).astype(np.float32) * np.float32(0.02)
    blob = oracle.q8_0_quantize(w).reshape(-1, 34)
    y = oracle.q8_0_dequantize(blob, 32, 512).reshape(-1, 32)
    d = blob[:, :2].copy().view(np.float16).astype(np.float64).reshape(-1)
    err = np.abs(w.reshape(-1, 32).astype(np.float64) - y)
    assert (err <= d[:, None] * 0.5 * (1 + 1e-3) + 1e-12).all()
