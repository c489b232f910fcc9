"""GPU pack / dequant kernels against the oracle's codecs: bit-exact bytes and values."""
import os

import numpy as np
import pytest
import torch

import oracle
from quantized_moe_expert_04_b300 import moe

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _inputs(kind, rows, cols, seed):
    g = torch.Generator().manual_seed(seed)
    w = torch.randn(rows, cols, generator=g) * 0.02
    if kind == "positive":
        w = w.abs() + 0.01
    elif kind == "negative":
        w = -w.abs() - 0.01
    elif kind == "wide":
        scale = 10.0 ** torch.randint(-4, 4, (rows, cols // 32, 1), generator=g).float()
        w = (w.view(rows, cols // 32, 32) * scale).view(rows, cols)
    elif kind == "sparse":
        w = w * (torch.rand(rows, cols, generator=g) < 0.1)
    elif kind == "zeros_signed":
        w = torch.zeros(rows, cols)
        w[::2] = -0.0
        w[min(1, rows - 1), 5] = 1e-30
    elif kind == "ties":
        # exact multiples that put many values on rounding ties
        w = torch.randint(-64, 64, (rows, cols), generator=g).float() / 64.0
    return w.float().contiguous()


KINDS = ["normal", "positive", "negative", "wide", "sparse", "zeros_signed", "ties"]


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 2560), (130, 4096)])
def test_pack_q4k_bit_exact(kind, rows, cols):
    w = _inputs(kind, rows, cols, seed=rows + cols)
    ref = oracle.q4k_quantize(w.numpy())
    out = torch.zeros(moe.moe_q4k_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_pack_q4k(w.cuda(), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu().numpy().reshape(ref.shape)
    assert np.array_equal(got, ref), "first differing byte at %s" % (np.argwhere(got != ref)[:3],)
    # dequantisation, both sides from the same bytes
    deq = torch.empty(rows, cols, dtype=torch.float32, device="cuda")
    moe.moe_dequant_q4k(out, rows, cols, deq)
    refd = oracle.q4k_dequantize(ref, rows, cols)
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), refd.view(np.uint32))


def test_pack_q4k_handmade_block():
    lines = [l.split() for l in open(os.path.join(GOLDEN, "q4k_handmade_block.txt")) if l.strip() and l[0] != "#"]
    sc = [int(v) for l in lines if l[0] == "sc" for v in l[1:]]
    m = [int(v) for l in lines if l[0] == "m" for v in l[1:]]
    expect = bytes(int(b, 16) for l in lines if l[0] == "bytes" for b in l[1:])
    x = torch.tensor([(2 * sc[j] * ((i + j) % 16) - m[j]) / 128.0 for j in range(8) for i in range(32)],
                     dtype=torch.float32)
    out = torch.zeros(144, dtype=torch.uint8, device="cuda")
    moe.moe_pack_q4k(x.view(1, 256).cuda(), out)
    assert bytes(out.cpu().numpy()) == expect
    deq = torch.empty(1, 256, dtype=torch.float32, device="cuda")
    moe.moe_dequant_q4k(out, 1, 256, deq)
    assert torch.equal(deq.cpu().view(-1), x)


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 2560), (130, 4096)])
def test_pack_q5k_bit_exact(kind, rows, cols):
    """Q5_K: the device quantiser's bytes equal the oracle's; the fp32 and the
    fp16 operand dequantisation (the decode kernel's device functions) equal
    the oracle's bit for bit."""
    w = _inputs(kind, rows, cols, seed=7 * rows + cols)
    ref = oracle.q5k_quantize(w.numpy())
    out = torch.zeros(moe.moe_q5k_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    moe.moe_pack_q5k(w.cuda(), out, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    got = out.cpu().numpy().reshape(ref.shape)
    assert np.array_equal(got, ref), "first differing byte at %s" % (np.argwhere(got != ref)[:3],)
    deq = torch.empty(rows, cols, dtype=torch.float32, device="cuda")
    moe.moe_dequant_q5k(out, rows, cols, deq)
    refd = oracle.q5k_dequantize(ref, rows, cols)
    assert np.array_equal(deq.cpu().numpy().view(np.uint32), refd.view(np.uint32))
    h = torch.empty(rows, cols, dtype=torch.int16, device="cuda")
    moe.moe_dequant_q5k_f16(out, rows, cols, h)
    bad = np.argwhere(h.cpu().numpy().view(np.uint16) != oracle.q5k_dequantize_f16(ref, rows, cols))
    assert bad.size == 0, "first differing fp16 weights at %s" % (bad[:3],)


def test_pack_q5k_uses_the_fifth_bit():
    """A ramp over 0..31 steps per sub-block: the quants span all 32 levels, so
    every qh bit position is exercised both ways."""
    j = np.arange(256)
    x = ((j % 32) * (1 + j // 32) / 64.0 - 0.25).astype(np.float32).reshape(1, 256)
    ref = oracle.q5k_quantize(x)
    assert ref[0, 16:48].min() == 0 and ref[0, 16:48].max() == 255
    out = torch.zeros(176, dtype=torch.uint8, device="cuda")
    moe.moe_pack_q5k(torch.from_numpy(x).cuda(), out)
    assert np.array_equal(out.cpu().numpy(), ref.reshape(-1))


@pytest.mark.parametrize("bad", [float("nan"), float("inf")])
def test_pack_q5k_flags_bad_input(bad):
    w = torch.zeros(2, 512, dtype=torch.float32)
    w[1, 300] = bad
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(moe.moe_q5k_bytes(2, 512), dtype=torch.uint8, device="cuda")
    moe.moe_pack_q5k(w.cuda(), out, st)
    assert int(st.item()) == moe.MOE_ERR_DEVICE_FAULT


@pytest.mark.parametrize("kind", ["normal", "wide", "sparse", "ties"])
def test_pack_q8_0_bit_exact(kind):
    rows, cols = 33, 4096
    w = _inputs(kind, rows, cols, seed=5)
    ref = oracle.q8_0_quantize(w.numpy())
    out = torch.zeros(moe.moe_q8_0_bytes(rows, cols), dtype=torch.uint8, device="cuda")
    moe.moe_pack_q8_0(w.cuda(), out)
    got = out.cpu().numpy().reshape(ref.shape)
    assert np.array_equal(got, ref)
    deq = torch.empty(rows, cols, dtype=torch.float32, device="cuda")
    moe.moe_dequant_q8_0(out, rows, cols, deq)
    assert np.array_equal(deq.cpu().numpy(), oracle.q8_0_dequantize(ref, rows, cols))


@pytest.mark.parametrize("bad", [float("nan"), float("inf"), 3e38])
def test_pack_flags_bad_input(bad):
    w = torch.zeros(2, 512, dtype=torch.float32)
    w[1, 300] = bad
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = torch.zeros(moe.moe_q4k_bytes(2, 512), dtype=torch.uint8, device="cuda")
    moe.moe_pack_q4k(w.cuda(), out, st)
    assert int(st.item()) == moe.MOE_ERR_DEVICE_FAULT
    st.zero_()
    out8 = torch.zeros(moe.moe_q8_0_bytes(2, 512), dtype=torch.uint8, device="cuda")
    moe.moe_pack_q8_0(w.cuda(), out8, st)
    assert int(st.item()) == moe.MOE_ERR_DEVICE_FAULT     # 3e38/127 overflows fp16 too


@pytest.mark.parametrize("kind", KINDS)
@pytest.mark.parametrize("rows,cols", [(1, 256), (37, 2560), (130, 4096)])
def test_fused_dequant_f16_bit_exact(kind, rows, cols):
    """The fp16 weights the fused tensor-core kernels multiply (their own
    device functions, through moe_dequant_q4k_f16) equal the oracle's R9
    rounding bit for bit, every sub-block j = 0..7 of every block."""
    w = _inputs(kind, rows, cols, seed=3 * rows + cols)
    blob = oracle.q4k_quantize(w.numpy())
    ref = oracle.q4k_dequantize_f16(blob, rows, cols)
    out = torch.empty(rows, cols, dtype=torch.int16, device="cuda")
    moe.moe_dequant_q4k_f16(torch.from_numpy(blob).cuda(), rows, cols, out)
    got = out.cpu().numpy().view(np.uint16)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, "first differing weights at %s" % (bad[:3],)


@pytest.mark.parametrize("kind", ["normal", "wide", "ties", "zeros_signed"])
def test_fused_dequant_q8_0_f16_bit_exact(kind):
    rows, cols = 33, 4096
    w = _inputs(kind, rows, cols, seed=11)
    blob = oracle.q8_0_quantize(w.numpy())
    ref = oracle.q8_0_dequantize_f16(blob, rows, cols)
    out = torch.empty(rows, cols, dtype=torch.int16, device="cuda")
    moe.moe_dequant_q8_0_f16(torch.from_numpy(blob).cuda(), rows, cols, out)
    assert np.array_equal(out.cpu().numpy().view(np.uint16), ref)
