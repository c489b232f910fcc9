"""The AVX2 multi-token CPU expert kernel (cpu_baseline/) against the oracle:
same routing (the oracle's), the oracle's own Q4_K blobs; fp32 against fp64,
within the layer's tolerance.  CPU only."""
import numpy as np
import pytest

import cpu_baseline
import oracle
from quantized_moe_expert_04_b300 import synth
from parity import check_close, oracle_blobs, oracle_inputs

CASES = [
    (synth.WORKLOADS["tiny"], 4),
    (synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e16", hidden=512, n_experts=16, ff=320), 3),
    (synth.small_variant(synth.WORKLOADS["qwen_decode"], name="qwen_e8_t9", hidden=768, n_experts=8, ff=64,
                         top_k=3), 9),
]


@pytest.mark.parametrize("wl,T", CASES, ids=lambda c: getattr(c, "name", str(c)))
@pytest.mark.parametrize("threads", [1, 3])
def test_avx2_window_matches_the_oracle(wl, T, threads):
    xb, wr, b = oracle_inputs(wl, T)
    ids, w, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    blobs, _ = oracle_blobs(wl, ids.reshape(-1))
    ref = oracle.moe_forward(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, xb, wr, b, blobs, 0, None)
    y = cpu_baseline.moe_window(wl.hidden, wl.n_experts, wl.ff, wl.top_k, xb, ids, w, blobs, threads=threads)
    check_close(y, ref)


def test_avx2_window_rejects_bad_arguments():
    wl = synth.WORKLOADS["tiny"]
    xb, wr, b = oracle_inputs(wl, 2)
    ids, w, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
    with pytest.raises(RuntimeError):          # a selected expert without a blob
        cpu_baseline.moe_window(wl.hidden, wl.n_experts, wl.ff, wl.top_k, xb, ids, w, [None] * wl.n_experts)
    y = cpu_baseline.moe_window(wl.hidden, wl.n_experts, wl.ff, wl.top_k, xb[:0], ids[:0], w[:0],
                                [None] * wl.n_experts)
    assert y.shape == (0, wl.hidden)
