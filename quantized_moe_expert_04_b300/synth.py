"""Seeded synthetic inputs for the MoE layer: workload shapes and generators.

This module is the one thing the CUDA path and the CPU oracle share.  It holds
none of the layer's arithmetic: it only draws random tensors with the shapes
and distributions of the workloads and hands out plain arrays.

Workloads (shapes from the pages; distributions are synthetic):
  * tiny      -- H=256, 16 experts, top-2 softmax, FF=128, T=4.
  * qwen      -- H=2560, 512 experts, top-10 softmax, FF=320: the 48-layer x
                 512-expert, ~10-active model of the Strata teardown page
                 (lcz.me/topic/2098/5, section 二) whose expert blob is
                 1,382,400 bytes (DeepSeek-V4-Flash page, lcz.me/post/23082,
                 section 三 item 4).  Decode windows T in {1, 3, 5} (MTP
                 verify windows of 3-5 drafted tokens, teardown page section
                 二) and a 4096-token prefill.
  * deepseek  -- H=4096, 256 routed experts, top-6 sigmoid + per-expert bias,
                 FF=2048, plus one always-on shared expert in Q8_0 (GGUF
                 anatomy table, DeepSeek-V4-Flash page section 二).  Decode
                 windows T in {1, 4, 8}; a skewed 4096-token prefill whose
                 bias is ln(Zipf(1.2)) popularity.

Distributions: x ~ N(0, 1) rounded to bf16; router W ~ N(0, 1/H) (variance
1/H, so logits are ~N(0, 1)); expert W ~ N(0, 0.02^2) (std 0.02) before
quantisation; decode bias ~ N(0, 0.1^2).

Every tensor has its own seed derived from (seed, layer, stream, index), so any
one expert of any layer can be regenerated on its own, on either device.
Note that torch's CPU and CUDA generators give different numbers for one
seed: whichever device generates the fp32 weights, both sides must be handed
the same values.
"""
from dataclasses import dataclass, field
import math
from typing import Optional, Tuple

import numpy as np
import torch

SOFTMAX = 0
SIGMOID_BIAS = 1

STREAM_X, STREAM_ROUTER, STREAM_BIAS, STREAM_EXPERT, STREAM_SHARED = range(5)


@dataclass(frozen=True)
class Workload:
    name: str
    hidden: int
    n_experts: int
    ff: int
    top_k: int
    score_fn: int
    shared_ff: int          # 0: no shared expert
    bias: str               # "none" | "normal" | "zipf"
    layers: int             # distinct layers the benchmark rotates through
    tokens: Tuple[int, ...] = field(default=(1,))
    codec: int = 0          # routed experts' blocks: 0 Q4_K, 1 Q5_K

    @property
    def has_shared(self) -> bool:
        return self.shared_ff > 0

    @property
    def blob_bytes(self) -> int:
        """Bytes of one routed expert: 3 Q4_K matrices [FF][H] (144 B / 256 weights;
        Q5_K 176 B)."""
        return 3 * self.ff * (self.hidden // 256) * (176 if self.codec == 1 else 144)

    @property
    def shared_blob_bytes(self) -> int:
        """Bytes of the shared expert: 3 Q8_0 matrices [FF_s][H] (34 B / 32 weights)."""
        return 3 * self.shared_ff * (self.hidden // 32) * 34


WORKLOADS = {
    "tiny": Workload("tiny", 256, 16, 128, 2, SOFTMAX, 0, "none", 1, (4,)),
    "qwen_decode": Workload("qwen_decode", 2560, 512, 320, 10, SOFTMAX, 0, "none", 48, (1, 3, 5)),
    "deepseek_decode": Workload("deepseek_decode", 4096, 256, 2048, 6, SIGMOID_BIAS, 2048,
                                "normal", 8, (1, 4, 8)),
    "qwen_prefill": Workload("qwen_prefill", 2560, 512, 320, 10, SOFTMAX, 0, "none", 4, (4096,)),
    "deepseek_prefill_skewed": Workload("deepseek_prefill_skewed", 4096, 256, 2048, 6,
                                        SIGMOID_BIAS, 2048, "zipf", 2, (4096,)),
    # the decode shapes with Q5_K routed experts (a codec of the same GGUF family)
    "qwen_decode_q5k": Workload("qwen_decode_q5k", 2560, 512, 320, 10, SOFTMAX, 0, "none", 48, (3,), 1),
    "deepseek_decode_q5k": Workload("deepseek_decode_q5k", 4096, 256, 2048, 6, SIGMOID_BIAS, 2048,
                                    "normal", 8, (8,), 1),
}


def seed_for(seed: int, layer: int, stream: int, index: int = 0) -> int:
    """One 63-bit generator seed per (seed, layer, stream, index)."""
    return (((seed * 4096 + layer) * 16 + stream) * (1 << 24) + index) % (1 << 63)


def _gen(device, s: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(s)
    return g


def hidden_states(wl: Workload, T: int, seed: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    """x [T, H] bf16 ~ N(0, 1)."""
    g = _gen(device, seed_for(seed, layer, STREAM_X))
    return torch.randn(T, wl.hidden, generator=g, device=device, dtype=torch.float32).to(torch.bfloat16)


def router_weight(wl: Workload, seed: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    """Wr [E, H] fp32 ~ N(0, 1/H)."""
    g = _gen(device, seed_for(seed, layer, STREAM_ROUTER))
    w = torch.randn(wl.n_experts, wl.hidden, generator=g, device=device, dtype=torch.float32)
    return w * (1.0 / math.sqrt(wl.hidden))


def router_bias(wl: Workload, seed: int = 0, layer: int = 0, device="cpu") -> Optional[torch.Tensor]:
    """Per-expert router bias [E] fp32, or None.

    normal: N(0, 0.1^2).  zipf: ln(p_e) with p_e proportional to (e+1)^-1.2,
    normalised over the experts (expert 0 the most popular)."""
    if wl.bias == "none":
        return None
    if wl.bias == "normal":
        g = _gen(device, seed_for(seed, layer, STREAM_BIAS))
        return 0.1 * torch.randn(wl.n_experts, generator=g, device=device, dtype=torch.float32)
    if wl.bias == "zipf":
        rank = np.arange(1, wl.n_experts + 1, dtype=np.float64)
        p = rank ** -1.2
        p /= p.sum()
        return torch.from_numpy(np.log(p).astype(np.float32)).to(device)
    raise ValueError(wl.bias)


def expert_weight(wl: Workload, e: int, seed: int = 0, layer: int = 0, device="cpu") -> torch.Tensor:
    """Expert e's fp32 weights [3, FF, H] (gate, up, down stored [FF][H]) ~ N(0, 0.02^2)."""
    g = _gen(device, seed_for(seed, layer, STREAM_EXPERT, e))
    return 0.02 * torch.randn(3, wl.ff, wl.hidden, generator=g, device=device, dtype=torch.float32)


def shared_weight(wl: Workload, seed: int = 0, layer: int = 0, device="cpu") -> Optional[torch.Tensor]:
    """Shared expert fp32 weights [3, FF_s, H] ~ N(0, 0.02^2), or None."""
    if not wl.has_shared:
        return None
    g = _gen(device, seed_for(seed, layer, STREAM_SHARED))
    return 0.02 * torch.randn(3, wl.shared_ff, wl.hidden, generator=g, device=device, dtype=torch.float32)


def bf16_bits(x: torch.Tensor) -> np.ndarray:
    """bf16 tensor -> numpy uint16 bit patterns (host)."""
    return x.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)


def small_variant(wl: Workload, **changes) -> Workload:
    """A copy of a workload with some fields changed (for scaled-down test shapes)."""
    d = dict(wl.__dict__)
    d.update(changes)
    return Workload(**d)
