"""Device-resident layer state for the C ABI: packed experts, router, workspace.

Plumbing around the binding: the fp32 expert weights come from the seeded
generators in ``synth`` and are packed on the GPU by ``moe_pack_q4k`` (or
``moe_pack_q5k``) / ``moe_pack_q8_0``; the pointer table, the router tensors and the workspace are
plain torch allocations.  No arithmetic of the layer happens here.
"""
from dataclasses import dataclass
from typing import List, Optional

import torch

from . import moe, synth


@dataclass
class PackedLayer:
    wl: synth.Workload
    router_w: torch.Tensor              # fp32 [E, H]
    router_bias: Optional[torch.Tensor] # fp32 [E] or None
    blobs: torch.Tensor                 # uint8 [E, blob_bytes]
    table: torch.Tensor                 # int64 [E] device pointers into blobs
    shared: Optional[torch.Tensor]      # uint8 [shared_bytes] or None

    @property
    def cfg(self) -> moe.moe_config:
        return moe.config_for(self.wl)


def pack_layer(wl: synth.Workload, seed: int = 0, layer: int = 0, gen_device: str = "cuda",
               experts: Optional[List[int]] = None) -> PackedLayer:
    """Generate and pack one layer on the current CUDA device.

    gen_device is where the fp32 weights are drawn ("cpu" gives the same
    numbers as the CPU-side tests; "cuda" is fast for the large workloads).
    experts, if given, restricts packing to those ids (others stay zero)."""
    dev = torch.device("cuda")
    cfg = moe.config_for(wl)
    nbytes = moe.moe_expert_bytes(cfg)
    assert nbytes == wl.blob_bytes
    blobs = torch.zeros(wl.n_experts, nbytes, dtype=torch.uint8, device=dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    pack = moe.moe_pack_q5k if wl.codec == moe.MOE_CODEC_Q5K else moe.moe_pack_q4k
    for e in (range(wl.n_experts) if experts is None else experts):
        w = synth.expert_weight(wl, e, seed, layer, device=gen_device).to(dev)
        pack(w.reshape(3 * wl.ff, wl.hidden), blobs[e], status)
    shared = None
    if wl.has_shared:
        sw = synth.shared_weight(wl, seed, layer, device=gen_device).to(dev)
        shared = torch.zeros(moe.moe_shared_bytes(cfg), dtype=torch.uint8, device=dev)
        moe.moe_pack_q8_0(sw.reshape(3 * wl.shared_ff, wl.hidden), shared, status)
    if int(status.item()) != 0:
        raise moe.MoeError(int(status.item()), "pack_layer")
    table = torch.tensor([blobs[e].data_ptr() for e in range(wl.n_experts)], dtype=torch.int64, device=dev)
    rw = synth.router_weight(wl, seed, layer, device=gen_device).to(dev).contiguous()
    rb = synth.router_bias(wl, seed, layer, device=gen_device)
    rb = None if rb is None else rb.to(dev).contiguous()
    return PackedLayer(wl, rw, rb, blobs, table, shared)


class LayerStack:
    """Pointer tables of a list of packed layers for moe_forward_stack."""

    def __init__(self, layers: List[PackedLayer]):
        dev = torch.device("cuda")
        wl = layers[0].wl
        self.layers, self.wl = layers, wl
        ptrs = lambda ts: torch.tensor([t.data_ptr() for t in ts], dtype=torch.int64, device=dev)
        self.router_w = ptrs([pl.router_w for pl in layers])
        self.router_bias = ptrs([pl.router_bias for pl in layers]) if layers[0].router_bias is not None else None
        self.blobs = torch.cat([pl.table for pl in layers]).contiguous()
        self.shared = ptrs([pl.shared for pl in layers]) if wl.has_shared else None

    def forward(self, x: torch.Tensor, ws: torch.Tensor, y: Optional[torch.Tensor] = None,
                y_f32: Optional[torch.Tensor] = None, residual: bool = True, flags: int = 0, stream=None):
        """x: bf16 [L][T][H] (residual: x[0] is read, x[1:] written); returns y [L][T][H]."""
        L, T = len(self.layers), x.shape[1]
        if y is None:
            y = torch.empty(L, T, self.wl.hidden, dtype=torch.bfloat16, device="cuda")
        cfg = moe.config_for(self.wl, flags | (moe.MOE_FLAG_RESIDUAL if residual else 0))
        moe.moe_forward_stack(cfg, L, x, self.router_w, self.router_bias, self.blobs, self.shared, T, y, y_f32,
                              ws, stream)
        return y


def workspace(cfg: moe.moe_config, max_tokens: int) -> torch.Tensor:
    """A zero-initialised workspace for calls of up to max_tokens tokens."""
    nbytes = moe.moe_workspace_bytes(cfg, max_tokens)
    if nbytes == 0:
        raise moe.MoeError(moe.MOE_ERR_UNSUPPORTED_SHAPE, "moe_workspace_bytes")
    ws = torch.empty(nbytes, dtype=torch.uint8, device="cuda")
    moe.moe_workspace_init(ws)
    return ws


def forward(pl: PackedLayer, x: torch.Tensor, ws: torch.Tensor, y: Optional[torch.Tensor] = None,
            y_f32: Optional[torch.Tensor] = None, cfg: Optional[moe.moe_config] = None, stream=None):
    T = x.shape[0]
    if y is None:
        y = torch.empty(T, pl.wl.hidden, dtype=torch.bfloat16, device="cuda")
    moe.moe_forward(cfg or pl.cfg, x, pl.router_w, pl.router_bias, pl.table, pl.shared, T, y, y_f32, ws,
                    stream)
    return y


def routing_views(cfg: moe.moe_config, T: int, ws: torch.Tensor):
    """ids [T,k], w [T,k], offsets [E+1], assign [T*k] of the last forward, as views into ws."""
    addrs = moe.moe_workspace_routing(cfg, T, ws)
    base = ws.data_ptr()
    k, E = cfg.top_k, cfg.n_experts

    def view(addr, n, dtype):
        off = addr - base
        return ws[off:off + 4 * n].view(dtype)

    ids = view(addrs[0], T * k, torch.int32).view(T, k)
    w = view(addrs[1], T * k, torch.float32).view(T, k)
    offsets = view(addrs[2], E + 1, torch.int32)
    assign = view(addrs[3], T * k, torch.int32)
    return ids, w, offsets, assign


class TieredLayer:
    """A packed layer whose experts live in pinned host memory, n_slots of them
    also in a device cache (moe_cache_*): per window the router's selection
    decides the pointer table; missed experts are copied into slots by the copy
    engine before the window's forward (the least recently used slots make
    room), and a missed expert that finds no slot is read by the kernels from
    host memory."""

    def __init__(self, pl: PackedLayer, n_slots: int):
        self.pl = pl
        E, bb = pl.wl.n_experts, pl.wl.blob_bytes
        self.host = pl.blobs.cpu().pin_memory()
        addrs = [moe.moe_host_address(self.host[e]) for e in range(E)]
        self.slots = torch.empty(max(1, n_slots) * bb, dtype=torch.uint8, device="cuda")
        self.cache = moe.ExpertCache(E, bb, addrs, self.slots, n_slots)
        self.table = torch.empty(E, dtype=torch.int64, device="cuda")
        self.copy_stream = torch.cuda.Stream()

    def forward(self, x: torch.Tensor, ws: torch.Tensor, y: Optional[torch.Tensor] = None,
                y_f32: Optional[torch.Tensor] = None, cfg: Optional[moe.moe_config] = None):
        pl, T = self.pl, x.shape[0]
        cfg = cfg or pl.cfg
        if T > 8 and not (cfg.flags & moe.MOE_FLAG_FORCE_GEMV):
            raise ValueError("host-resident experts are read by the decode path only (T <= 8)")
        k = pl.wl.top_k
        ids = torch.empty(T, k, dtype=torch.int32, device="cuda")
        w = torch.empty(T, k, dtype=torch.float32, device="cuda")
        off = torch.empty(pl.wl.n_experts + 1, dtype=torch.int32, device="cuda")
        asg = torch.empty(T * k, dtype=torch.int32, device="cuda")
        moe.moe_route(cfg, x, pl.router_w, pl.router_bias, T, ids, w, off, asg, ws)
        table, fills = self.cache.plan(ids.cpu().reshape(-1).tolist())
        self.cache.issue(torch.cuda.current_stream(), self.copy_stream)   # the forward waits for the fills
        self.table.copy_(torch.tensor(table, dtype=torch.int64))
        if y is None:
            y = torch.empty(T, pl.wl.hidden, dtype=torch.bfloat16, device="cuda")
        moe.moe_forward(cfg, x, pl.router_w, pl.router_bias, self.table, pl.shared, T, y, y_f32, ws)
        return y, fills

    def stats(self):
        return self.cache.stats()
