#!/usr/bin/env python
"""Benchmark: MoE-layer tokens/s of the Q4_K sparse-MoE layer on B300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                    [--workload qwen_decode] [--tokens T]

One step = one pass of the whole layer (route, bucket, gate/up + SiLU*mul,
down + weighted combine) over every distinct layer of the workload, each
with a T-token window: the qwen_decode workload has 48 distinct layers of
512 Q4_K experts (~34 GB resident, far larger than L2), so consecutive calls
never find their weights in L2.  The step is captured once as a CUDA graph
and replayed; `value` = T * layers * K / time (tokens per second per layer).

Also reported: the dominant kernel's achieved bandwidth (or throughput)
against the measured peak, timed with CUDA events on the launching stream in
a separate eager pass; an end-to-end figure through the C ABI with host
buffers (pinned H2D of x and D2H of y inside the timed region); the CPU
oracle on a bounded sample of the same workload; SM clocks during the run.

Multi-GPU (torchrun): the layer does not shard here -- every rank runs an
independent replica ("replicas only"); value sums all ranks' tokens over the
slowest rank's time.
"""
import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from quantized_moe_expert_04_b300 import moe, synth  # noqa: E402
from quantized_moe_expert_04_b300.layer import (LayerStack, TieredLayer, pack_layer, routing_views,  # noqa: E402
                                                workspace)

DEFAULT_TOKENS = {"tiny": 4, "qwen_decode": 3, "deepseek_decode": 4, "qwen_prefill": 4096,
                  "deepseek_prefill_skewed": 4096, "qwen_decode_q5k": 3, "deepseek_decode_q5k": 8}
METRIC = "MoE-layer tokens/s"
UNIT = "tokens/s"


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            p = json.load(fh)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]), "source": "measured"}
    except Exception:
        return {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0, "source": "fallback"}


# ------------------------------------------------------------------ dist

def dist_init():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        dist.init_process_group(backend)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def all_max(v, world):
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons while running."""
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        fd, self.path = tempfile.mkstemp(suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.index), "--query-gpu=" + self.QUERY,
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.25)
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        rows = []
        try:
            for line in open(self.path):
                f = [c.strip() for c in line.split(",")]
                if len(f) >= 9 and f[1].replace(".", "").isdigit():
                    rows.append(f)
        except Exception:
            pass
        finally:
            try:
                os.unlink(self.path)
            except Exception:
                pass
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        sm = [float(r[1]) for r in rows]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, v in zip(names, r[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][2]),
                "reasons": sorted(reasons), "samples": len(rows),
                "power_w_max": max(float(r[3]) for r in rows if r[3].replace(".", "").isdigit()) if rows else None}


# ------------------------------------------------------------------ oracle leg

def oracle_sample(wl, T, layers, x_layers, gpu_ids=None, gpu_y32=None, time_budget_s=10.0, wall_budget_s=40.0,
                  max_tokens=None, gen_device="cuda"):
    """Time the CPU oracle on a bounded sample: the first layers (and, for
    large T, the first max_tokens tokens) of the same workload.  Packing the
    oracle's blobs is untimed set-up; routing, bucketing, dequantisation and
    the FFNs are timed.  Where the GPU's ids and fp32 outputs of those layers
    are given, the sample doubles as a parity check: ids compared (differences
    are near-ties, counted), y compared by rel-L2 / max-abs (the oracle rerun
    with the GPU's ids where they differ).
    Returns (tokens/s per layer, threads, description, parity or None)."""
    import oracle
    threads = oracle.set_threads(0)
    done_tok, spent, used_layers = 0, 0.0, 0
    num = den = 0.0
    max_err = max_ref = 0.0
    ties = compared = 0
    wall0 = time.perf_counter()
    for l in layers:
        x = x_layers[l].cpu()
        if max_tokens is not None:
            x = x[:max_tokens]
        xb = synth.bf16_bits(x)
        Ts = xb.shape[0]
        wr = synth.router_weight(wl, 0, l, device=gen_device).cpu().numpy()
        b = synth.router_bias(wl, 0, l, device=gen_device)
        b = None if b is None else b.cpu().numpy()
        oids, _, kth, nxt = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
        forced = None
        if gpu_ids is not None:
            g = gpu_ids[l][:Ts]
            diff = [t for t in range(Ts) if not np.array_equal(g[t], oids[t])]
            ties += len(diff)
            compared += Ts
            if diff:
                forced = g
        used = set(oids.reshape(-1).tolist()) | (set(forced.reshape(-1).tolist()) if forced is not None else set())
        blobs = [None] * wl.n_experts
        for e in sorted(used):
            blobs[e] = oracle.pack_expert(synth.expert_weight(wl, e, 0, l, device=gen_device).cpu().numpy(), wl.codec)
        sblob = None
        if wl.has_shared:
            sblob = oracle.pack_shared_q8_0(synth.shared_weight(wl, 0, l, device=gen_device).cpu().numpy())
        t0 = time.perf_counter()
        ref = oracle.moe_forward(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, xb, wr, b, blobs,
                                 wl.shared_ff, sblob, forced_ids=forced, codec=wl.codec)
        spent += time.perf_counter() - t0
        if gpu_y32 is not None and l in gpu_y32:
            got = gpu_y32[l][:Ts].astype(np.float64)
            num += float(((got - ref) ** 2).sum())
            den += float((ref ** 2).sum())
            max_err = max(max_err, float(np.abs(got - ref).max()))
            max_ref = max(max_ref, float(np.abs(ref).max()))
        done_tok += Ts
        used_layers += 1
        if spent >= time_budget_s or time.perf_counter() - wall0 >= wall_budget_s:
            break
    desc = "%d layer(s) x %d token(s) of %s (oracle: fp64 route+bucket+dequant+FFN; packing untimed)" % (
        used_layers, done_tok // max(used_layers, 1), wl.name)
    parity = None
    if gpu_y32 is not None and den > 0:
        parity = {"rel_l2": float("%.3e" % math.sqrt(num / den)), "max_abs_over_max_ref": float("%.3e" % (max_err / max_ref)),
                  "near_tie_tokens": ties, "tokens_compared": compared, "bar": {"rel_l2": 5e-3, "max_abs": 2e-2},
                  "ok": math.sqrt(num / den) <= 5e-3 and max_err <= 2e-2 * max_ref,
                  "sample": desc.split(" (")[0]}
    return done_tok / spent, threads, desc, parity


def cpu_kernel_sample(wl, T, layers, time_budget_s=8.0):
    """Time the AVX2 multi-token CPU expert kernel (cpu_baseline/) on the host
    cores: the experts' FFN and combine of one window per layer (the oracle's
    routing and Q4_K blobs, both untimed set-up), the first layers of the
    workload within the budget.  Returns tokens/s per layer, the selected
    experts' bytes per second, the threads and a description."""
    import cpu_baseline
    import oracle
    threads = os.cpu_count() or 1
    done_tok, spent, moved, used = 0, 0.0, 0, 0
    for l in range(layers):
        xb = synth.bf16_bits(synth.hidden_states(wl, T, 0, l))
        wr = synth.router_weight(wl, 0, l, device="cuda").cpu().numpy()
        b = synth.router_bias(wl, 0, l, device="cuda")
        b = None if b is None else b.cpu().numpy()
        ids, w, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
        sel = sorted(set(ids.reshape(-1).tolist()))
        U = len(sel)
        blobs = [None] * wl.n_experts
        for e in sel:
            blobs[e] = oracle.pack_expert_q4k(synth.expert_weight(wl, e, 0, l, device="cuda").cpu().numpy())
        cpu_baseline.moe_window(wl.hidden, wl.n_experts, wl.ff, wl.top_k, xb, ids, w, blobs, threads=threads)
        t0 = time.time()
        cpu_baseline.moe_window(wl.hidden, wl.n_experts, wl.ff, wl.top_k, xb, ids, w, blobs, threads=threads)
        spent += time.time() - t0
        done_tok += T
        moved += U * wl.blob_bytes
        used += 1
        if spent > time_budget_s:
            break
    return {"value": round(done_tok / spent, 2), "unit": UNIT, "gbs": round(moved / spent / 1e9, 2),
            "cores": threads, "kind": "avx2 multi-token expert kernel",
            "sample": "%d layer(s) x %d token(s) of %s (expert FFN + combine; routing and packing untimed)"
                      % (used, T, wl.name)}


# ------------------------------------------------------------------ algorithmic work

def algorithmic(wl, T, ids_per_layer):
    """Bytes and flops one layer call must move / compute, from its routing.

    Bytes: each selected expert's blob once per window (+ shared blob), the
    fp32 router matrix, bias, x in, y out, ids and weights.  Per kernel of the
    decode path: router E*H*4 + T*H*2; layer U*blob + shared blob (U = distinct
    experts the window selected).  Flops:
    router 2*T*E*H + 2*T*k*3*H*FF (+ 2*T*3*H*FF_s shared); padding not
    counted."""
    E, H, FF, k = wl.n_experts, wl.hidden, wl.ff, wl.top_k
    total_bytes, per_kernel = [], {"dec_route": [], "dec_layer": []}
    for ids in ids_per_layer:
        U = len(np.unique(ids))
        b = U * wl.blob_bytes + wl.shared_blob_bytes + E * H * 4 + (E * 4 if wl.bias != "none" else 0)
        b += 2 * T * H * 2 + T * k * 8
        total_bytes.append(b)
        per_kernel["dec_route"].append(E * H * 4 + T * H * 2)
        per_kernel["dec_layer"].append(U * wl.blob_bytes + wl.shared_blob_bytes)
    flops = 2 * T * E * H + 2 * T * k * 3 * H * FF + (2 * T * 3 * H * wl.shared_ff if wl.has_shared else 0)
    gemm_gateup_flops = 2 * T * k * 2 * H * FF
    return np.mean(total_bytes), {n: float(np.mean(v)) for n, v in per_kernel.items()}, flops, gemm_gateup_flops


# The sources a kernel's code comes from: its own file and the shared headers.
KERNEL_SOURCES = {
    "dec": ["decode.cu", "moe_internal.cuh", "dequant_f16.cuh"],
    "gemm": ["gemm_tc.cu", "moe_internal.cuh", "tc_ptx.cuh", "dequant_f16.cuh", "debug_hooks.cuh"],
}


def _code_only(text):
    """C/CUDA source with comments and whitespace removed (string literals kept)."""
    out, i, n = [], 0, len(text)
    while i < n:
        c = text[i]
        if c == '"':                                   # string literal, copied as is
            j = i + 1
            while j < n and text[j] != '"':
                j += 2 if text[j] == "\\" else 1
            out.append(text[i:j + 1])
            i = j + 1
        elif text.startswith("//", i):
            j = text.find("\n", i)
            i = n if j < 0 else j
        elif text.startswith("/*", i):
            j = text.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c.isspace():
            i += 1
        else:
            out.append(c)
            i += 1
    return "".join(out)


def kernel_source_hash(kernel):
    """Hash of the code (comments and whitespace aside) of the CUDA sources the kernel is
    built from: its DRAM traffic figures go stale when that code changes."""
    import hashlib
    h = hashlib.sha256()
    for fn in KERNEL_SOURCES[kernel.split("_")[0]]:
        with open(os.path.join(ROOT, "quantized_moe_expert_04_b300", "csrc", fn), encoding="utf-8") as fh:
            h.update(_code_only(fh.read()).encode("utf-8"))
    return h.hexdigest()[:16]


def profiled_traffic(kernel, workload, T):
    """DRAM bytes per launch from a committed ncu summary, if it still matches the source."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        rec = d.get("%s:%s:T%d" % (kernel, workload, T))
        if rec and rec.get("source_hash") == kernel_source_hash(kernel):
            return rec["dram_bytes_per_launch"]
    except Exception:
        pass
    return None


# ------------------------------------------------------------------ arms

# The five workloads: the headline (the Qwen-shaped MTP window of 3 tokens)
# plus every other window size and the two prefill batches, each measured in
# the same process after the headline.
STACK_SET = [("qwen_decode", 3), ("qwen_decode", 1), ("deepseek_decode", 8)]
CONFIG_SET = [("qwen_decode", 1), ("qwen_decode", 3), ("qwen_decode", 5), ("deepseek_decode", 1),
              ("deepseek_decode", 4), ("deepseek_decode", 8), ("qwen_prefill", 4096),
              ("deepseek_prefill_skewed", 4096), ("qwen_decode_q5k", 3), ("deepseek_decode_q5k", 8)]


def measure(args, wl, T, nL, world, rank, local, K=None, soak_s=0.0, target_s=0.3, e2e=False,
            cpu_budget=None, parity_layers=2):
    """Pack nL distinct layers of workload wl, then time K graph replays of one
    step (the nL layer calls with T-token inputs).  Returns the measurement
    dict (value, roofline, clocks, ...)."""
    dev = torch.device("cuda", local)
    flags = {"auto": 0, "gemv": moe.MOE_FLAG_FORCE_GEMV, "gemm": moe.MOE_FLAG_FORCE_GEMM}[args.path]
    flags |= moe.MOE_FLAG_STATIC_WEIGHTS     # the layers' weights are never rewritten
    cfg = moe.config_for(wl, flags)
    t_setup = time.time()
    layers = [pack_layer(wl, 0, l, gen_device="cuda") for l in range(nL)]
    xs = [synth.hidden_states(wl, T, 0, l, device="cuda").contiguous() for l in range(nL)]
    ys = [torch.empty(T, wl.hidden, dtype=torch.bfloat16, device=dev) for _ in range(nL)]
    ws = workspace(cfg, T)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup

    def step():
        for l in range(nL):
            pl = layers[l]
            moe.moe_forward(cfg, xs[l], pl.router_w, pl.router_bias, pl.table, pl.shared, T, ys[l], None, ws,
                            stream)

    # routing of each layer (for the algorithmic byte counts), fp32 outputs of
    # the first layers (for the parity sample) and the device status
    ids_per_layer, y32 = [], {}
    with torch.cuda.stream(stream):
        for l in range(nL):
            pl = layers[l]
            yf = torch.empty(T, wl.hidden, dtype=torch.float32, device=dev) if l < parity_layers else None
            moe.moe_forward(cfg, xs[l], pl.router_w, pl.router_bias, pl.table, pl.shared, T, ys[l], yf, ws,
                            stream)
            ids, _, _, _ = routing_views(cfg, T, ws)
            ids_per_layer.append(ids.cpu().numpy().copy())
            if yf is not None:
                y32[l] = yf.cpu().numpy()
    st = moe.moe_last_device_status(ws, stream)
    if st != moe.MOE_OK:
        raise moe.MoeError(st, "device status after the first pass (%s T=%d)" % (wl.name, T))

    # launches per layer call + per-kernel durations (eager, event-bracketed pass)
    moe.moe_profile_enable(True)
    prof_steps = max(3, min(K or 20, 20))
    with torch.cuda.stream(stream):
        for _ in range(prof_steps):
            step()
    stream.synchronize()
    prof = moe.moe_profile_read()
    moe.moe_profile_enable(False)
    launches_per_call = sum(v[0] for v in prof.values()) / (prof_steps * nL)

    # CUDA graph of one step
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        step()
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            step()
    torch.cuda.synchronize()
    for _ in range(args.warmup):
        graph.replay()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        graph.replay()
    torch.cuda.synchronize()
    per = (time.perf_counter() - t0) / 3
    if K is None:
        K = int(max(10, min(20000, target_s / max(per, 1e-7))))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        # the soak keeps the GPU busy with the same replays for >= soak_s inside the
        # sampled window (untimed), so the clock record reflects the timed steps
        n_soak = int(soak_s / max(per, 1e-7)) if soak_s > 0 else 0
        with torch.cuda.stream(stream):
            for _ in range(n_soak):
                graph.replay()
            ev0.record(stream)
            for _ in range(K):
                graph.replay()
            ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = all_max(ev0.elapsed_time(ev1), world)
    clocks = clk.summary()
    step_ms = ms / K
    value = T * nL * K * world / (ms / 1e3)

    out = {"workload": wl.name, "tokens_per_window": T, "distinct_layers": nL, "value": round(value, 2),
           "unit": UNIT, "steps": K, "ms_per_step": round(step_ms, 5), "us_per_layer": round(step_ms * 1e3 / nL, 3),
           "setup_s": round(setup_s, 1), "clocks": clocks,
           "timed_region_s": round(ms / 1e3, 3), "soak_replays": n_soak}

    # roofline: whole layer and the dominant kernel
    pk = peaks()
    step_bytes, kernel_bytes, flops, gemm_flops = algorithmic(wl, T, ids_per_layer)
    kernel_ms = {name: (v[2] / v[1] if v[1] else float("nan")) for name, v in prof.items()}
    share = {name: v[2] for name, v in prof.items()}
    decode = "dec_layer" in prof
    layer_s = step_ms / 1e3 / nL
    out["hbm"] = {"algorithmic_bytes_per_call": int(step_bytes), "gbs": round(step_bytes / layer_s / 1e9, 1),
                  "frac": round(step_bytes / layer_s / 1e9 / pk["hbm_gbs"], 4)}
    out["tflops"] = {"algorithmic_flops_per_call": int(flops), "achieved": round(flops / layer_s / 1e12, 3),
                     "frac": round(flops / layer_s / 1e12 / pk["bf16_tflops"], 4)}
    if decode:
        cands = [n for n in kernel_bytes if n in share]
        dom = max(cands, key=lambda n: share[n])
        achieved = kernel_bytes[dom] / (kernel_ms[dom] / 1e3) / 1e9
        out["roofline"] = {"bound": "hbm", "kernel": dom, "achieved": round(achieved, 1), "peak": pk["hbm_gbs"],
                           "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                           "traffic": profiled_traffic(dom, wl.name, T),
                           "peak_source": pk["source"] + " (burst copy)",
                           "avg_launch_us": round(kernel_ms[dom] * 1e3, 3),
                           "algorithmic_bytes_per_launch": int(kernel_bytes[dom]),
                           "per_kernel_gbs": {n: round(kernel_bytes[n] / (kernel_ms[n] / 1e3) / 1e9, 1)
                                              for n in kernel_bytes if n in kernel_ms}}
    else:
        dom = "gemm_gateup" if "gemm_gateup" in prof else max(share, key=share.get)
        achieved = gemm_flops / (kernel_ms[dom] / 1e3) / 1e12
        out["roofline"] = {"bound": "tensor", "kernel": dom, "achieved": round(achieved, 2),
                           "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": round(achieved / pk["bf16_tflops"], 4),
                           "traffic": profiled_traffic(dom, wl.name, T),
                           "peak_source": pk["source"] + " (fp16 operands; same nominal rate as bf16)",
                           "avg_launch_us": round(kernel_ms[dom] * 1e3, 3),
                           "algorithmic_flops_per_launch": int(gemm_flops)}
    out["kernels_ms_per_launch"] = {k: round(v, 5) for k, v in kernel_ms.items()}
    out["kernel_share"] = {k: round(v / sum(share.values()), 4) for k, v in share.items()}
    out["gpu_launches"] = int(round(launches_per_call * nL * K))
    out["dtype"] = "f16xf16->f32 (tensor-core MMAs), f32 combine"

    if e2e:
        # end to end through the C ABI with host buffers: every step copies its
        # inputs (the nL layers' x, one pinned host -> device copy), makes the
        # step's nL layer calls, and reads its results (the nL layers' y) back
        # into pinned host memory with one copy
        xh = torch.stack([x.cpu() for x in xs]).pin_memory()                   # [nL][T][H]
        yh = torch.empty(nL, T, wl.hidden, dtype=torch.bfloat16).pin_memory()
        xd = torch.empty(xh.shape, dtype=xh.dtype, device=dev)
        yd = torch.empty(yh.shape, dtype=yh.dtype, device=dev)
        Ke = max(3, min(K, 50))

        def e2e_step():
            xd.copy_(xh, non_blocking=True)
            for l in range(nL):
                pl = layers[l]
                moe.moe_forward(cfg, xd[l], pl.router_w, pl.router_bias, pl.table, pl.shared, T, yd[l], None, ws,
                                stream)
            yh.copy_(yd, non_blocking=True)

        with torch.cuda.stream(stream):
            for _ in range(2):
                e2e_step()
            stream.synchronize()
            barrier(world)
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(Ke):
                e2e_step()
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_ms = all_max(e0.elapsed_time(e1), world)
        out["e2e"] = {"value": round(T * nL * Ke * world / (e2e_ms / 1e3), 2), "unit": UNIT,
                      "h2d_bytes_per_step": int(nL * T * wl.hidden * 2),
                      "d2h_bytes_per_step": int(nL * T * wl.hidden * 2),
                      "path": "per step: one pinned H2D copy of the nL layers' x -> nL moe_forward calls -> "
                              "one D2H copy of their y, eager"}

    if rank == 0 and cpu_budget is not None:
        v, threads, desc, parity = oracle_sample(wl, T, list(range(nL)), xs, gpu_ids=ids_per_layer, gpu_y32=y32,
                                                 time_budget_s=cpu_budget, wall_budget_s=4 * cpu_budget + 10,
                                                 max_tokens=args.cpu_tokens if T > 64 else None)
        out["cpu_baseline"] = {"value": round(v, 3), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
        out["parity"] = parity
    del graph, layers, xs, ys, ws
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_stack(args, wl, T, nL, world, rank, local, target_s=1.0, cpu_budget=None, parity_layers=2,
                  layers=None):
    """The window through all nL layers in one launch (moe_forward_stack), every
    layer reading its own seeded input (the inputs of measure(): the two lines
    are the same work), layer l + 1 after layer l has finished.  (The residual
    stream of moe_forward_stack has no normalisation between layers: on the
    DeepSeek shapes it leaves the fp16 range within a few layers, so it is
    tested, not benchmarked.)  A step is one call: an 8-byte memset of the grid
    barrier words and the cooperative kernel.  Timing, clocks and roofline as
    measure(); the routing of every layer, for the byte counts, comes from
    moe_route on the same inputs."""
    dev = torch.device("cuda", local)
    t_setup = time.time()
    if layers is None:
        layers = [pack_layer(wl, 0, l, gen_device="cuda") for l in range(nL)]
    st = LayerStack(layers)
    cfg = moe.config_for(wl)
    ws = workspace(cfg, T)
    x = torch.stack([synth.hidden_states(wl, T, 0, l, device="cuda") for l in range(nL)]).contiguous()
    y = torch.empty(nL, T, wl.hidden, dtype=torch.bfloat16, device=dev)
    y32 = torch.empty(nL, T, wl.hidden, dtype=torch.float32, device=dev)
    stream = torch.cuda.Stream()
    torch.cuda.synchronize()
    setup_s = time.time() - t_setup

    def step(yf=None):
        moe.moe_forward_stack(cfg, nL, x, st.router_w, st.router_bias, st.blobs, st.shared, T, y, yf, ws, stream)

    with torch.cuda.stream(stream):
        step(y32)
    status = moe.moe_last_device_status(ws, stream)
    if status != moe.MOE_OK:
        raise moe.MoeError(status, "device status of the layer stack (%s T=%d)" % (wl.name, T))
    # every layer's routing on the kernel's own inputs (the library's router, one call a layer)
    rcfg = moe.config_for(wl, moe.MOE_FLAG_FORCE_GEMM)
    rws = workspace(rcfg, T)
    ids_per_layer = []
    rid = torch.empty(T, wl.top_k, dtype=torch.int32, device=dev)
    rw = torch.empty(T, wl.top_k, dtype=torch.float32, device=dev)
    roff = torch.empty(wl.n_experts + 1, dtype=torch.int32, device=dev)
    ras = torch.empty(T * wl.top_k, dtype=torch.int32, device=dev)
    for l in range(nL):
        moe.moe_route(rcfg, x[l], layers[l].router_w, layers[l].router_bias, T, rid, rw, roff, ras, rws)
        ids_per_layer.append(rid.cpu().numpy().copy())
    gpu_y32 = {l: y32[l].cpu().numpy() for l in range(min(parity_layers, nL))}

    for _ in range(max(args.warmup, 3)):
        step()
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(3):
        step()
    torch.cuda.synchronize()
    per = (time.perf_counter() - t0) / 3
    K = args.steps if args.stack_only and args.steps else int(max(10, min(20000, target_s / max(per, 1e-7))))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(local) as clk:
        with torch.cuda.stream(stream):
            ev0.record(stream)
            for _ in range(K):
                step()
            ev1.record(stream)
        torch.cuda.synchronize()
    barrier(world)
    ms = all_max(ev0.elapsed_time(ev1), world)
    step_ms = ms / K
    pk = peaks()
    step_bytes, _, _, _ = algorithmic(wl, T, ids_per_layer)
    launch_bytes = step_bytes * nL
    achieved = launch_bytes / (step_ms / 1e3) / 1e9
    out = {"workload": wl.name, "tokens_per_window": T, "distinct_layers": nL,
           "value": round(T * nL * K * world / (ms / 1e3), 2), "unit": UNIT, "steps": K,
           "ms_per_step": round(step_ms, 5), "us_per_layer": round(step_ms * 1e3 / nL, 3),
           "setup_s": round(setup_s, 1), "clocks": clk.summary(), "timed_region_s": round(ms / 1e3, 3),
           "hbm": {"algorithmic_bytes_per_call": int(step_bytes),
                   "gbs": round(achieved, 1), "frac": round(achieved / pk["hbm_gbs"], 4)},
           "roofline": {"bound": "hbm", "kernel": "dec_stack", "achieved": round(achieved, 1),
                        "peak": pk["hbm_gbs"], "unit": "GB/s", "frac": round(achieved / pk["hbm_gbs"], 4),
                        "traffic": profiled_traffic("dec_stack", wl.name, T),
                        "peak_source": pk["source"] + " (burst copy)",
                        "avg_launch_us": round(step_ms * 1e3, 3), "algorithmic_bytes_per_launch": int(launch_bytes)},
           "gpu_launches": K, "inputs": "each layer's own seeded x (the per-layer calls' inputs)"}
    if rank == 0 and cpu_budget is not None:
        xs = [x[l] for l in range(nL)]
        v, threads, desc, parity = oracle_sample(wl, T, list(range(min(parity_layers, nL))), xs,
                                                 gpu_ids=ids_per_layer, gpu_y32=gpu_y32,
                                                 time_budget_s=cpu_budget, wall_budget_s=4 * cpu_budget + 10)
        out["cpu_baseline"] = {"value": round(v, 3), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc}
        out["parity"] = parity
    del layers, st, ws, rws, x, y, y32
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def measure_tiered(wl, T, nL, n_slots, windows):
    """Host tier of the experts: every expert of nL layers in pinned host memory,
    a device cache of n_slots per layer.  Each decode step runs the nL layer
    calls eagerly (route -> ids to the host -> cache plan -> fills of the missed
    experts on a copy stream, waited for by the compute stream -> pointer table
    to the device -> moe_forward), windows steps in a row with fresh inputs (the
    synthetic routing has no locality, so the hit rate stays near the cache's
    share of the experts).  Reports tokens/s per layer, the hit rate, the rate at
    which missed experts' bytes cross from host memory and the fill rate."""
    cfg = moe.config_for(wl)
    layers = [TieredLayer(pack_layer(wl, 0, l, gen_device="cuda"), n_slots) for l in range(nL)]
    ws = workspace(cfg, T)
    xs = [[synth.hidden_states(wl, T, 1 + w, l, device="cuda") for l in range(nL)] for w in range(windows)]
    for l in range(nL):                      # one untimed step
        layers[l].forward(xs[0][l], ws)
    torch.cuda.synchronize()
    base = [tl.stats() for tl in layers]
    t0 = time.time()
    for w in range(windows):
        for l in range(nL):
            layers[l].forward(xs[w][l], ws)
    torch.cuda.synchronize()
    dt = time.time() - t0
    st = [tl.stats() for tl in layers]
    hits = sum(a["hits"] - b["hits"] for a, b in zip(st, base))
    misses = sum(a["misses"] - b["misses"] for a, b in zip(st, base))
    filled = sum(a["bytes"] - b["bytes"] for a, b in zip(st, base))
    status = moe.moe_last_device_status(ws)
    out = {"workload": wl.name, "tokens_per_window": T, "distinct_layers": nL, "slots_per_layer": n_slots,
           "experts_per_layer": wl.n_experts, "windows": windows, "status": status,
           "value": round(T * nL * windows / dt, 1), "unit": UNIT, "us_per_layer": round(dt * 1e6 / (nL * windows), 1),
           "hit_rate": round(hits / max(1, hits + misses), 4),
           "missed_bytes_gbs": round(misses * wl.blob_bytes / dt / 1e9, 2),
           "fill_gbs": round(filled / dt / 1e9, 2),
           "path": "eager per layer: route, ids to host, plan, fills (copy stream), table to device, forward"}
    for tl in layers:
        tl.cache.close()
    del layers, ws, xs
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    return out


def run_ours(args, world, rank, local):
    torch.cuda.set_device(local)
    if args.stack_only:
        wl = synth.WORKLOADS[args.workload or "qwen_decode"]
        T = args.tokens or DEFAULT_TOKENS[wl.name]
        r = measure_stack(args, wl, T, wl.layers if args.layers is None else args.layers, world, rank, local,
                          cpu_budget=None if args.no_cpu_baseline else min(args.cpu_budget, 4.0))
        if rank == 0:
            print(json.dumps({"stack": r}), flush=True)
        return
    wl = synth.WORKLOADS[args.workload or "qwen_decode"]
    T = args.tokens or DEFAULT_TOKENS[wl.name]
    nL = wl.layers if args.layers is None else args.layers
    cpu = None if args.no_cpu_baseline else args.cpu_budget
    head = measure(args, wl, T, nL, world, rank, local, K=args.steps, soak_s=args.soak, target_s=3.0, e2e=True,
                   cpu_budget=cpu)
    out = {
        "metric": METRIC, "value": head["value"], "unit": UNIT, "n_gpus": world, "steps": head["steps"],
        "warmup": args.warmup, "ms_per_step": head["ms_per_step"], "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": head["dtype"],
        "data": "synthetic (seeded; x~N(0,1) bf16, router W~N(0,1/H), experts N(0,0.02^2) packed to %s)" % ("Q5_K" if wl.codec else "Q4_K"),
        "config": {"workload": wl.name, "tokens_per_window": T, "hidden": wl.hidden, "experts": wl.n_experts,
                   "top_k": wl.top_k, "ff": wl.ff, "shared_ff": wl.shared_ff, "distinct_layers": nL,
                   "resident_expert_gb": round(nL * (wl.n_experts * wl.blob_bytes + wl.shared_blob_bytes) / 1e9, 2),
                   "l2": "inputs larger than L2 (distinct layers rotated)", "graph": "one CUDA graph per step",
                   "static_weights": True, "path": args.path, "parallelism": "replicas x%d" % world},
        "hbm": head["hbm"], "tflops": head["tflops"], "roofline": head["roofline"],
        "kernels_ms_per_launch": head["kernels_ms_per_launch"], "kernel_share": head["kernel_share"],
        "gpu_launches": head["gpu_launches"], "e2e": head["e2e"], "clocks": head["clocks"],
        "timed_region_s": head["timed_region_s"], "soak_replays": head["soak_replays"], "setup_s": head["setup_s"],
    }
    if "cpu_baseline" in head:
        out["cpu_baseline"] = head["cpu_baseline"]
        out["parity"] = head["parity"]
        if not wl.has_shared and wl.codec == 0 and T <= 64 and rank == 0:
            try:
                out["cpu_kernel"] = cpu_kernel_sample(wl, T, 8)
            except Exception as exc:          # no AVX2/FMA on this host, or no compiler
                out["cpu_kernel"] = {"unavailable": str(exc).splitlines()[0][:200]}
    if args.workload is None and not args.no_configs:
        confs = []
        for name, Tc in CONFIG_SET:
            wlc = synth.WORKLOADS[name]
            r = measure(args, wlc, Tc, wlc.layers, world, rank, local, K=None, soak_s=0.0, target_s=0.3,
                        e2e=False, cpu_budget=None if cpu is None else min(cpu, 4.0))
            confs.append({k: r[k] for k in ("workload", "tokens_per_window", "distinct_layers", "value", "unit",
                                            "steps", "ms_per_step", "us_per_layer", "hbm", "tflops", "roofline",
                                            "kernel_share", "clocks", "cpu_baseline", "parity") if k in r})
        out["configs"] = confs
        # host tier of the experts (decode windows): 4 layers, a quarter of each layer's experts cached
        out["tiered"] = measure_tiered(synth.WORKLOADS["qwen_decode"], 3, 4, 128, 20)
        # the window through each decode workload's whole layer stack in one launch
        packed = {}
        out["stack"] = []
        for name, Tc in STACK_SET:
            wls = synth.WORKLOADS[name]
            if name not in packed:
                packed.clear()
                torch.cuda.empty_cache()
                packed[name] = [pack_layer(wls, 0, l, gen_device="cuda") for l in range(wls.layers)]
            out["stack"].append(measure_stack(args, wls, Tc, wls.layers, world, rank, local,
                                              cpu_budget=None if cpu is None else min(cpu, 4.0),
                                              layers=packed[name]))
        packed.clear()
    if rank == 0:
        print(json.dumps(out), flush=True)


def run_reference(args, world, rank):
    """The CPU oracle as the reference arm, on this arm's workload and metric."""
    if rank != 0:
        return
    wl = synth.WORKLOADS[args.workload or "qwen_decode"]
    T = args.tokens or DEFAULT_TOKENS[wl.name]
    gen = "cuda" if torch.cuda.is_available() else "cpu"
    nL = min(wl.layers if args.layers is None else args.layers, 8)
    Ts = T if T <= 64 else args.cpu_tokens
    xs = [synth.hidden_states(wl, T, 0, l, device=gen)[:Ts] for l in range(nL)]
    import oracle
    threads = oracle.set_threads(0)
    prepared = []
    for l in range(nL):
        xb = synth.bf16_bits(xs[l])
        wr = synth.router_weight(wl, 0, l, device=gen).cpu().numpy()
        b = synth.router_bias(wl, 0, l, device=gen)
        b = None if b is None else b.cpu().numpy()
        ids, _, _, _ = oracle.route(xb, wr, b, wl.top_k, wl.score_fn)
        blobs = [None] * wl.n_experts
        for e in sorted(set(ids.reshape(-1).tolist())):
            blobs[e] = oracle.pack_expert(synth.expert_weight(wl, e, 0, l, device=gen).cpu().numpy(), wl.codec)
        sblob = oracle.pack_shared_q8_0(synth.shared_weight(wl, 0, l, device=gen).cpu().numpy()) \
            if wl.has_shared else None
        prepared.append((xb, wr, b, blobs, sblob))

    def step(i):
        xb, wr, b, blobs, sblob = prepared[i % nL]
        oracle.moe_forward(wl.hidden, wl.n_experts, wl.ff, wl.top_k, wl.score_fn, xb, wr, b, blobs,
                           wl.shared_ff, sblob, codec=wl.codec)

    for i in range(args.warmup):
        step(i)
    K = args.steps if args.steps is not None else 10
    t0 = time.perf_counter()
    for i in range(K):
        step(i)
    dt = time.perf_counter() - t0
    value = Ts * K / dt
    desc = "%d token(s) of a %d-token window, layers rotated over %d" % (Ts, T, nL)
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": round(dt / K * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic (seeded)",
        "config": {"workload": wl.name, "tokens_per_window": T, "hidden": wl.hidden, "experts": wl.n_experts,
                   "top_k": wl.top_k, "ff": wl.ff, "shared_ff": wl.shared_ff},
        "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": threads, "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=None)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(synth.WORKLOADS), default=None,
                    help="one workload only (default: the qwen_decode T=3 headline, then every config)")
    ap.add_argument("--tokens", type=int, default=None)
    ap.add_argument("--stack-only", action="store_true",
                    help="only the one-launch layer stack of --workload (default qwen_decode) at --tokens")
    ap.add_argument("--layers", type=int, default=None)
    ap.add_argument("--cpu-budget", type=float, default=10.0)
    ap.add_argument("--cpu-tokens", type=int, default=16)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="headline only")
    ap.add_argument("--soak", type=float, default=1.2,
                    help="seconds of untimed replays inside the clock-sampled window before the timed steps")
    ap.add_argument("--path", choices=["auto", "gemv", "gemm"], default="auto",
                    help="expert kernels: auto (GEMV for T <= 8, tensor-core GEMM above), or force one")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    world, rank, local = dist_init()
    if args.impl == "reference":
        run_reference(args, world, rank)
    else:
        if not torch.cuda.is_available():
            raise SystemExit("bench.py: the CUDA path needs a GPU (no CPU fallback)")
        run_ours(args, world, rank, local)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
