#!/usr/bin/env python3
"""Benchmark of the routed MoE-FFN step on GB300: tokens/s and HBM roofline.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

A step is one token through one MoE-FFN layer (router, top-k, routed experts,
shared expert, combine) of the Flint-shaped decode layer (H=2048, 256 experts,
top-6, F=512, shared F=1024, Q4_1). Weights are synthetic (seeded, drawn on the
device) and rotate over enough distinct layers that every weight byte is cold
in L2 when it is read again. Timed on the device with CUDA events around a
replayed CUDA graph of the steps; rank 0 prints one JSON line.

The line also carries a "prefill" object: the same layer over a batch of 512
tokens per step (the batched path: router GEMM, selection, expert sort, tensor-
core grouped GEMMs), timed the same way, and under "prefill_configs" the
Ling-shaped K-quant layer (Q4_K gate/up, Q6_K down) over 512 tokens. With
``--workload flint_prefill_t512`` the batched step is the headline instead.

``--impl reference`` times the CPU oracle (float64, one thread) on a bounded
sample of the same workload instead.
"""

from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "MoE-FFN tokens/s (decode T=1, prefill T=512); % of HBM/tensor roofline"
UNIT = "tokens/s"


QTYPE_NAMES = {2: "Q4_0", 3: "Q4_1", 12: "Q4_K", 14: "Q6_K"}

# The decode chain's two activation arithmetics (the default, and MOE_F32_ACT).
ARITH_DTYPE = {False: "f32", True: "q4 x i16 block fixed point -> f32"}
ARITH_TEXT = {
    False: "4-bit weights dequantised exactly to f32 (d*q + m), f32 activations, f32 FMA accumulation "
           "(d * sum(q x) + m * sum(x) per block); router and routing in f32",
    True: "4-bit weights x activations in 16-bit block fixed point (15 bits and sign, power-of-two scale per "
          "16 values): exact int32 dots per half block (dp4a), f32 scaling and accumulation; router and routing "
          "in f32",
}
# Decode workloads timed beside the headline, each in a sub-object of the line.
OTHER_DECODE = ("flint_decode_t1", "lfm25_decode_t1", "ling_decode_t1", "ling_kq_decode_t1")
# batched workloads besides the Flint one, each a sub-object of the line's "prefill_configs"
OTHER_PREFILL = ("ling_kq_prefill_t512",)


def record_bytes(w, ff):
    """Bytes of one expert record of intermediate size ff (gate/up and down rows in
    their own block types)."""
    from expert_ffn_decode_gb300 import synth
    return synth.record_bytes(w["hidden"], ff, w["qtype"], w.get("qtype_down", 0))


def qtype_label(w):
    qd = w.get("qtype_down") or w["qtype"]
    return QTYPE_NAMES[w["qtype"]] + ("" if qd == w["qtype"] else "/" + QTYPE_NAMES[qd])


def layer_bytes(w):
    """Algorithmic bytes of one token's step: router, the k picked experts, the
    shared expert, x and out (the experts not picked are never read)."""
    H, E, K, F, Fs = w["hidden"], w["n_experts"], w["top_k"], w["expert_ff"], w["shared_ff"]
    rec = lambda ff: record_bytes(w, ff)
    router = E * H * 4 + (E * 4 if w.get("bias_std") is not None else 0)
    return router + K * rec(F) + (rec(Fs) if Fs else 0) + 2 * H * 4


# Sources of each profiled kernel: a committed capture's counters are used only while
# these files hash to what they were when it was taken.
KERNEL_SOURCES = {
    "decode_chain": ["decode.cu", "decode_host.h", "common.cuh", "plan.h", "select.cuh"],
    "tile_gemm": ["prefill_tc.cu", "prefill.cu", "prefill_host.h", "common.cuh", "plan.h", "tc.cuh", "select.cuh"],
}


def code_only(src):
    """C/CUDA source without its comments, whitespace runs collapsed: what the compiler sees.
    String and character literals are kept as they are."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
            out.append(" ")
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(kernel):
    """Hash of the code (comments and layout ignored) of the files a capture depends on."""
    import hashlib
    h = hashlib.sha256()
    for name in KERNEL_SOURCES[kernel]:
        with open(os.path.join(ROOT, "expert_ffn_decode_gb300", "csrc", name), encoding="utf-8") as f:
            h.update(name.encode() + b"\0" + code_only(f.read()).encode())
    return h.hexdigest()


def profile_counters(stem, kernel):
    """Counters of the committed ncu capture profiles/<stem>.json, or None when the kernel's
    sources changed since it was taken."""
    p = os.path.join(ROOT, "profiles", stem + ".json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    return d if d.get("source_sha256") == source_hash(kernel) else None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *a):
        self.out = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.out, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.out, _ = self.proc.communicate()

    def summary(self):
        rows = []
        for line in (self.out or "").strip().splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 7:
                continue
            try:
                rows.append((float(parts[0]), float(parts[1]), parts[3:7]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for _, _, r in rows for i, v in enumerate(r) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[0] for r in rows), "sm_max_mhz": max(r[1] for r in rows),
                "reasons": reasons, "samples": len(rows)}


def cpu_baseline(workload: str, seconds: float = 12.0, warmup: int = 0, max_tokens: int = 10 ** 9,
                 threads: int = 1):
    """The oracle, as it stands, on one thread, on a bounded sample of the workload:
    single-token calls on one synthetic layer until `seconds` or `max_tokens` is reached."""
    code = f"""
import json, os, sys, time
sys.path.insert(0, {ROOT!r})
import numpy as np
from expert_ffn_decode_gb300 import synth
from oracle import moe_oracle as mo
w = synth.WORKLOADS[{workload!r}]
layer = synth.make_layer(w)
cfg = mo.MoeConfig(hidden=w["hidden"], n_experts=w["n_experts"], top_k=w["top_k"], expert_ff=w["expert_ff"],
                   shared_ff=w["shared_ff"], n_groups=w["n_groups"], groups_used=w["groups_used"],
                   qtype=w["qtype"], qtype_down=w.get("qtype_down", 0), weights_scale=w["weights_scale"])
it = synth.token_stream(w["seed"], w["hidden"], 9)
call = lambda x: mo.moe_ffn(x, layer["router_w"], layer["bias"], layer["expert_blocks"],
                            layer["shared_blocks"], cfg)
for _ in range({warmup}):
    call(next(it)[None])
n, t0 = 0, time.perf_counter()
while n < {max_tokens} and (n == 0 or time.perf_counter() - t0 < {seconds}):
    call(next(it)[None])
    n += 1
dt = time.perf_counter() - t0
print(json.dumps({{"tokens": n, "seconds": dt}}))
"""
    env = dict(os.environ, OMP_NUM_THREADS=str(threads), OPENBLAS_NUM_THREADS=str(threads),
               MKL_NUM_THREADS=str(threads))
    r = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, env=env, timeout=900)
    if r.returncode != 0:
        return None, r.stderr[-400:]
    d = json.loads(r.stdout.strip().splitlines()[-1])
    return d, None


def dist_setup(n_gpus, backend="nccl"):
    """(rank, world, local rank) from the launcher's environment; with more than one rank,
    joins the process group (one process per GPU: NCCL; the CPU tests use gloo)."""
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group(backend)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v, world, dev):
    """The largest of every rank's v (the slowest rank's time)."""
    if world == 1:
        return float(v)
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v)], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_rate(units_per_rank, seconds, world, dev):
    """Whole-job throughput: the units all ranks processed over the slowest rank's time
    (every rank processes the same number of units)."""
    return units_per_rank * world / max_over_ranks(seconds, world, dev)


def layer_seed(rank, i, base=1000):
    """Seed of a rank's i-th benchmark layer: every rank draws its own layers."""
    return base + 7919 * rank + i


def run_reference(args, rank, world):
    """The oracle arm: warm-up steps, then the timed steps, one oracle token per
    step, within a 90 s budget (steps past the budget are not run; the line says
    how many were)."""
    if rank != 0:
        return
    from expert_ffn_decode_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    d, err = cpu_baseline(args.workload, seconds=90.0, warmup=min(args.warmup, 3), max_tokens=args.steps)
    if d is None:
        print(json.dumps({"impl": "reference", "unavailable": f"oracle failed: {err}"}))
        return
    v = d["tokens"] / d["seconds"] * w["n_tokens"]
    sample = (f"{d['tokens']} of the {args.steps} requested steps (one single-token oracle call each, "
              f"{d['seconds']:.1f} s) on one synthetic layer of the workload; numpy float64, one thread")
    line = {
        "impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "T": w["n_tokens"]},
        "cpu_baseline": {"value": v, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line))


def print_trace(ffn, w, layers, xs, L, NX, flags, dev, stream, chain=8, reps=5):
    """Per-phase timeline of the last launch of a chain of `chain` steps: for each
    trace point, the median and the max over CTAs of (time - earliest CTA start), us."""
    import torch
    cfg = ffn.make_cfg(**{**w, "n_tokens": 1, "flags": flags | ffn.MOE_TRACE})
    nbytes = ffn.moe_workspace_size(cfg)
    off = ffn.moe_trace_offset(cfg)
    ws = torch.zeros(nbytes, dtype=torch.uint8, device=dev)
    out = torch.empty(w["hidden"], device=dev)
    torch.cuda.synchronize(dev)  # the zeroed workspace before `stream` uses it
    nc = torch.cuda.get_device_properties(dev).multi_processor_count
    rows = []
    # the chain is captured in a CUDA graph and replayed, as the timed steps are, so the
    # timeline shows the kernels' overlap rather than the host's launch pace
    for i in range(chain):  # warm-up, and the kernels' attributes set outside the capture
        lay = layers[i % L]
        ffn.check(ffn.moe_ffn_forward_ex(xs[i % NX], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                         lay["shared_blocks"], cfg, out, ws, nbytes, stream))
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(chain):
            lay = layers[i % L]
            ffn.check(ffn.moe_ffn_forward_ex(xs[i % NX], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                             lay["shared_blocks"], cfg, out, ws, nbytes, stream))
    for rep in range(reps):
        g.replay()
        stream.synchronize()
        ffn.check(ffn.moe_workspace_status(ws, stream))
        rows.append(ws[off:off + nc * ffn.TRACE_STRIDE * 8].view(torch.int64).view(nc, ffn.TRACE_STRIDE).cpu().double())
    summary = {}
    for k, name in enumerate(ffn.TRACE_POINTS):
        if not name:
            continue
        med, mx = [], []
        for t in rows:
            col = t[:, k]
            col = col[col > 0]  # CTAs that recorded this point
            if col.numel() == 0:
                continue
            d = (col - t[t[:, 0] > 0, 0].min()) / 1e3
            med.append(float(d.median()))
            mx.append(float(d.max()))
        if med:
            summary[name] = [round(statistics.median(med), 2), round(statistics.median(mx), 2)]
    print("trace (us since first CTA start: [median over CTAs, max over CTAs]): " + json.dumps(summary),
          file=sys.stderr)


def active_bytes(w):
    """The second numerator: the bytes of the k picked experts and the shared expert only."""
    K, F, Fs = w["top_k"], w["expert_ff"], w["shared_ff"]
    return K * record_bytes(w, F) + (record_bytes(w, Fs) if Fs else 0)


def repeat_graph(step, K, L, stream, target_steps=1280, max_repeats=2048):
    """One CUDA graph of NR back-to-back repeats of exactly K consecutive steps (step i uses
    layer i % L). NR is a multiple of L / gcd(K, L), so the rotation over the layers
    continues from one replay to the next, and NR K is about `target_steps`, so a graph
    launch falls once in that many steps. Returns (graph, NR)."""
    import torch
    base = L // math.gcd(K, L)
    nr = base * max(1, math.ceil(math.ceil(target_steps / K) / base))
    nr = max(base, min(nr, base * max(1, max_repeats // base)))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(nr * K):
            step(i, stream)
    return g, nr


def timed_replays(g, stream, warm, min_ms, max_replays=10000):
    """`warm` untimed replays of the graph, then replays, each between two CUDA events on
    the replaying stream, until they add up to at least `min_ms` of device time. Returns the
    milliseconds of every timed replay."""
    import torch
    with torch.cuda.stream(stream):
        for _ in range(warm):
            g.replay()
    stream.synchronize()
    per = []
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    for _ in range(max_replays):
        with torch.cuda.stream(stream):
            e0.record(stream)
            g.replay()
            e1.record(stream)
        e1.synchronize()
        per.append(e0.elapsed_time(e1))
        if sum(per) >= min_ms and len(per) >= 5:
            break
    return per


def decode_timing(ffn, w, layers, xs, flags, dev, stream, K, warmup, min_ms):
    """The decode step of workload `w` (one token per step, step i on layer i % L and token
    i % NX): timed repeats of exactly K steps each, until at least `min_ms` of device time,
    after at least `warmup` warm-up steps and one whole rotation of the layers. Returns the
    median milliseconds per step over the repeats and how they were taken."""
    import torch
    L, NX, H = len(layers), len(xs), w["hidden"]
    cfg = ffn.make_cfg(**{**w, "n_tokens": 1, "flags": flags})
    ws_bytes = ffn.moe_workspace_size(cfg)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    outs = torch.zeros((2, H), device=dev)
    torch.cuda.synchronize(dev)  # the default stream's buffers are complete before `stream` uses them

    def step(i, st):
        lay = layers[i % L]
        ffn.check(ffn.moe_ffn_forward_ex(xs[i % NX], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                         lay["shared_blocks"], cfg, outs[i % 2], ws, ws_bytes, st))

    with torch.cuda.stream(stream):
        for i in range(2 * L):  # eager warm-up (plans, lazy module loading, shared-memory limits)
            step(i, stream)
    stream.synchronize()
    ffn.check(ffn.moe_workspace_status(ws, stream))
    g, nr = repeat_graph(step, K, L, stream)
    warm = max(1, math.ceil(max(warmup, L) / (nr * K)))
    per = timed_replays(g, stream, warm, min_ms)
    ffn.check(ffn.moe_workspace_status(ws, stream))
    med = statistics.median(per)
    return {"ms_per_step": med / (nr * K), "steps": K, "repeats": len(per) * nr, "timed_ms": round(sum(per), 3),
            "warmup_steps": warm * nr * K, "layers_rotated": L, "repeats_per_graph": nr, "replays": len(per),
            "replay_ms_min": round(min(per), 5), "replay_ms_max": round(max(per), 5)}


def decode_layers(synth, w, dev, rank, l2, layers=0):
    """Distinct device-resident layers of `w`, enough that 4 x L2 of step bytes pass between
    reuses of any weight byte, and 64 tokens."""
    L = layers or max(8, math.ceil(4 * l2 / layer_bytes(w)) + 1)
    lay = [synth.make_layer_torch(w, seed=layer_seed(rank, i), device=dev) for i in range(L)]
    return lay, synth.make_tokens_torch(77 + rank, w["hidden"], 64, dev)


def decode_roofline(w, ms, peak, peak_kind):
    achieved = layer_bytes(w) / (ms * 1e-3) / 1e9
    return {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
            "frac": round(achieved / peak, 4), "peak_kind": peak_kind, "bytes_per_step": layer_bytes(w),
            "active_bytes_per_step": active_bytes(w),
            "active_frac": round(active_bytes(w) / (ms * 1e-3) / 1e9 / peak, 4)}


def bench_chained(ffn, w, layers, L, dev, stream, reps=10, flags=0):
    """Per-layer latency with a real dependence between layers: x_{l+1} = x_l +
    FFN(rms_norm(x_l) * norm) (the residual form with the norm prologue, which keeps the
    layer's input bounded), rotating through the L distinct layers. One CUDA graph of G
    steps, replayed `reps` times; returns ms per step."""
    import torch
    H = w["hidden"]
    gen = torch.Generator(device=dev)
    gen.manual_seed(4242)
    norm = torch.empty(H, device=dev).uniform_(0.5, 1.5, generator=gen)
    x0 = torch.empty(H, device=dev).normal_(0.0, 1.0, generator=gen)
    cfg = ffn.make_cfg(**{**w, "n_tokens": 1, "flags": ffn.MOE_RESIDUAL | flags, "rms_eps": 1e-6, "ffn_norm": norm})
    ws_bytes = ffn.moe_workspace_size(cfg)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    bufs = torch.empty((2, H), device=dev)
    torch.cuda.synchronize(dev)  # norm, x0 and the zeroed workspace before `stream` reads them

    def step(i):
        lay = layers[i % L]
        ffn.check(ffn.moe_ffn_forward_ex(bufs[i % 2], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                         lay["shared_blocks"], cfg, bufs[(i + 1) % 2], ws, ws_bytes, stream))

    G = L * max(1, 320 // L)
    G += G % 2
    with torch.cuda.stream(stream):
        bufs[0].copy_(x0)
        for i in range(2 * L):
            step(i)
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(G):  # G is even: the graph starts and ends with x in bufs[0]
            step(i)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        bufs[0].copy_(x0)
        g.replay()
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    ffn.check(ffn.moe_workspace_status(ws, stream))
    if not bool(torch.isfinite(bufs[0]).all()):
        raise RuntimeError("chained layers left the f32 range")
    return ev0.elapsed_time(ev1) / (reps * G)


def bound_calls(ffn, layers, xs_host):
    """Per step: the C ABI call's pointer arguments as plain addresses, taken before the timed
    region the way a caller holding its buffers passes them."""
    lay = [tuple(ffn._ptr(l[k]) for k in ("router_w", "bias", "expert_blocks", "shared_blocks")) for l in layers]
    return [x.data_ptr() for x in xs_host], lay


def prefill_launches(w):
    """Kernel launches of one batched pass of at most 512 tokens. The tile path (all three
    matrices Q4_1, or all Q4_0, with H, F and Fs whole multiples of 128 (Q4_1) or 256 (Q4_0);
    or Q4_K gate/up with Q4_K or Q6_K down rows, H, F, Fs multiples of 256, Q6_K F, Fs <= 768):
    token images, router, top-k, sort, routed images, gate/up, down, combine. The general
    path: router, top-k, sort, x operand, gate/up, down, combine."""
    qt, qd = w["qtype"], w.get("qtype_down") or w["qtype"]
    H, F, Fs = w["hidden"], w["expert_ff"], w["shared_ff"]
    if qt == 12 and qd in (12, 14):
        tile = all(v % 256 == 0 for v in (H, F, Fs)) and (qd == 12 or (F <= 768 and Fs <= 768))
    else:
        kc = 128 if qt == 3 else 256
        tile = qt == qd and qt in (2, 3) and all(v % kc == 0 for v in (H, F, Fs))
    return 8 if tile else 7


def prefill_bytes(w, distinct):
    """Algorithmic bytes of one batched step: the router, every expert some token
    picked (`distinct` of them, each read once), the shared expert, x and out."""
    H, E, T, F, Fs = w["hidden"], w["n_experts"], w["n_tokens"], w["expert_ff"], w["shared_ff"]
    rec = lambda ff: record_bytes(w, ff)
    router = E * H * 4 + (E * 4 if w.get("bias_std") is not None else 0)
    return router + distinct * rec(F) + (rec(Fs) if Fs else 0) + 2 * T * H * 4


def bench_prefill(ffn, synth, workload, dev, rank, steps, warmup, e2e_steps=20, layers=0):
    """Batched steps of `workload` (T tokens per call) on rotating layers; returns a dict
    with tokens/s, ms per step, the HBM roofline of the step and the end-to-end figure."""
    import torch
    w = synth.WORKLOADS[workload]
    T, H, K = w["n_tokens"], w["hidden"], w["top_k"]
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    full = prefill_bytes(w, w["n_experts"])
    L = layers or max(2, math.ceil(2 * l2 / full) + 1)
    layers = [synth.make_layer_torch(w, seed=layer_seed(rank, i, 5000), device=dev) for i in range(L)]
    NX = 3
    xs = [synth.make_tokens_torch(300 + 17 * rank + j, H, T, dev) for j in range(NX)]
    out = torch.zeros((T, H), device=dev)
    cfg = ffn.make_cfg(**{**w, "n_tokens": T, "flags": 0})
    ws_bytes = ffn.moe_workspace_size(cfg)
    ws = torch.zeros(ws_bytes, dtype=torch.uint8, device=dev)
    stream = torch.cuda.Stream(dev)
    ids = torch.empty((T, K), dtype=torch.int32, device=dev)
    # the layers, tokens and zeroed buffers are drawn on the default stream: complete them
    # before the side stream reads them (and before it reuses memory their temporaries held)
    torch.cuda.synchronize(dev)

    def step(i, st, want_ids=False):
        lay = layers[i % L]
        ffn.check(ffn.moe_ffn_forward_ex(xs[i % NX], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                         lay["shared_blocks"], cfg, out, ws, ws_bytes, st,
                                         ids if want_ids else None))

    # distinct experts per step, from the routing of each (layer, batch) pair the steps use
    distinct = []
    with torch.cuda.stream(stream):
        for i in range(L * NX):
            ids.fill_(-1)
            step(i, stream, want_ids=True)
            stream.synchronize()
            lo, hi = int(ids.min()), int(ids.max())
            if lo < 0 or hi >= w["n_experts"]:  # every pick is an expert of the layer
                raise RuntimeError(f"{workload}: routing call {i} returned picks in [{lo}, {hi}]")
            distinct.append(int(torch.unique(ids).numel()))
    ffn.check(ffn.moe_workspace_status(ws, stream))
    G = L * NX * max(1, 24 // (L * NX))
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for i in range(G):
            step(i, stream)
    reps = max(1, steps // G)
    with torch.cuda.stream(stream):
        for _ in range(max(1, warmup // G)):
            g.replay()
    stream.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for _ in range(reps):
            g.replay()
        ev1.record(stream)
    ev1.synchronize()
    ffn.check(ffn.moe_workspace_status(ws, stream))
    n = reps * G
    ms = ev0.elapsed_time(ev1) / n
    step_bytes = prefill_bytes(w, statistics.mean(distinct))
    # end to end: pinned host x in, host out back, synchronised every step
    cfg_h = ffn.make_cfg(**{**w, "n_tokens": T, "flags": ffn.MOE_HOST_IO | ffn.MOE_GRAPH})
    wsh_bytes = ffn.moe_workspace_size(cfg_h)
    wsh = torch.zeros(wsh_bytes, dtype=torch.uint8, device=dev)
    xh = [x.cpu().pin_memory() for x in xs]
    oh = torch.empty((T, H), dtype=torch.float32).pin_memory()
    for i in range(2 * math.lcm(NX, L)):  # every pair twice: the second call captures its graph
        lay = layers[i % L]
        ffn.check(ffn.moe_ffn_forward_ex(xh[i % NX], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                         lay["shared_blocks"], cfg_h, oh, wsh, wsh_bytes, stream))
        stream.synchronize()
    xp, lp = bound_calls(ffn, layers, xh)
    op, wp, sp = oh.data_ptr(), wsh.data_ptr(), stream.cuda_stream
    t0 = time.perf_counter()
    for i in range(e2e_steps):
        ffn.check(ffn.moe_ffn_forward_ex(xp[i % NX], *lp[i % L], cfg_h, op, wp, wsh_bytes, sp))
        stream.synchronize()
    e2e = e2e_steps * T / (time.perf_counter() - t0)
    ffn.check(ffn.moe_workspace_status(wsh, stream))
    return {"workload": workload, "T": T, "value": round(T / (ms * 1e-3), 1), "unit": "tokens/s",
            "ms_per_step": ms, "steps": n, "layers_rotated": L, "distinct_experts_per_step": statistics.mean(distinct),
            "bytes_per_step": step_bytes, "launches_per_step": prefill_launches(w) * -(-T // 512), "e2e": round(e2e, 1), "e2e_steps": e2e_steps,
            "h2d_bytes_per_step": T * H * 4, "d2h_bytes_per_step": T * H * 4}


def sweep_tokens(args, ffn, synth, w, dev, layers_n=4, calls=8, reps=5):
    """Microseconds per call for each T of --sweep-tokens: the library's own path (decode
    below the batched threshold, the batched path from it) against T single-token calls.
    Each is a CUDA graph of `calls` calls over `layers_n` rotated layers, replayed `reps`
    times after a warm replay, timed with CUDA events on the replaying stream."""
    import torch
    layers = [synth.make_layer_torch(w, 100 + i, dev) for i in range(layers_n)]
    H = w["hidden"]
    st = torch.cuda.Stream(dev)
    table = {}
    for T in [int(v) for v in args.sweep_tokens.split(",") if v]:
        x = torch.randn(T, H, device=dev)
        out = torch.empty(T, H, device=dev)
        cfg_t = ffn.make_cfg(**{**w, "n_tokens": T})
        cfg_1 = ffn.make_cfg(**{**w, "n_tokens": 1})
        n_t, n_1 = ffn.moe_workspace_size(cfg_t), ffn.moe_workspace_size(cfg_1)
        ws_t = torch.zeros(n_t, dtype=torch.uint8, device=dev)
        ws_1 = torch.zeros(n_1, dtype=torch.uint8, device=dev)
        torch.cuda.synchronize(dev)  # before the side stream uses them

        def whole(i):
            lay = layers[i % layers_n]
            ffn.check(ffn.moe_ffn_forward_ex(x, lay["router_w"], lay["bias"], lay["expert_blocks"],
                                             lay["shared_blocks"], cfg_t, out, ws_t, n_t, st))

        def tokenwise(i):
            lay = layers[i % layers_n]
            for t in range(T):
                ffn.check(ffn.moe_ffn_forward_ex(x[t], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                                 lay["shared_blocks"], cfg_1, out[t], ws_1, n_1, st))

        row = {}
        for name, fn in (("library", whole), ("tokenwise", tokenwise)):
            with torch.cuda.stream(st):
                for i in range(3):
                    fn(i)
            st.synchronize()
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=st):
                for i in range(calls):
                    fn(i)
            with torch.cuda.stream(st):
                g.replay()
                e0 = torch.cuda.Event(enable_timing=True)
                e1 = torch.cuda.Event(enable_timing=True)
                e0.record(st)
                for _ in range(reps):
                    g.replay()
                e1.record(st)
            st.synchronize()
            row[name] = round(e0.elapsed_time(e1) * 1000 / (reps * calls), 1)
        table[T] = row
    print(json.dumps({"workload": args.workload, "us_per_call": table}))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=320, help="steps per timed repeat")
    ap.add_argument("--warmup", type=int, default=64)
    ap.add_argument("--min-ms", type=float, default=1500.0,
                    help="device time the headline's timed repeats add up to at least")
    ap.add_argument("--no-other-decode", action="store_true", help="skip the other decode workloads")
    ap.add_argument("--workload", default="flint_decode_t1")
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--layers", type=int, default=0, help="distinct layers to rotate (0 = auto)")
    ap.add_argument("--e2e-steps", type=int, default=3000)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-pdl", action="store_true")
    ap.add_argument("--f32-act", action="store_true",
                    help="decode with f32 activations in the block dots (MOE_F32_ACT) instead of the default "
                         "16-bit block fixed point")
    ap.add_argument("--prefill-steps", type=int, default=480, help="timed batched steps (0: skip)")
    ap.add_argument("--trace", action="store_true",
                    help="after timing, print the kernel's per-CTA phase timeline (stderr)")
    ap.add_argument("--sweep-tokens", default="",
                    help="comma-separated tokens per call: time one call of each on the workload's "
                         "layer (the library's choice of path against token-by-token decode), print the "
                         "table as JSON and exit")
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)

    rank, world, local = dist_setup(args.gpus)
    if args.impl == "reference":
        run_reference(args, rank, world)
        return

    import torch
    import expert_ffn_decode_gb300 as ffn
    from expert_ffn_decode_gb300 import synth

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if not os.path.exists(ffn.LIB_PATH):
        from expert_ffn_decode_gb300 import build
        build.build()
    w = synth.WORKLOADS[args.workload]
    T, H = w["n_tokens"], w["hidden"]
    if args.sweep_tokens:
        return sweep_tokens(args, ffn, synth, w, dev)
    if T != 1:
        return main_prefill(args, ffn, synth, dev, rank, world, local)
    step_bytes = layer_bytes(w)
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    layers, xs = decode_layers(synth, w, dev, rank, l2, args.layers)
    L, NX = len(layers), len(xs)
    base_flags = ffn.MOE_NO_PDL if args.no_pdl else 0
    flags = base_flags | (ffn.MOE_F32_ACT if args.f32_act else 0)
    stream = torch.cuda.Stream(dev)
    barrier(world)
    with ClockSampler(local) as clk:
        torch.cuda.synchronize()
        head = decode_timing(ffn, w, layers, xs, flags, dev, stream, args.steps, args.warmup, args.min_ms)
        # the other arithmetic of the decode chain, timed the same way (A/B)
        ab = decode_timing(ffn, w, layers, xs, flags ^ ffn.MOE_F32_ACT, dev, stream, args.steps,
                           args.warmup, args.min_ms / 4)
        torch.cuda.synchronize()
    ms_per_step = max_over_ranks(head["ms_per_step"], world, dev)
    value = T * world / (ms_per_step * 1e-3)
    ab_ms = max_over_ranks(ab["ms_per_step"], world, dev)
    others = {}
    if not args.no_other_decode:
        for name in OTHER_DECODE:
            if name == args.workload:
                continue
            wo = synth.WORKLOADS[name]
            lo, xo = decode_layers(synth, wo, dev, rank, l2)
            with ClockSampler(local) as clk_o:
                r = decode_timing(ffn, wo, lo, xo, flags, dev, stream, args.steps, args.warmup, args.min_ms / 4)
            r["ms_per_step"] = max_over_ranks(r["ms_per_step"], world, dev)
            r["value"] = round(wo["n_tokens"] * world / (r["ms_per_step"] * 1e-3), 1)
            r["unit"] = UNIT
            r["qtype"] = qtype_label(wo)
            r["clocks"] = clk_o.summary()
            others[name] = r
            del lo, xo
            torch.cuda.empty_cache()

    if args.trace:
        print_trace(ffn, w, layers, xs, L, NX, flags, dev, stream)
    chained_ms = max_over_ranks(bench_chained(ffn, w, layers, L, dev, stream, flags=flags), world, dev)

    # ---- end to end through the C ABI with host buffers (pinned) ----
    cfg_h = ffn.make_cfg(**{**w, "n_tokens": 1, "flags": flags | ffn.MOE_HOST_IO | ffn.MOE_GRAPH})
    wsh_bytes = ffn.moe_workspace_size(cfg_h)
    wsh = torch.zeros(wsh_bytes, dtype=torch.uint8, device=dev)
    xh = torch.empty((NX, H), dtype=torch.float32).pin_memory()
    xh.copy_(xs.cpu())
    oh = torch.empty((H,), dtype=torch.float32).pin_memory()
    n_e2e = args.e2e_steps
    torch.cuda.synchronize()
    # warm-up: every (token, layer) pair the timed calls use, twice (the library captures a
    # set's graph the second time it sees it)
    for i in range(2 * math.lcm(NX, L)):
        lay = layers[i % L]
        ffn.check(ffn.moe_ffn_forward_ex(xh[i % NX], lay["router_w"], lay["bias"], lay["expert_blocks"],
                                         lay["shared_blocks"], cfg_h, oh, wsh, wsh_bytes, stream))
        stream.synchronize()
    xp, lp = bound_calls(ffn, layers, [xh[j] for j in range(NX)])
    op, wp, sp = oh.data_ptr(), wsh.data_ptr(), stream.cuda_stream
    t0 = time.perf_counter()
    for i in range(n_e2e):
        rc = ffn.moe_ffn_forward_ex(xp[i % NX], *lp[i % L], cfg_h, op, wp, wsh_bytes, sp)
        if rc != 0:
            raise RuntimeError(ffn.moe_last_error())
        stream.synchronize()  # the step's result is on the host
    e2e_sec = time.perf_counter() - t0
    ffn.check(ffn.moe_workspace_status(wsh, stream))
    e2e_val = job_rate(n_e2e * T, e2e_sec, world, dev)

    pre = None
    pre_other = {}
    if args.prefill_steps > 0:
        pre = bench_prefill(ffn, synth, "flint_prefill_t512", dev, rank, args.prefill_steps, 24)
        reduce_prefill(pre, world, dev)
        for name in OTHER_PREFILL:
            pre_other[name] = bench_prefill(ffn, synth, name, dev, rank, args.prefill_steps, 24)
            reduce_prefill(pre_other[name], world, dev)
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    for p in [pre, *pre_other.values()]:
        if p is None:
            continue
        a = p["bytes_per_step"] / (p["ms_per_step"] * 1e-3) / 1e9
        pp = profile_counters(f"tile_gemm_{p['workload']}", "tile_gemm")
        p["roofline"] = {"bound": "hbm", "achieved": round(a, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(a / peak, 4), "peak_kind": peak_kind, "over": "the whole batched step",
                         "traffic": pp["dram_bytes_per_step"] if pp else None,
                         "tensor_pipe_active": pp["tensor_pipe_active"] if pp else None}
    prof = profile_counters(f"decode_chain_{args.workload}", "decode_chain")
    roof = decode_roofline(w, ms_per_step, peak, peak_kind)
    roof.update({"traffic": prof["dram_bytes_per_step"] if prof else None,
                 "kernel": "decode chain: dec_router -> dec_gate_up -> dec_down",
                 "over": "the whole step (three kernels overlapped by programmatic dependent launch)"})
    for name, r in others.items():
        r["roofline"] = decode_roofline(synth.WORKLOADS[name], r["ms_per_step"], peak, peak_kind)
        pr = profile_counters(f"decode_chain_{name}", "decode_chain")
        r["roofline"]["traffic"] = pr["dram_bytes_per_step"] if pr else None
    cpu = None
    if not args.no_cpu_baseline:
        d, err = cpu_baseline(args.workload)
        if d is not None:
            cpu = {"value": d["tokens"] / d["seconds"] * T, "unit": UNIT, "cores": 1, "kind": "oracle",
                   "sample": f"{d['tokens']} single-token oracle calls in {d['seconds']:.1f} s on one "
                             f"layer of the workload (numpy float64, one thread)"}
            # the same oracle with its numpy BLAS on every host core
            nproc = os.cpu_count() or 1
            d2, _ = cpu_baseline(args.workload, seconds=6.0, threads=nproc)
            if d2 is not None:
                cpu["all_cores"] = {"value": d2["tokens"] / d2["seconds"] * T, "cores": nproc,
                                    "sample": f"{d2['tokens']} calls in {d2['seconds']:.1f} s"}
        else:
            cpu = {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {err}"}
    clocks = clk.summary()
    fixed = not (flags & ffn.MOE_F32_ACT)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": ARITH_DTYPE[fixed], "data": "synthetic",
        "config": {"workload": args.workload, "T": T, "hidden": H, "n_experts": w["n_experts"],
                   "top_k": w["top_k"], "expert_ff": w["expert_ff"], "shared_ff": w["shared_ff"],
                   "qtype": qtype_label(w), "parallelism": f"replicas{world}",
                   "layers_rotated": L,
                   "l2": f"inputs larger than L2: {L} distinct layers, {L * step_bytes / 1e6:.0f} MB of "
                         f"step bytes between reuses of any weight byte (L2 {l2 / 1e6:.0f} MB)",
                   "pdl": not args.no_pdl},
        "timing": dict(head, how=f"{head['repeats']} timed repeats of exactly {args.steps} steps, run "
                                 f"{head['repeats_per_graph']} to a CUDA graph (one graph launch per "
                                 f"{head['repeats_per_graph'] * args.steps} steps), {head['replays']} replays each "
                                 f"between two CUDA events on the replaying stream, the layer rotation continuing "
                                 f"from repeat to repeat; ms_per_step is the median replay over its steps"),
        "arith": ARITH_TEXT[fixed],
        "roofline": roof,
        "ab_arith": {"dtype": ARITH_DTYPE[not fixed], "arith": ARITH_TEXT[not fixed], "ms_per_step": ab_ms,
                     "value": round(T * world / (ab_ms * 1e-3), 1), "unit": UNIT, "repeats": ab["repeats"],
                     "how": "the same steps with the decode chain's other activation arithmetic, timed the "
                            "same way right after the headline"},
        "decode_configs": others,
        "chained": {"ms_per_step": chained_ms, "value": round(T * world / (chained_ms * 1e-3), 1), "unit": UNIT,
                    "how": "x of layer l+1 = x_l + FFN(rms_norm(x_l) * norm): the residual form with the "
                           "norm prologue, each layer waiting on the last, same rotated layers, one CUDA graph"},
        "cpu_baseline": cpu,
        "e2e": {"value": round(e2e_val, 1), "unit": UNIT, "h2d_bytes_per_step": H * 4 * T,
                "d2h_bytes_per_step": H * 4 * T, "steps": n_e2e,
                "how": "moe_ffn_forward_ex with MOE_HOST_IO | MOE_GRAPH from pinned host memory (each "
                       "call one launch of the library's cached graph of its work), stream synchronised "
                       "every step"},
        "gpu_launches": 3 * args.steps * head["repeats"],
        "clocks": clocks,
        "prefill": pre,
        "prefill_configs": pre_other,
    }
    print(json.dumps(line))


def reduce_prefill(pre, world, dev):
    """A batched result over all ranks: the slowest rank's step time and e2e time, the
    tokens of every rank."""
    pre["ms_per_step"] = max_over_ranks(pre["ms_per_step"], world, dev)
    pre["value"] = round(pre["T"] * world / (pre["ms_per_step"] * 1e-3), 1)
    pre["e2e"] = round(job_rate(pre["T"], pre["T"] / pre["e2e"], world, dev), 1)


def main_prefill(args, ffn, synth, dev, rank, world, local):
    """The batched workload as the headline line."""
    import torch
    w = synth.WORKLOADS[args.workload]
    barrier(world)
    with ClockSampler(local) as clk:
        pre = bench_prefill(ffn, synth, args.workload, dev, rank, args.steps, args.warmup,
                            e2e_steps=min(args.e2e_steps, 50), layers=args.layers)
    reduce_prefill(pre, world, dev)
    ms = pre["ms_per_step"]
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    a = pre["bytes_per_step"] / (ms * 1e-3) / 1e9
    T = w["n_tokens"]
    pp = profile_counters(f"tile_gemm_{args.workload}", "tile_gemm")
    cpu = None
    if not args.no_cpu_baseline:
        d, err = cpu_baseline(args.workload, max_tokens=64)
        cpu = ({"value": d["tokens"] / d["seconds"], "unit": UNIT, "cores": 1, "kind": "oracle",
                "sample": f"{d['tokens']} single-token oracle calls of the workload's layer in {d['seconds']:.1f} s "
                          f"(numpy float64, one thread)"} if d is not None else
               {"value": None, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": f"failed: {err}"})
    line = {
        "metric": METRIC, "value": round(T * world / (ms * 1e-3), 1), "unit": UNIT, "n_gpus": world,
        "steps": pre["steps"], "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f16xf16->f32", "data": "synthetic",
        "config": {"workload": args.workload, "T": T, "hidden": w["hidden"], "n_experts": w["n_experts"],
                   "top_k": w["top_k"], "expert_ff": w["expert_ff"], "shared_ff": w["shared_ff"],
                   "qtype": qtype_label(w), "parallelism": f"replicas{world}",
                   "layers_rotated": pre["layers_rotated"],
                   "l2": "inputs larger than L2: every step reads over 400 MB of weights"},
        "roofline": {"bound": "hbm", "achieved": round(a, 1), "peak": peak, "unit": "GB/s", "frac": round(a / peak, 4),
                     "traffic": pp["dram_bytes_per_step"] if pp else None, "peak_kind": peak_kind,
                     "over": "the whole batched step", "bytes_per_launch": pre["bytes_per_step"],
                     "tensor_pipe_active": pp["tensor_pipe_active"] if pp else None},
        "cpu_baseline": cpu,
        "e2e": {"value": pre["e2e"], "unit": UNIT, "h2d_bytes_per_step": pre["h2d_bytes_per_step"],
                "d2h_bytes_per_step": pre["d2h_bytes_per_step"], "steps": pre["e2e_steps"]},
        "gpu_launches": pre["steps"] * pre["launches_per_step"],
        "clocks": clk.summary(),
        "detail": pre,
    }
    print(json.dumps(line))


if __name__ == "__main__":
    main()
