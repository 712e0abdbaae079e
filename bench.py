#!/usr/bin/env python3
"""Benchmark of the decode MoE-layer tail on GB300 (one JSON line on stdout).

Headline workload: the decode tail of one MoE layer at T=64 tokens, H=6144,
E=256 routed experts, top-8, one shared expert -- the router GEMM (BF16 x BF16
-> FP32 logits), then the fused tail: top-k routing (softmax over the top-8 x
2.5, ids and weights written out), finalize + shared add + residual add +
RMSNorm, in one launch.  One step is one layer; the steps walk through 75
distinct layers' buffers (gate weights, activations, expert rows: about 1 GB,
several times the L2), so every step reads cold HBM.  Steps are replayed from
a CUDA graph and timed with CUDA events on the launching stream.  The metric
is microseconds per layer (lower is better).  The same layer through the
three separate entry points (router, top-k, finalize) is reported beside it.

Extra keys: ``roofline`` (the dominant kernel's algorithmic GB/s against the
measured HBM copy peak), ``e2e`` (the same step with pinned-host inputs copied
in and outputs copied out inside the timed region), ``clocks``,
``cpu_baseline`` (the FP64 oracle on the host cores, a bounded sample) and
``sweep`` (decode / verify / prefill / partial-sum shapes, T = 1..8192).

``--impl reference`` times the CPU oracle on the same workload instead.
Multi-GPU (torchrun): every rank runs the same per-rank workload as an
independent replica (token rows need no exchange); the step time is the
maximum over ranks.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "µs/layer and HBM GB/s (% of GB300 peak) for fused MoE tail, T=1..8192"
UNIT = "µs/layer"
T_DEC, H_DEC, E_DEC, K_DEC, SCALE = 64, 6144, 256, 8, 2.5
N_LAYERS = 75  # distinct layer buffer sets the steps rotate through
WORKLOAD = ("decode tail T=64 H=6144 E=256 k=8 +1 shared expert: router GEMM -> fused tail (top-k route "
            "with ids and weights out, finalize+shared+residual+RMSNorm)")


def parse_args():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=3000)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-sweep", action="store_true", help="skip the T=1..8192 sweep")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--min-timed-s", type=float, default=1.0,
                    help="repeat the K-step timed region until this much time is covered")
    ap.add_argument("--ncu-case", choices=["decode", "decode1", "prefill", "router"], default=None,
                    help="run a small fixed case for an ncu capture and exit (no timing, no JSON)")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# algorithmic bytes (each input read once, each output written once)
# ---------------------------------------------------------------------------

def bytes_tail(T, H, k, shared=True, R=0, E=0, route_out=False):
    per_tok = k * H * 2 + (H * 2 if shared else 0) + H * 2 + 8 * k + 2 * H * 2 + R * H * 2
    if E:
        per_tok += 4 * E - 4 * k  # logits instead of the weights
        if route_out:
            per_tok += 8 * k
    return T * per_tok + 4 * H


def bytes_router(T, H, E):
    return E * H * 2 + T * H * 2 + T * E * 4


def bytes_route(T, E, k):
    return T * E * 4 + T * k * 8


# ---------------------------------------------------------------------------
# peaks, clocks, ncu traffic
# ---------------------------------------------------------------------------

def load_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi clock / throttle sampling while the timed region runs."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.path = None

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.index}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100", "-f", self.path], stdout=subprocess.DEVNULL, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()

    def summary(self):
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"samples": 0}

        def num(v):
            try:
                return float(v)
            except ValueError:
                return None
        sm = [num(r[1]) for r in rows if num(r[1]) is not None]
        smax = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower().startswith("active")})
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def source_digest(files):
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def ncu_traffic(kernel_tag, units_per_launch):
    """Per-launch DRAM bytes from the committed ncu summary of `kernel_tag`,
    scaled to `units_per_launch`; None if absent or the source changed since."""
    path = os.path.join(ROOT, "profiles", f"{kernel_tag}.md")
    if not os.path.exists(path):
        return None
    info = {}
    with open(path) as f:
        for line in f:
            if line.startswith("- ") and ": " in line:
                kk, vv = line[2:].split(": ", 1)
                info[kk.strip()] = vv.strip().strip("`")
    try:
        files = info["source_files"].split()
        if source_digest(files) != info["source_sha256"]:
            return None
        per_unit = float(info["dram_bytes_per_launch"]) / float(info["units_per_launch"])
        return per_unit * units_per_launch
    except Exception:
        return None


# ---------------------------------------------------------------------------
# timing helpers
# ---------------------------------------------------------------------------

def capture(torch, fn, stream):
    """CUDA graph of fn() captured on `stream` (after one eager warm-up run)."""
    with torch.cuda.stream(stream):
        fn()
    stream.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    return g


def time_replays(torch, graphs_and_counts, stream):
    """Replay [(graph, n)] in order once; returns elapsed ms (CUDA events)."""
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for g, n in graphs_and_counts:
            for _ in range(n):
                g.replay()
        e1.record(stream)
    e1.synchronize()
    return e0.elapsed_time(e1)


def graph_time_per_unit(torch, fn_per_set, nsets, stream, min_ms=150.0, min_reps=10):
    """Capture one graph that runs fn_per_set(i) for every buffer set i, then
    replay it until min_ms is covered; returns (median µs per set, p20, p80)."""
    g = capture(torch, lambda: [fn_per_set(i) for i in range(nsets)], stream)
    for _ in range(2):
        g.replay()
    stream.synchronize()
    per, total = [], 0.0
    while len(per) < min_reps or total < min_ms:
        ms = time_replays(torch, [(g, 1)], stream)
        per.append(ms * 1000.0 / nsets)
        total += ms
        if len(per) > 2000:
            break
    per.sort()
    q = lambda f: per[min(len(per) - 1, int(f * len(per)))]
    return statistics.median(per), q(0.2), q(0.8)


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------

def run_ours(args):
    import torch
    import torch.distributed as dist

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (there is no CPU path)")
    torch.cuda.set_device(local)
    if world > 1:
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))

    import moe_decode_layer_logits_gb300 as M
    from moe_decode_layer_logits_gb300.inputs import device_layer
    from moe_decode_layer_logits_gb300.sharding import max_over_ranks
    M.lib()

    dev = torch.device("cuda", local)
    stream = torch.cuda.Stream(device=dev)
    props = torch.cuda.get_device_properties(dev)
    l2 = getattr(props, "L2_cache_size", 126 * 2 ** 20) or 126 * 2 ** 20
    peak, peak_kind = load_peak()

    # -- headline buffers: 75 layers, each its own gate weight and activations
    layers = [device_layer(T_DEC, H_DEC, E_DEC, K_DEC, seed=1000 * rank + i, scale=SCALE) for i in range(N_LAYERS)]
    torch.cuda.synchronize()
    s = stream.cuda_stream

    def router(d):
        M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"], stream=s)

    def route(d):
        M.moe_topk_route(d["logits"], K_DEC, SCALE, topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)

    def finalize(d):
        M.moe_finalize_add_rmsnorm(d["rows"], d["map"], d["topk_w"], d["shared"], d["residual"], d["gamma"],
                                   d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"], stream=s)

    def fused_tail(d):
        M.moe_tail_fused(d["logits"], K_DEC, SCALE, d["rows"], d["map"], d["shared"], d["residual"], d["gamma"],
                         d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                         topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)

    def step(i):
        d = layers[i % N_LAYERS]
        router(d)
        fused_tail(d)

    def chain3_step(i):
        d = layers[i % N_LAYERS]
        router(d)
        route(d)
        finalize(d)

    # warm-up: W untimed steps (eager), then graphs
    for i in range(max(args.warmup, 3)):
        step(i)
    stream.synchronize()
    K = args.steps
    # Timed region: exactly K steps, step j on layer (first + j) mod 75.  With
    # K >= 75 a region walks every layer; with fewer steps each repeat of the
    # region starts where the previous one stopped, so consecutive regions
    # touch different layers and every step still reads cold HBM.
    plans = []
    if K >= N_LAYERS:
        g_full = capture(torch, lambda: [step(i) for i in range(N_LAYERS)], stream)
        rem = K % N_LAYERS
        g_rem = capture(torch, lambda: [step(i) for i in range(rem)], stream) if rem else None
        plans.append([(g_full, K // N_LAYERS)] + ([(g_rem, 1)] if g_rem else []))
    else:
        nwin = math.ceil(N_LAYERS / K)
        for w in range(nwin):
            gw = capture(torch, lambda w=w: [step(w * K + j) for j in range(K)], stream)
            plans.append([(gw, 1)])
    for _ in range(max(1, args.warmup // max(1, min(K, N_LAYERS)))):
        for pl in plans:
            for g, n in pl:
                g.replay()
    stream.synchronize()
    layers_per_region = min(K, N_LAYERS)
    layer_mb = bytes_router(T_DEC, H_DEC, E_DEC) / 1e6 + bytes_tail(T_DEC, H_DEC, K_DEC, E=E_DEC, route_out=True) / 1e6

    # -- timed region: exactly K steps, repeated to cover --min-timed-s
    times = []
    with ClockSampler(local) as clk:
        while len(times) < 3 or sum(times) < args.min_timed_s * 1000.0:
            if world > 1:
                dist.barrier()
            torch.cuda.synchronize()
            ms = time_replays(torch, plans[len(times) % len(plans)], stream)
            torch.cuda.synchronize()
            if world > 1:
                dist.barrier()
            times.append(max_over_ranks(ms))
            if len(times) >= 200:
                break
    clocks = clk.summary()
    ms_region = statistics.median(times)
    us_layer = ms_region * 1000.0 / K

    # -- per-kernel device time (each kernel alone, same cold rotation)
    kern = {}
    kern["fused_tail"] = graph_time_per_unit(torch, lambda i: fused_tail(layers[i]), N_LAYERS, stream)
    kern["router"] = graph_time_per_unit(torch, lambda i: router(layers[i]), N_LAYERS, stream)
    kern["route"] = graph_time_per_unit(torch, lambda i: route(layers[i]), N_LAYERS, stream)
    kern["finalize"] = graph_time_per_unit(torch, lambda i: finalize(layers[i]), N_LAYERS, stream)
    b = {"fused_tail": bytes_tail(T_DEC, H_DEC, K_DEC, E=E_DEC, route_out=True),
         "router": bytes_router(T_DEC, H_DEC, E_DEC), "route": bytes_route(T_DEC, E_DEC, K_DEC),
         "finalize": bytes_tail(T_DEC, H_DEC, K_DEC)}
    dom = max(("fused_tail", "router"), key=lambda n: kern[n][0])  # the headline step's two kernels
    dom_us = kern[dom][0]
    achieved = b[dom] / (dom_us * 1e-6) / 1e9
    tag = {"fused_tail": "tail_kernel_fused_decode_T64", "router": "router_kernel_decode_T64"}[dom]
    traffic = ncu_traffic(tag, T_DEC)

    # -- the same layer through the three separate entry points
    chain3_us = graph_time_per_unit(torch, chain3_step, N_LAYERS, stream)

    # -- L2-warm figures: the same layer replayed on one buffer set (labelled
    #    apart from the cold headline)
    warm = {}
    d0 = layers[0]
    warm["decode_layer_T64"] = graph_time_per_unit(torch, lambda i: (router(d0), fused_tail(d0)), 20, stream)[0]
    warm["router_T64"] = graph_time_per_unit(torch, lambda i: router(d0), 20, stream)[0]
    warm["fused_tail_T64"] = graph_time_per_unit(torch, lambda i: fused_tail(d0), 20, stream)[0]

    # -- the router at every decode size: cold (75 distinct gate weights) and
    #    warm, with the gate-weight read rate (the router's dominant bytes)
    router_dec = run_router_decode(torch, M, stream, layers)
    for T, dd in router_dec.items():
        if T != T_DEC:
            warm[f"decode_layer_T{T}"] = dd.pop("warm_layer_us")
    warm = {k: round(v, 3) for k, v in warm.items()}

    # -- end to end through the C ABI with pinned host buffers
    e2e = run_e2e(torch, M, layers, stream, K, args.warmup)

    del layers
    torch.cuda.empty_cache()
    sweep = None if args.no_sweep else run_sweep(torch, M, stream, l2, peak)

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline()

    line = {
        "metric": METRIC, "value": round(us_layer, 4), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": round(us_layer / 1000.0, 7), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "fp32", "io_dtype": "bf16", "data": "synthetic",
        "config": {"workload": WORKLOAD, "T": T_DEC, "H": H_DEC, "E": E_DEC, "k": K_DEC, "routed_scale": SCALE,
                   "layers_rotated": N_LAYERS, "layers_per_timed_region": layers_per_region,
                   "l2": (f"cold: each timed region of {K} steps walks {layers_per_region} distinct layers "
                          f"({layers_per_region * layer_mb:.0f} MB of algorithmic bytes; {N_LAYERS} layers, "
                          f"{N_LAYERS * layer_mb:.0f} MB, across repeats) against an L2 of {l2 / 2**20:.0f} MB"),
                   "timing": "CUDA-graph replay, CUDA events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "repeats": len(times), "gpu_launches": 2 * K,
        "clocks": clocks,
        "roofline": {"kernel": dom, "bound": "hbm", "achieved": round(achieved, 1), "peak": peak,
                     "peak_kind": f"{peak_kind} (hbm_gbs)", "unit": "GB/s", "frac": round(achieved / peak, 4),
                     "algorithmic_bytes_per_launch": b[dom], "launch_us": round(dom_us, 3),
                     "traffic": None if traffic is None else round(traffic)},
        "kernels_us": {n: {"median": round(v[0], 3), "p20": round(v[1], 3), "p80": round(v[2], 3),
                           "GBps": round(b[n] / (v[0] * 1e-6) / 1e9, 1)} for n, v in kern.items()},
        "router_decode": {str(T): v for T, v in router_dec.items()},
        "l2_warm_us": {**warm, "what": "the same step or kernel replayed on one buffer set (the inputs stay in the "
                                       "L2); the headline and kernels_us rotate cold buffers"},
        "three_launch_chain_us_per_layer": {"median": round(chain3_us[0], 3), "p20": round(chain3_us[1], 3),
                                            "p80": round(chain3_us[2], 3),
                                            "what": "router GEMM -> top-k route -> finalize (3 launches)"},
        "e2e": e2e,
        "cpu_baseline": cpu,
        "sweep": sweep,
    }
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        dist.barrier()
        dist.destroy_process_group()


def run_router_decode(torch, M, stream, layers64):
    """The router GEMM at T = 1, 4, 64 over 75 distinct gate weights (cold),
    with the gate-weight read rate, plus (T = 1, 4) the warm decode layer."""
    from moe_decode_layer_logits_gb300.inputs import device_layer
    s = stream.cuda_stream
    out = {}
    for T in (1, 4, T_DEC):
        sets = layers64 if T == T_DEC else [device_layer(T, H_DEC, E_DEC, K_DEC, seed=5000 + i, scale=SCALE)
                                            for i in range(N_LAYERS)]
        torch.cuda.synchronize()

        def rtr(d):
            M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"], stream=s)
        med, p20, p80 = graph_time_per_unit(torch, lambda i: rtr(sets[i]), len(sets), stream)
        wb = E_DEC * H_DEC * 2
        entry = {"us": round(med, 3), "p20": round(p20, 3), "p80": round(p80, 3),
                 "weight_read_GBps": round(wb / (med * 1e-6) / 1e9, 1),
                 "GBps": round(bytes_router(T, H_DEC, E_DEC) / (med * 1e-6) / 1e9, 1),
                 "TFLOPs": round(2.0 * T * E_DEC * H_DEC / (med * 1e-6) / 1e12, 2)}
        if T != T_DEC:
            d0 = sets[0]

            def layer(i):
                rtr(d0)
                M.moe_tail_fused(d0["logits"], K_DEC, SCALE, d0["rows"], d0["map"], d0["shared"], d0["residual"],
                                 d0["gamma"], d0["eps"], residual_out=d0["residual_out"], normed_out=d0["normed_out"],
                                 topk_ids=d0["topk_ids"], topk_w=d0["topk_w"], stream=s)
            entry["warm_layer_us"] = graph_time_per_unit(torch, layer, 20, stream)[0]
        out[T] = entry
        if T != T_DEC:
            del sets
    return out


def run_e2e(torch, M, layers, stream, K, warmup):
    """Same step with host buffers, as a serving loop would run it: every step
    copies its activations (x, expert rows, map, shared, residual) from one
    pinned host staging buffer to the device in a single copy, makes the two
    C-ABI calls (router, fused tail), and copies both outputs back to pinned host memory in a
    single copy.  Copies in, compute and copies out run on three streams with
    events between them (step i+1's input copy overlaps step i's compute); 8
    device buffer sets rotate; 8 steps are captured in one CUDA graph and the
    graph is replayed.  Gate weights and gamma stay resident (model
    parameters).  Timed with events around the replays, which include every
    copy in and out."""
    d0 = layers[0]
    names_in = ["x", "rows", "map", "shared", "residual"]
    names_out = ["residual_out", "normed_out"]

    def layout(names):
        offs, o = {}, 0
        for n in names:
            offs[n] = o
            o += (d0[n].numel() * d0[n].element_size() + 255) // 256 * 256
        return offs, o

    offs_in, n_in = layout(names_in)
    offs_out, n_out = layout(names_out)

    def views(buf, offs, names):
        v = {}
        for n in names:
            nb = d0[n].numel() * d0[n].element_size()
            v[n] = buf[offs[n]:offs[n] + nb].view(d0[n].dtype).view(d0[n].shape)
        return v

    host_in = torch.empty(n_in, dtype=torch.uint8).pin_memory()
    hv = views(host_in, offs_in, names_in)
    for n in names_in:
        hv[n].copy_(d0[n].cpu())
    host_out = torch.empty(n_out, dtype=torch.uint8).pin_memory()
    nsets = 8
    dev = d0["x"].device
    dev_in = [torch.empty(n_in, dtype=torch.uint8, device=dev) for _ in range(nsets)]
    dev_out = [torch.empty(n_out, dtype=torch.uint8, device=dev) for _ in range(nsets)]
    dvi = [views(b, offs_in, names_in) for b in dev_in]
    dvo = [views(b, offs_out, names_out) for b in dev_out]
    h2d = sum(hv[n].numel() * hv[n].element_size() for n in names_in)
    d2h = sum(d0[n].numel() * d0[n].element_size() for n in names_out)
    s_in, s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
    s = stream.cuda_stream

    def steps(n):
        # step j: copy in on s_in, compute on `stream`, copy out on s_out
        s_in.wait_stream(stream)
        s_out.wait_stream(stream)
        for j in range(n):
            d = layers[j % len(layers)]
            a, o = dvi[j % nsets], dvo[j % nsets]
            with torch.cuda.stream(s_in):
                dev_in[j % nsets].copy_(host_in, non_blocking=True)
            stream.wait_stream(s_in)
            with torch.cuda.stream(stream):
                M.moe_router_logits_fp32(a["x"], d["w_gate"], logits_out=d["logits"], stream=s)
                M.moe_tail_fused(d["logits"], K_DEC, SCALE, a["rows"], a["map"], a["shared"], a["residual"],
                                 d["gamma"], d["eps"], residual_out=o["residual_out"], normed_out=o["normed_out"],
                                 topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)
            s_out.wait_stream(stream)
            with torch.cuda.stream(s_out):
                host_out.copy_(dev_out[j % nsets], non_blocking=True)
        stream.wait_stream(s_in)
        stream.wait_stream(s_out)

    # a serving loop replays captured steps: one graph of `nsets` steps
    with torch.cuda.stream(stream):
        steps(nsets)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        steps(nsets)
    reps = max(1, (min(K, 750) + nsets - 1) // nsets)
    n_steps = reps * nsets
    for _ in range(max(1, warmup // nsets)):
        g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(reps):
            g.replay()
        e1.record(stream)
    e1.synchronize()
    us = e0.elapsed_time(e1) * 1000.0 / n_steps
    return {"value": round(us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "steps": n_steps,
            "what": "per step: one pinned host -> device copy of the activations, 2 C-ABI calls, one device -> "
                    "pinned host copy of both outputs; copies in / compute / copies out on three streams, "
                    "8 steps per captured graph"}


def run_sweep(torch, M, stream, l2, peak):
    """µs and GB/s of the tail over the decode / verify / prefill / partials shapes."""
    from moe_decode_layer_logits_gb300.inputs import device_layer
    s = stream.cuda_stream
    out = []

    def nsets_for(set_bytes):
        return int(min(N_LAYERS, max(2, math.ceil(3 * l2 / set_bytes))))

    def add(name, T, H, fn, nb, sets):
        med, p20, p80 = graph_time_per_unit(torch, lambda i: fn(sets[i]), len(sets), stream, min_ms=100.0)
        gbs = nb / (med * 1e-6) / 1e9
        out.append({"case": name, "T": T, "H": H, "us": round(med, 3), "p20": round(p20, 3), "p80": round(p80, 3),
                    "GBps": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4), "bytes": nb})

    # decode + verify layers: full path (router -> route -> finalize) and fused
    for T, H in [(1, 6144), (4, 6144), (64, 6144), (12, 6144), (28, 6144), (12, 2048), (28, 2048)]:
        nb = bytes_router(T, H, E_DEC) + bytes_route(T, E_DEC, K_DEC) + bytes_tail(T, H, K_DEC)
        sets = [device_layer(T, H, E_DEC, K_DEC, seed=7000 + i, scale=SCALE) for i in range(nsets_for(nb))]
        torch.cuda.synchronize()  # the buffers are drawn on torch's stream; the kernels run on `stream`

        def full(d):
            M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"], stream=s)
            M.moe_topk_route(d["logits"], K_DEC, SCALE, topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)
            M.moe_finalize_add_rmsnorm(d["rows"], d["map"], d["topk_w"], d["shared"], d["residual"], d["gamma"],
                                       d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                                       stream=s)

        def fin(d):
            M.moe_finalize_add_rmsnorm(d["rows"], d["map"], d["topk_w"], d["shared"], d["residual"], d["gamma"],
                                       d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                                       stream=s)

        def fusedl(d):
            M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"], stream=s)
            M.moe_tail_fused(d["logits"], K_DEC, SCALE, d["rows"], d["map"], d["shared"], d["residual"],
                             d["gamma"], d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                             topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)
        nbf = bytes_router(T, H, E_DEC) + bytes_tail(T, H, K_DEC, E=E_DEC, route_out=True)
        add("decode layer: router+fused tail", T, H, fusedl, nbf, sets)
        add("decode layer: router+route+finalize", T, H, full, nb, sets)
        add("finalize+shared+residual+RMSNorm", T, H, fin, bytes_tail(T, H, K_DEC), sets)
        del sets
    # prefill: router-less fused tail on supplied logits, and finalize alone
    for T in [512, 2048, 8192]:
        H = 6144
        nb = bytes_tail(T, H, K_DEC, E=E_DEC)
        sets = [device_layer(T, H, E_DEC, K_DEC, seed=8000 + i, scale=SCALE, router=False, logits=True)
                for i in range(nsets_for(nb))]
        torch.cuda.synchronize()
        for d in sets:
            M.moe_topk_route(d["logits"], K_DEC, SCALE, topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)

        def fused(d):
            M.moe_tail_fused(d["logits"], K_DEC, SCALE, d["rows"], d["map"], d["shared"], d["residual"],
                             d["gamma"], d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                             want_route=False, stream=s)

        def fin(d):
            M.moe_finalize_add_rmsnorm(d["rows"], d["map"], d["topk_w"], d["shared"], d["residual"], d["gamma"],
                                       d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                                       stream=s)
        add("prefill fused tail (logits supplied)", T, H, fused, nb, sets)
        add("finalize+shared+residual+RMSNorm", T, H, fin, bytes_tail(T, H, K_DEC), sets)
        del sets
        torch.cuda.empty_cache()
    # router GEMM at prefill sizes (a dense contraction near the tensor ridge)
    for T in [512, 2048, 8192]:
        H = H_DEC
        nb = bytes_router(T, H, E_DEC)
        sets = [device_layer(T, H, E_DEC, 1, seed=9500 + i, shared=False, router=True)
                for i in range(nsets_for(nb))]
        torch.cuda.synchronize()

        def rtr(d):
            M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"], stream=s)
        add("router GEMM (BF16 -> FP32 logits)", T, H, rtr, nb, sets)
        out[-1]["TFLOPs"] = round(2.0 * T * E_DEC * H / (out[-1]["us"] * 1e-6) / 1e12, 1)
        del sets
        torch.cuda.empty_cache()
    # E = 168, the real checkpoint's expert count, beside the E = 256 rows
    for T in [64, 8192]:
        H, E = H_DEC, 168
        k = K_DEC if T == 64 else 1
        nb = bytes_router(T, H, E)
        nbl = nb + (bytes_tail(T, H, K_DEC, E=E, route_out=True) if T == 64 else 0)
        sets = [device_layer(T, H, E, k, seed=9700 + i, shared=T == 64, router=True, scale=SCALE)
                for i in range(nsets_for(nbl))]
        torch.cuda.synchronize()

        def rtr(d):
            M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"], stream=s)
        add("router GEMM E=168 (BF16 -> FP32 logits)", T, H, rtr, nb, sets)
        out[-1]["TFLOPs"] = round(2.0 * T * E * H / (out[-1]["us"] * 1e-6) / 1e12, 1)
        if T == 64:
            def layer168(d):
                rtr(d)
                M.moe_tail_fused(d["logits"], K_DEC, SCALE, d["rows"], d["map"], d["shared"], d["residual"],
                                 d["gamma"], d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                                 topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)
            add("decode layer E=168: router+fused tail", T, H, layer168, nbl, sets)
        del sets
        torch.cuda.empty_cache()
    # rows in the expert-grouped layout an expert GEMM writes (groups padded to
    # 128 rows) instead of a random permutation: same bytes, other addresses
    T, H = 2048, 6144
    nb = bytes_tail(T, H, K_DEC)
    sets = [device_layer(T, H, E_DEC, K_DEC, seed=9800 + i, scale=SCALE, router=False, logits=True,
                         map_layout="expert_sorted", expert_block=128) for i in range(nsets_for(nb))]
    torch.cuda.synchronize()
    for d in sets:
        M.moe_topk_route(d["logits"], K_DEC, SCALE, topk_ids=d["topk_ids"], topk_w=d["topk_w"], stream=s)

    def fin_sorted(d):
        M.moe_finalize_add_rmsnorm(d["rows"], d["map"], d["topk_w"], d["shared"], d["residual"], d["gamma"],
                                   d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"], stream=s)
    add("finalize+shared+residual+RMSNorm, expert-grouped rows", T, H, fin_sorted, nb, sets)
    del sets
    torch.cuda.empty_cache()
    # row-parallel partials: R=4 local partial buffers replace gather + shared
    for T in [1, 64, 2048]:
        H = 6144
        nb = bytes_tail(T, H, 0, shared=False, R=4)
        sets = [device_layer(T, H, E_DEC, 0, seed=9000 + i, shared=False, R=4, router=False)
                for i in range(nsets_for(nb))]
        torch.cuda.synchronize()

        def part(d):
            M.moe_finalize_add_rmsnorm(None, None, None, None, d["residual"], d["gamma"], d["eps"],
                                       partials=d["partials"], residual_out=d["residual_out"],
                                       normed_out=d["normed_out"], stream=s)
        add("R=4 partials+residual+RMSNorm", T, H, part, nb, sets)
        del sets
        torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle legs
# ---------------------------------------------------------------------------

_CPU_ENV = {"OMP_NUM_THREADS": "1", "OPENBLAS_NUM_THREADS": "1", "MKL_NUM_THREADS": "1"}

# The oracle's per-config baseline: (name, kind, T, H, E, k, routed scale, R,
# shared expert, tokens in the sample).  kind "layer": router -> top-k ->
# tail; "prefill": top-k on supplied logits -> tail; "partials": R partial
# buffers + residual + RMSNorm.  Large batches are timed on a token sample
# and scaled to the batch (the oracle's cost per token does not depend on T).
ORACLE_CONFIGS = [
    ("tiny T=4 H=2048 E=64 k=4", "layer", 4, 2048, 64, 4, 1.0, 0, True, 4),
    ("decode T=1", "layer", 1, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 1),
    ("decode T=4", "layer", 4, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 4),
    ("decode T=64", "layer", 64, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 64),
    ("verify T=4 H=6144", "layer", 4, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 4),
    ("verify T=12 H=6144", "layer", 12, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 12),
    ("verify T=28 H=6144", "layer", 28, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 28),
    ("verify T=4 H=2048", "layer", 4, 2048, E_DEC, K_DEC, SCALE, 0, True, 4),
    ("verify T=12 H=2048", "layer", 12, 2048, E_DEC, K_DEC, SCALE, 0, True, 12),
    ("verify T=28 H=2048", "layer", 28, 2048, E_DEC, K_DEC, SCALE, 0, True, 28),
    ("prefill T=512", "prefill", 512, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 128),
    ("prefill T=2048", "prefill", 2048, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 128),
    ("prefill T=8192", "prefill", 8192, H_DEC, E_DEC, K_DEC, SCALE, 0, True, 128),
    ("partials T=1 R=4", "partials", 1, H_DEC, E_DEC, 0, SCALE, 4, False, 1),
    ("partials T=64 R=4", "partials", 64, H_DEC, E_DEC, 0, SCALE, 4, False, 64),
    ("partials T=2048 R=4", "partials", 2048, H_DEC, E_DEC, 0, SCALE, 4, False, 128),
]

_ORACLE_CACHE = {}


def _oracle_case(cfg):
    """Inputs of one oracle-baseline config in a worker (drawn once)."""
    key = tuple(cfg)
    if key not in _ORACLE_CACHE:
        sys.path.insert(0, ROOT)
        from moe_decode_layer_logits_gb300.inputs import tail_case
        _, kind, T, H, E, k, scale, R, shared, ns = cfg
        _ORACLE_CACHE[key] = tail_case(ns, H, E, k, seed=1, scale=scale, R=R, shared=shared,
                                       router=kind == "layer", logits=kind == "prefill", weights=False)
    return _ORACLE_CACHE[key]


def _oracle_init(configs):
    """Pool initializer: every worker draws every config's inputs up front,
    so no timed call draws or imports anything."""
    sys.path.insert(0, ROOT)
    import oracle  # noqa: F401
    for cfg in configs:
        _oracle_case(cfg)


def _oracle_shard(task):
    """One worker's share of an oracle layer: tokens [a, b) of the sample."""
    cfg, a, b = task
    import oracle as O
    c = _oracle_case(cfg)
    kind, k, scale = cfg[1], cfg[5], cfg[6]
    tok = slice(a, b)
    if kind == "partials":
        O.finalize_add_rmsnorm(None, c["map"][tok], c["map"][tok].astype("float32"), None, c["partials"][:, tok],
                               c["residual"][tok], c["gamma"], c["eps"])
        return b - a
    if kind == "layer":
        L, _ = O.router_logits(c["x"][tok], c["w_gate"])
        lg = L.astype("float32")
    else:
        lg = c["logits"][tok]
    _, w32, _ = O.topk_route(lg, k, scale)
    sh = None if c["shared"] is None else c["shared"][tok]
    O.finalize_add_rmsnorm(c["rows"], c["map"][tok], w32, sh, None, c["residual"][tok], c["gamma"], c["eps"])
    return b - a


def _oracle_child(spec):
    """Runs in a fresh process: a spawn pool of `cores` single-threaded
    workers; each timed layer splits its token sample over the workers.
    Prints one JSON line per config."""
    import multiprocessing as mp
    ctx = mp.get_context("spawn")
    cores = spec["cores"]
    with ctx.Pool(cores, initializer=_oracle_init, initargs=([tuple(c) for c in spec["configs"]],)) as pool:
        for cfg in spec["configs"]:
            ns = cfg[-1]
            n = max(1, min(cores, ns))
            bounds = [(tuple(cfg), ns * i // n, ns * (i + 1) // n) for i in range(n)]
            for _ in range(max(1, spec.get("warm", 1))):
                pool.map(_oracle_shard, bounds)  # draws the inputs in every worker once
            times, reps, t_all = [], spec.get("reps", 3), time.perf_counter()
            while len(times) < reps or (spec.get("budget_s") and time.perf_counter() - t_all < spec["budget_s"]):
                t0 = time.perf_counter()
                pool.map(_oracle_shard, bounds)
                times.append(time.perf_counter() - t0)
                if spec.get("max_reps") and len(times) >= spec["max_reps"]:
                    break
            T = cfg[2]
            print(json.dumps({"config": cfg[0], "s_per_layer": statistics.median(times) * T / ns,
                              "reps": len(times), "sample_tokens": ns, "T": T, "workers": n,
                              "timed_s": sum(times)}), flush=True)


def run_oracle_child(configs, cores=None, reps=3, warm=1, budget_s=None, max_reps=None):
    """Launch _oracle_child in a fresh interpreter; returns its JSON lines."""
    cores = cores or os.cpu_count() or 1
    spec = {"configs": configs, "cores": cores, "reps": reps, "warm": warm, "budget_s": budget_s,
            "max_reps": max_reps}
    env = dict(os.environ, **_CPU_ENV)
    r = subprocess.run([sys.executable, os.path.abspath(__file__), "--oracle-child", json.dumps(spec)], env=env,
                       capture_output=True, text=True)
    if r.returncode != 0:
        return None, (r.stderr.strip().splitlines() or ["oracle failed"])[-1], cores
    return [json.loads(l) for l in r.stdout.strip().splitlines() if l.startswith("{")], None, cores


def cpu_baseline():
    """The FP64 oracle on the host cores: the headline decode layer (T=64)
    and every workload config, each layer's tokens split over a spawn pool of
    single-threaded workers (one per core)."""
    rows, err, cores = run_oracle_child(ORACLE_CONFIGS, reps=5)
    if rows is None:
        return {"error": err}
    per = {r["config"]: {"us_per_layer": round(r["s_per_layer"] * 1e6, 1), "sample_tokens": r["sample_tokens"],
                         "T": r["T"], "workers": r["workers"]} for r in rows}
    head = per["decode T=64"]
    return {"value": head["us_per_layer"], "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"decode layer T=64 (H=6144, E=256, k=8): all 64 tokens split over {head['workers']} "
                       f"single-threaded FP64 numpy workers (spawn pool, one per host core), median of 5 layers; "
                       f"prefill and large partial configs timed on a 128-token sample and scaled"),
            "per_config": per}


def run_reference(args):
    """The oracle as it stands, on this workload: W untimed + exactly K timed
    layers of the decode step (T=64), each split over the host cores."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    cfg = [c for c in ORACLE_CONFIGS if c[0] == "decode T=64"]
    rows, err, cores = run_oracle_child(cfg, reps=max(1, args.steps), warm=max(1, args.warmup), max_reps=args.steps)
    if rows is None:
        print(json.dumps({"impl": "reference", "unavailable": f"oracle failed: {err}"}), flush=True)
        return
    r = rows[0]
    v = round(r["s_per_layer"] * 1e6, 1)
    res = {"value": v, "unit": UNIT, "cores": cores, "kind": "oracle",
           "sample": (f"{r['reps']} decode layers of 64 tokens (H=6144, E=256, k=8), FP64 numpy, tokens split over "
                      f"{r['workers']} single-threaded workers, {r['timed_s']:.1f} s timed")}
    line = {"impl": "reference", "metric": METRIC, "value": v, "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": v / 1000.0,
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": WORKLOAD, "T": T_DEC, "H": H_DEC, "E": E_DEC, "k": K_DEC,
                       "routed_scale": SCALE},
            "cpu_baseline": res,
            "e2e": {"value": v, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def run_ncu_case(case):
    """Small cases for ncu captures (a few hundred MB, more than the L2):
    decode -- 12 layers at T=64 (162 MB), router -> route -> finalize -> fused
    tail on each layer, twice; decode1 -- the same with 48 layers at T=1
    (154 MB, mostly gate weights); prefill -- 2 sets at T=2048 (605 MB), route, finalize and the
    router-less fused tail on each set, twice; router -- the router GEMM on 2
    inputs at T=8192 (x 100 MB each), twice."""
    import torch
    import moe_decode_layer_logits_gb300 as M
    from moe_decode_layer_logits_gb300.inputs import device_layer
    M.lib()
    if case == "router":
        # 2 router inputs at T=8192 (x 100 MB each): the tensor-memory router kernel, twice each
        sets = [device_layer(8192, H_DEC, E_DEC, 1, seed=200 + i, shared=False) for i in range(2)]
        torch.cuda.synchronize()
        for _ in range(2):
            for d in sets:
                M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"])
        torch.cuda.synchronize()
        return
    if case == "decode":
        sets = [device_layer(T_DEC, H_DEC, E_DEC, K_DEC, seed=i, scale=SCALE) for i in range(12)]
    elif case == "decode1":
        sets = [device_layer(1, H_DEC, E_DEC, K_DEC, seed=i, scale=SCALE) for i in range(48)]
    else:
        sets = [device_layer(2048, H_DEC, E_DEC, K_DEC, seed=100 + i, scale=SCALE, router=False, logits=True)
                for i in range(2)]
    torch.cuda.synchronize()
    for _ in range(2):
        for d in sets:
            if case in ("decode", "decode1"):
                M.moe_router_logits_fp32(d["x"], d["w_gate"], logits_out=d["logits"])
            M.moe_topk_route(d["logits"], K_DEC, SCALE, topk_ids=d["topk_ids"], topk_w=d["topk_w"])
            M.moe_finalize_add_rmsnorm(d["rows"], d["map"], d["topk_w"], d["shared"], d["residual"], d["gamma"],
                                       d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"])
            if case in ("decode", "decode1"):
                M.moe_tail_fused(d["logits"], K_DEC, SCALE, d["rows"], d["map"], d["shared"], d["residual"],
                                 d["gamma"], d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                                 topk_ids=d["topk_ids"], topk_w=d["topk_w"])
            if case == "prefill":
                M.moe_tail_fused(d["logits"], K_DEC, SCALE, d["rows"], d["map"], d["shared"], d["residual"],
                                 d["gamma"], d["eps"], residual_out=d["residual_out"], normed_out=d["normed_out"],
                                 want_route=False)
    torch.cuda.synchronize()


def main():
    if len(sys.argv) == 3 and sys.argv[1] == "--oracle-child":
        _oracle_child(json.loads(sys.argv[2]))
        return
    args = parse_args()
    if args.ncu_case:
        run_ncu_case(args.ncu_case)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
