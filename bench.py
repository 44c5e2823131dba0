#!/usr/bin/env python
"""Benchmark of the OEA MoE decode layer on GB300.

A step is one pass of the whole layer (router, routing, grouped SwiGLU
experts, combine) over one decode batch.  Steps cycle through 8 layers with
distinct seeded weights (about 1.2 GB of expert weights per layer at the
Qwen3-30B-A3B shapes, far larger than the 126 MB L2), so every step streams
its activated experts from HBM.

value     = algorithmic bytes / device time for the headline routing run
            (whole job: summed over ranks, divided by the slowest rank's
            time).  Algorithmic bytes per layer = T * 3*d*d_ff*2 (the
            activated experts, read once) + the router weights
            N*d*2 + activations (x read twice, scores, output).
roofline  = the expert kernel alone: its algorithmic bytes per launch over
            its mean launch time (CUDA events on the launching stream,
            recorded around every launch in a second timed pass of the same
            steps; the headline pass has events only at its two ends),
            against the measured HBM copy bandwidth.
e2e       = the same metric through moe_decode_layer with host buffers: the
            step's hidden states are copied from pinned host memory and the
            output read back inside the timed region.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--sweep-out FILE]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import synth  # noqa: E402

METRIC = "MoE decode layer µs & HBM GB/s (T·expert bytes roofline) vs B, OEA vs top-k"
UNIT = "GB/s"
DEFAULT_WORKLOAD = "qwen3_30b_a3b_uniform_b16"
HEADLINE = {"qwen3_30b_a3b_uniform_b16": "oea_k0_3", "qwen3_30b_a3b_zipf_sweep": "oea_k0_5_p0.7",
            "qwen3_235b_a22b_zipf_b64": "oea_k0_5_p0.7", "qwen3_30b_a3b_mixed_int4_b32": "oea_k0_5"}
N_LAYERS = 8          # default rotation; --layers changes it


def log(*a):
    print(*a, file=sys.stderr, flush=True)


# ---------------------------------------------------------------------------
# byte accounting
# ---------------------------------------------------------------------------
def expert_kernel_bytes(w: synth.Workload, B: int, T: float) -> float:
    """Algorithmic bytes of one expert-kernel launch: activated experts once,
    hidden states in, output out."""
    return T * w.expert_bytes + 2 * B * w.d * 2


def layer_bytes(w: synth.Workload, B: int, T: float) -> float:
    router = w.N * w.d * 2 + B * w.d * 2 + B * w.N * 4
    return router + expert_kernel_bytes(w, B, T)


def mixed_kernel_bytes(w: synth.Workload, B: int, n_hot_active: int, n_cold_active: int) -> float:
    """Expert-kernel bytes with bf16 hot and INT4 cold experts."""
    return (n_hot_active * w.expert_bytes + n_cold_active * synth.int4_expert_bytes(w.d, w.F)
            + 2 * B * w.d * 2)


def mixed_layer_bytes(w: synth.Workload, B: int, n_hot_active: int, n_cold_active: int) -> float:
    return w.N * w.d * 2 + B * w.d * 2 + B * w.N * 4 + mixed_kernel_bytes(w, B, n_hot_active, n_cold_active)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def expert_kernel(w: synth.Workload) -> tuple:
    """(kernel name, source file) of the expert kernel that runs the workload
    (the tcgen05 kernel for bf16 and mixed bf16/INT4 experts)."""
    return ("ffn_tc_kernel", "ffn_tc.cu")


def kernel_source_hash(source: str = "ffn_tc.cu") -> str:
    h = hashlib.sha256()
    for f in (source, "common.cuh"):
        with open(os.path.join(ROOT, "aware_expert_routing_gb300", "csrc", f), "rb") as fh:
            h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str, run: str, algo_bytes_per_launch: float, source: str = "ffn_tc.cu"):
    """DRAM bytes per launch of the expert kernel from a committed ncu
    capture of the same workload and run, scaled from the captured launch's
    algorithmic bytes to this run's mean (traffic grows in proportion to the
    experts streamed); None if the capture predates the kernel source."""
    p = os.path.join(ROOT, "profiles", "expert_kernel_traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(f"{workload}/{run}")
    if not e or e.get("kernel_source_hash") != kernel_source_hash(source):
        return None
    return round(e["dram_bytes"] * algo_bytes_per_launch / e["algorithmic_bytes"])


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    NAMES = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")

    def __init__(self, gpu_id: str):
        self.lines = []
        self.proc = None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", gpu_id, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def window(self, t0, t1):
        """Only samples taken between t0 and t1 (local wall clock) count."""
        self.t0, self.t1 = t0, t1

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                if not (self.t0 <= ts <= self.t1):
                    continue
            except (ValueError, AttributeError):
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
                power.append(float(f[3]))
            except ValueError:
                continue
            for name, v in zip(self.NAMES, f[5:9]):
                if v.lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(power) if power else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def gpu_smi_id(torch, dev) -> str:
    try:
        u = str(torch.cuda.get_device_properties(dev).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except Exception:
        return str(dev.index or 0)


# ---------------------------------------------------------------------------
# the CPU oracle as a baseline (bounded sample, scaled to one layer)
# ---------------------------------------------------------------------------
class OracleInputs:
    """Layer-0 inputs of a workload on the host, and 8 of its activated
    experts, made once before any timing."""

    def __init__(self, w: synth.Workload, B: int, run: tuple):
        import oracle
        oracle.build()
        self.x = synth.make_tensor(w, 0, synth.T_X, B)
        self.wr = synth.make_tensor(w, 0, synth.T_ROUTER)
        self.bias = synth.make_bias(w, 0)
        self.mode = oracle.OEA if run[1] == "oea" else oracle.TOPK
        lg = oracle.router_logits(self.x, self.wr, self.bias)
        r = oracle.route(lg.astype(np.float32), self.mode, w.k, run[2], run[3])
        self.experts = [synth.make_expert(w, 0, int(e)) for e in r["active"][:8]]


def oracle_layer_time(w: synth.Workload, B: int, run: tuple, budget_s: float, inp=None) -> dict:
    """Times the oracle on host cores: router + routing of the full batch,
    then expert FFNs on (token, expert) pairs cycling over 8 experts until
    the budget is spent (at least one pair); the layer time is route time +
    (token, expert) pairs of the layer * time per pair (the oracle's cost
    per pair does not depend on which expert)."""
    import oracle
    inp = inp or OracleInputs(w, B, run)
    label, mode, k0, p = run
    x = inp.x
    t0 = time.perf_counter()
    lg = oracle.router_logits(x, inp.wr, inp.bias)
    r = oracle.route(lg.astype(np.float32), inp.mode, w.k, k0, p)
    t_route = time.perf_counter() - t0
    experts = inp.experts
    pairs = 0
    t0 = time.perf_counter()
    while True:
        e = experts[pairs % len(experts)]
        oracle.expert_ffn(x[pairs % B], *e)
        pairs += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    per_pair = el / pairs
    n_pairs = int((r["idx"] >= 0).sum())
    t_layer = t_route + n_pairs * per_pair
    return {"seconds_per_layer": t_layer, "T": r["T"], "pairs_timed": pairs, "route_s": t_route,
            "per_pair_s": per_pair, "pairs_per_layer": n_pairs}


def cpu_baseline(w, B, run, budget_s, unit_bytes_fn):
    o = oracle_layer_time(w, B, run, budget_s)
    value = unit_bytes_fn(o["T"]) / o["seconds_per_layer"] / 1e9
    return {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{w.name} run {run[0]}: oracle router+routing on the full B={B} batch, then "
                       f"{o['pairs_timed']} single-token expert FFNs (8 experts cycled) timed for "
                       f"{budget_s:.0f} s and scaled to the layer's {o['pairs_per_layer']} (token, expert) "
                       f"pairs; {o['seconds_per_layer'] * 1e3:.1f} ms per layer, single thread"),
            "ms_per_layer": o["seconds_per_layer"] * 1e3}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def build_mixed(moe, torch, w: synth.Workload, layer: int, D: dict, dev):
    """Hot set from a 200-step EMA trace of plain top-k on fresh seeded
    batches of 32 tokens; hot experts stay bf16 (device pool), cold experts
    are generated on the device, packed to INT4 on the host and uploaded."""
    bf = torch.bfloat16
    prm_t = moe.RouteParams(B=32, d=w.d, N=w.N, k=w.k)
    rt = moe.Routing(prm_t, dev)
    wst = moe.alloc_workspace(prm_t, 0, dev)
    xt = torch.empty(32, w.d, dtype=bf, device=dev)
    counts = []
    for step in range(200):
        moe.moe_synth_normal(xt, synth.trace_seed(w, layer, step), float(synth.scale_f32(1.0)))
        moe.moe_route(xt, D["w_router"], D["bias"], prm_t, rt, wst)
        counts.append(rt.counts.cpu().numpy())
    hot = [int(e) for e in moe.ema_hot_set(np.array(counts), w.hot_n)]
    cold = [e for e in range(w.N) if e not in hot]
    slot = np.empty(w.N, np.int32)
    for i, e in enumerate(hot):
        slot[e] = i
    for i, e in enumerate(cold):
        slot[e] = -1 - i
    hot_idx = torch.tensor(hot, device=dev)
    pools = {k: D[k].index_select(0, hot_idx).contiguous() for k in ("w_gate", "w_up", "w_down")}
    q = {k: [] for k in ("w_gate", "w_up", "w_down")}
    for e in cold:
        g, u, dn = (D[k][e].float().cpu().numpy() for k in ("w_gate", "w_up", "w_down"))
        (pg, pu, pd), _ = synth.pack_int4_expert(g, u, dn)
        q["w_gate"].append(pg)
        q["w_up"].append(pu)
        q["w_down"].append(pd)
    qt = {k: torch.from_numpy(np.stack(v)).to(dev) for k, v in q.items()}
    mixed = moe.MixedExperts(torch.from_numpy(slot).to(dev), qt["w_gate"], qt["w_up"], qt["w_down"],
                             len(hot), len(cold))
    for k in ("w_gate", "w_up", "w_down"):   # the full bf16 tensors are not needed any more
        D[k] = None
    D["hot"] = pools
    D["mixed"] = mixed
    D["is_hot"] = np.isin(np.arange(w.N), hot)


def build_layers(moe, torch, w: synth.Workload, B: int, dev):
    bf = torch.bfloat16
    layers = []
    for l in range(N_LAYERS):  # noqa: E741
        D = {}
        for name, tid in (("w_router", synth.T_ROUTER), ("w_gate", synth.T_GATE), ("w_up", synth.T_UP),
                          ("w_down", synth.T_DOWN)):
            t = torch.empty(synth.tensor_shape(w, tid, B), dtype=bf, device=dev)
            moe.moe_synth_normal(t, synth.tensor_seed(w.seed, l, tid),
                                 float(synth.scale_f32(synth.tensor_std(w, tid))))
            D[name] = t
        x = torch.empty((B, w.d), dtype=bf, device=dev)
        moe.moe_synth_normal(x, synth.tensor_seed(w.seed, l, synth.T_X), float(synth.scale_f32(1.0)))
        D["x"] = x
        b = synth.make_bias(w, l)
        D["bias"] = torch.from_numpy(b).to(dev) if b is not None else None
        if w.int4_cold:
            build_mixed(moe, torch, w, l, D, dev)
            torch.cuda.empty_cache()
        layers.append(D)
    torch.cuda.synchronize(dev)
    return layers


def expert_call(moe, w, D, prm, routing, out, ws, stream, x=None):
    x = D["x"] if x is None else x
    if "mixed" in D:
        h = D["hot"]
        moe.moe_expert_ffn_mixed(x, h["w_gate"], h["w_up"], h["w_down"], D["mixed"], w.F, prm, routing, out, ws,
                                 stream)
    else:
        moe.moe_expert_ffn(x, D["w_gate"], D["w_up"], D["w_down"], w.F, prm, routing, out, ws, stream)


def run_mode(moe, torch, w, B, layers, run, steps, warmup, dev, stream, clocks_for=None, detail_steps=2000):
    label, mode, k0, p = run
    prm = moe.RouteParams(B=B, d=w.d, N=w.N, k=w.k, mode=moe.MODE_OEA if mode == "oea" else moe.MODE_TOPK,
                          k0=k0, p=p)
    routing = moe.Routing(prm, dev)
    ws = moe.alloc_workspace(prm, w.F, dev)
    out = torch.empty((B, w.d), dtype=torch.bfloat16, device=dev)

    # T of each layer (routing is deterministic for fixed inputs), and for
    # mixed layers the active experts' formats
    Ts, kbytes, lbytes = [], [], []
    with torch.cuda.stream(stream):
        for D in layers:
            moe.moe_route(D["x"], D["w_router"], D["bias"], prm, routing, ws, stream)
            T = int(routing.T.item())
            Ts.append(T)
            if "mixed" in D:
                act = routing.active[:T].cpu().numpy()
                nh = int(D["is_hot"][act].sum())
                kbytes.append(mixed_kernel_bytes(w, B, nh, T - nh))
                lbytes.append(mixed_layer_bytes(w, B, nh, T - nh))
            else:
                kbytes.append(expert_kernel_bytes(w, B, T))
                lbytes.append(layer_bytes(w, B, T))
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")

    def step(i, ev_pre=None, ev_post=None):
        D = layers[i % N_LAYERS]
        if ev_pre is None and "mixed" not in D:
            # the whole layer through the public call (routing, then experts)
            moe.moe_decode_layer(D["x"], D["w_router"], D["bias"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm,
                                 routing, out, ws, stream)
            return
        moe.moe_route(D["x"], D["w_router"], D["bias"], prm, routing, ws, stream)
        if ev_pre is not None:
            ev_pre.record(stream)
        expert_call(moe, w, D, prm, routing, out, ws, stream)
        if ev_post is not None:
            ev_post.record(stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # Timed region 1 (the headline): K steps back to back, one event pair
    # around all of them, so consecutive kernels overlap their launch and
    # prologue as they do in use.
    clocks = Clocks(clocks_for) if clocks_for else None
    if clocks:
        time.sleep(0.5)          # nvidia-smi start-up
    barrier(torch)
    torch.cuda.synchronize(dev)
    t_start = datetime.datetime.now()
    ev_a, ev_b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ev_a.record(stream)
    for i in range(steps):
        step(i)
    ev_b.record(stream)
    torch.cuda.synchronize(dev)
    t_end = datetime.datetime.now()
    barrier(torch)
    clk = None
    if clocks:
        time.sleep(0.2)
        clocks.window(t_start, t_end)
        clk = clocks.stop()
    total_ms = ev_a.elapsed_time(ev_b)

    # Timed region 2: the same steps with an event at every step boundary
    # and around every expert-kernel launch (per-step percentiles and the
    # expert kernel's launch duration for the roofline).  An event between
    # two kernels keeps the second from starting early, so these steps run
    # slower than region 1's.
    n2 = min(steps, detail_steps)
    ev_step = [torch.cuda.Event(enable_timing=True) for _ in range(n2 + 1)]
    ev_pre = [torch.cuda.Event(enable_timing=True) for _ in range(n2)]
    ev_post = [torch.cuda.Event(enable_timing=True) for _ in range(n2)]
    barrier(torch)
    torch.cuda.synchronize(dev)
    ev_step[0].record(stream)
    for i in range(n2):
        step(i, ev_pre[i], ev_post[i])
        ev_step[i + 1].record(stream)
    torch.cuda.synchronize(dev)
    barrier(torch)
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")
    step_us = [ev_step[i].elapsed_time(ev_step[i + 1]) * 1e3 for i in range(n2)]
    ffn_us = [ev_pre[i].elapsed_time(ev_post[i]) * 1e3 for i in range(n2)]
    layer_b = sum(lbytes[i % N_LAYERS] for i in range(steps))
    ffn_b = sum(kbytes[i % N_LAYERS] for i in range(n2))
    return {
        "label": label, "T_mean": float(np.mean(Ts)), "T_per_layer": Ts, "layer_bytes": lbytes,
        "total_ms": total_ms, "bytes": layer_b,
        "us_per_layer": total_ms * 1e3 / steps,
        "us_per_layer_p10_p50_p90": [float(np.percentile(step_us, q)) for q in (10, 50, 90)],
        "us_per_layer_with_kernel_events": float(np.mean(step_us)),
        "gbs": layer_b / (total_ms * 1e-3) / 1e9,
        "tokens_per_s": B * steps / (total_ms * 1e-3),
        "ffn_us_mean": float(np.mean(ffn_us)),
        "ffn_gbs": ffn_b / (sum(ffn_us) * 1e-6) / 1e9,
        "ffn_bytes_per_launch": ffn_b / n2,
        "clocks": clk, "launches": moe.moe_layer_launches(prm, w.F) * steps,
        "objs": (prm, routing, ws, out),
    }


def run_e2e(moe, torch, w, B, layers, run, steps, warmup, dev, stream, lbytes):
    """moe_decode_layer with the hidden states copied in from pinned host
    memory and the output copied back, every step, inside the timed region."""
    label, mode, k0, p = run
    prm = moe.RouteParams(B=B, d=w.d, N=w.N, k=w.k, mode=moe.MODE_OEA if mode == "oea" else moe.MODE_TOPK,
                          k0=k0, p=p)
    routing = moe.Routing(prm, dev)
    ws = moe.alloc_workspace(prm, w.F, dev)
    x_host = [D["x"].cpu().pin_memory() for D in layers]
    out_host = torch.empty((B, w.d), dtype=torch.bfloat16).pin_memory()
    x_dev = torch.empty((B, w.d), dtype=torch.bfloat16, device=dev)
    out = torch.empty((B, w.d), dtype=torch.bfloat16, device=dev)

    def step(i):
        D = layers[i % N_LAYERS]
        with torch.cuda.stream(stream):
            x_dev.copy_(x_host[i % N_LAYERS], non_blocking=True)
            if "mixed" in D:
                moe.moe_route(x_dev, D["w_router"], D["bias"], prm, routing, ws, stream)
                expert_call(moe, w, D, prm, routing, out, ws, stream, x=x_dev)
            else:
                moe.moe_decode_layer(x_dev, D["w_router"], D["bias"], D["w_gate"], D["w_up"], D["w_down"],
                                     w.F, prm, routing, out, ws, stream)
            out_host.copy_(out, non_blocking=True)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    barrier(torch)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for i in range(steps):
        step(i)
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(torch)
    ms = e0.elapsed_time(e1)
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")
    b = sum(lbytes[i % N_LAYERS] for i in range(steps))
    return {"value": b / (ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": B * w.d * 2,
            "d2h_bytes_per_step": B * w.d * 2, "us_per_layer": ms * 1e3 / steps, "_bytes": b, "_ms": ms}


# ---------------------------------------------------------------------------
# distributed plumbing: one replica per GPU, no data-path collective
# ---------------------------------------------------------------------------
_dist = {"on": False}


def init_dist(torch):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
        _dist["on"] = True
    return int(os.environ.get("RANK", "0")), world, int(os.environ.get("LOCAL_RANK", "0"))


def barrier(torch):
    if _dist["on"]:
        import torch.distributed as dist
        dist.barrier()


def reduce_max(torch, dev, x: float) -> float:
    if not _dist["on"]:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(torch, dev, x: float) -> float:
    if not _dist["on"]:
        return x
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def main_ours(args):
    import torch
    import aware_expert_routing_gb300 as moe
    from aware_expert_routing_gb300 import build as moe_build

    rank, world, local = init_dist(torch)
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if rank == 0:
        moe_build.build()
    barrier(torch)
    moe.load()
    w = synth.WORKLOADS[args.workload]
    B = args.batch or w.B
    runs = {r[0]: r for r in w.runs}
    head = runs[HEADLINE.get(w.name, w.runs[-1][0])]
    stream = torch.cuda.Stream(dev)
    layers = build_layers(moe, torch, w, B, dev)
    smi = gpu_smi_id(torch, dev)

    results = {}
    if args.only_run:
        runs = {args.only_run: runs[args.only_run]}
        head = runs[args.only_run]
    for label, run in runs.items():
        res = run_mode(moe, torch, w, B, layers, run, args.steps, args.warmup, dev, stream,
                       clocks_for=smi if label == head[0] else None)
        res.pop("objs")
        results[label] = res
    hr = results[head[0]]
    e2e = run_e2e(moe, torch, w, B, layers, head, args.steps, args.warmup, dev, stream, hr["layer_bytes"])

    # whole job: bytes of all ranks / slowest rank
    t_max = reduce_max(torch, dev, hr["total_ms"])
    b_all = reduce_sum(torch, dev, hr["bytes"])
    value = b_all / (t_max * 1e-3) / 1e9
    e2e_ms = reduce_max(torch, dev, e2e.pop("_ms"))
    e2e["value"] = round(reduce_sum(torch, dev, e2e.pop("_bytes")) / (e2e_ms * 1e-3) / 1e9, 1)
    e2e["us_per_layer"] = round(e2e["us_per_layer"], 2)

    if rank != 0:
        return
    peaks = measured_peaks()
    ach = hr["ffn_gbs"]
    roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4),
            "traffic": recorded_traffic(w.name, head[0], hr["ffn_bytes_per_launch"], expert_kernel(w)[1]),
            "kernel": expert_kernel(w)[0], "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": round(hr["ffn_bytes_per_launch"]),
            "mean_launch_us": round(hr["ffn_us_mean"], 2)}
    base = None
    if not args.no_cpu_baseline:
        mean_b = float(np.mean(hr["layer_bytes"]))
        base = cpu_baseline(w, B, head, args.cpu_budget,
                            (lambda T: mean_b) if w.int4_cold else (lambda T: layer_bytes(w, B, T)))
    modes = {}
    for label, r in results.items():
        modes[label] = {"T": round(r["T_mean"], 2), "us_per_layer": round(r["us_per_layer"], 2),
                        "us_p10_p50_p90": [round(v, 2) for v in r["us_per_layer_p10_p50_p90"]],
                        "gbs": round(r["gbs"], 1), "tokens_per_s": round(r["tokens_per_s"]),
                        "frac_of_measured_hbm": round(r["gbs"] / peaks["hbm_gbs"], 4),
                        "us_per_layer_with_kernel_events": round(r["us_per_layer_with_kernel_events"], 2),
                        "ffn_us": round(r["ffn_us_mean"], 2), "ffn_gbs": round(r["ffn_gbs"], 1)}
    if "topk" in results:
        for label, r in results.items():
            if label != "topk":
                modes[label]["latency_vs_topk"] = round(r["us_per_layer"] / results["topk"]["us_per_layer"], 4)
                modes[label]["T_vs_topk"] = round(r["T_mean"] / results["topk"]["T_mean"], 4)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / args.steps, 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded SplitMix64/Irwin-Hall weights and hidden states, random init",
        "config": {"workload": w.name, "B": B, "N": w.N, "k": w.k, "d": w.d, "d_ff": w.F,
                   "routing": head[0], "layers_rotated": N_LAYERS, "runs": sorted(runs),
                   "l2": "inputs larger than L2: %d-layer rotation, %.2f GB of expert weights per layer"
                         % (N_LAYERS, w.N * w.expert_bytes / 1e9),
                   "parallelism": f"replicas x{world}"},
        "modes": modes, "roofline": roof, "cpu_baseline": base, "e2e": e2e,
        "clocks": hr["clocks"], "gpu_launches": hr["launches"],
    }
    print(json.dumps(line), flush=True)
    if args.sweep_out:
        sweep(moe, torch, w, dev, stream, args)
    if args.linearity_out:
        linearity(moe, torch, w, dev, stream, args)


def sweep(moe, torch, w, dev, stream, args):
    """Per-B rows for the workload's batch sweep (written to a file)."""
    rows = []
    for B in (w.batch_sweep or (w.B,)):
        layers = build_layers(moe, torch, w, B, dev)
        for run in w.runs:
            r = run_mode(moe, torch, w, B, layers, run, max(50, args.steps // 4), args.warmup, dev, stream)
            r.pop("objs")
            rows.append({"workload": w.name, "B": B, "run": run[0], "T": r["T_mean"],
                         "us_per_layer": r["us_per_layer"], "p10_p50_p90": r["us_per_layer_p10_p50_p90"],
                         "tokens_per_s": r["tokens_per_s"], "gbs": r["gbs"], "ffn_us": r["ffn_us_mean"],
                         "ffn_gbs": r["ffn_gbs"]})
            log(json.dumps(rows[-1]))
        del layers
        torch.cuda.empty_cache()
    with open(args.sweep_out, "w") as f:
        json.dump(rows, f, indent=1)


def linear_fit(X: np.ndarray, y: np.ndarray) -> dict:
    """Least squares y = X beta; coefficients and R^2."""
    beta, *_ = np.linalg.lstsq(X, y, rcond=None)
    pred = X @ beta
    ss_res = float(np.sum((y - pred) ** 2))
    ss_tot = float(np.sum((y - y.mean()) ** 2))
    return {"coef": [float(b) for b in beta], "r2": 1.0 - ss_res / ss_tot if ss_tot > 0 else 1.0}


def linearity(moe, torch, w, dev, stream, args):
    """Latency against T (distinct activated experts) and sum(cnt_e) (token-
    expert pairs), the OEA page's cost model (section 4: latency grows with
    the number of activated experts).  T is forced by a router bias of +20 on
    T experts drawn with a seeded generator (every token's top-k then lies
    among them) with top-min(k, T) routing, so sum(cnt_e) = B min(k, T);
    B in {1, 4, 16, 64} varies sum(cnt_e) independently of T.  Fits
    us = a sum(cnt_e) + b T + c for the whole layer and the expert kernel;
    b is the cost of one more activated expert, 3 d d_ff 2 / b its
    streaming rate.  32 distinct layers rotate (1.2 GB of experts each at
    the 30B shapes), so even T = 1 streams 300 MB per rotation, above the
    126 MB L2."""
    import dataclasses
    global N_LAYERS
    saved, N_LAYERS = N_LAYERS, 32
    rows = []
    steps = max(100, args.steps // 20)
    for B in (1, 4, 16, 64):
        base = build_layers(moe, torch, w, B, dev)
        for Tt in (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128):
            if Tt > w.N:
                continue
            k = min(w.k, Tt)
            wk = dataclasses.replace(w, k=k)
            bias = np.zeros(w.N, np.float32)
            bias[np.random.default_rng(1000 + Tt).choice(w.N, Tt, replace=False)] = 20.0
            bias_d = torch.from_numpy(bias).to(dev)
            layers = [dict(D, bias=bias_d) for D in base]
            r = run_mode(moe, torch, wk, B, layers, ("topk", "topk", k, 1.0), steps, args.warmup, dev, stream,
                         detail_steps=steps)
            r.pop("objs")
            rows.append({"B": B, "k": k, "T_forced": Tt, "T": r["T_mean"], "sum_cnt": B * k,
                         "us_per_layer": r["us_per_layer"], "ffn_us": r["ffn_us_mean"]})
            log(json.dumps(rows[-1]))
        del base
        torch.cuda.empty_cache()
    N_LAYERS = saved
    X = np.array([[r["sum_cnt"], r["T"], 1.0] for r in rows])
    out = {"workload": w.name, "model": "us = a * sum_cnt + b * T + c", "layers_rotated": 32, "rows": rows}
    for key, col in (("fit_layer", "us_per_layer"), ("fit_expert_kernel", "ffn_us")):
        f = linear_fit(X, np.array([r[col] for r in rows]))
        a, b, c = f["coef"]
        out[key] = {"a_us_per_pair": a, "b_us_per_expert": b, "c_us": c, "r2": f["r2"],
                    "expert_bytes": w.expert_bytes,
                    "streaming_gbs_per_added_expert": w.expert_bytes / (b * 1e-6) / 1e9 if b > 0 else None}
    with open(args.linearity_out, "w") as f:
        json.dump(out, f, indent=1)
    log(json.dumps({k: v for k, v in out.items() if k.startswith("fit")}))


# ---------------------------------------------------------------------------
# reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------
def main_reference(args):
    if int(os.environ.get("RANK", "0")) != 0:
        return
    w = synth.WORKLOADS[args.workload]
    B = args.batch or w.B
    runs = {r[0]: r for r in w.runs}
    head = runs[HEADLINE.get(w.name, w.runs[-1][0])]
    budget = args.cpu_budget / max(1, args.steps + args.warmup)
    inp = OracleInputs(w, B, head)
    vals = []
    for i in range(args.warmup + args.steps):
        o = oracle_layer_time(w, B, head, budget, inp)
        if i >= args.warmup:
            vals.append(o)
    sec = float(np.mean([o["seconds_per_layer"] for o in vals]))
    value = layer_bytes(w, B, vals[0]["T"]) / sec / 1e9
    sample = (f"per step: oracle router+routing on the full B={B} batch and single-token expert FFNs "
              f"(8 experts cycled, at least one, for {budget:.3f} s), scaled to one layer's "
              f"(token, expert) pairs; single thread")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": {"workload": w.name, "B": B, "N": w.N, "k": w.k, "d": w.d, "d_ff": w.F,
                       "routing": head[0]},
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--sweep-out", default="")
    ap.add_argument("--linearity-out", default="", help="latency-vs-T sweep and fit, written to this file")
    ap.add_argument("--layers", type=int, default=8, help="distinct layers rotated through")
    ap.add_argument("--only-run", default="", help="time only this routing run (profiling)")
    args = ap.parse_args()
    global N_LAYERS
    N_LAYERS = args.layers
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
