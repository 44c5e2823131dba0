#!/usr/bin/env python
"""Benchmark of the OEA MoE decode layer on GB300.

A step is one pass of the whole layer (router, routing, grouped SwiGLU
experts, combine) over one decode batch, through one public call
(moe_decode_layer, or moe_decode_layer_mixed for bf16/INT4 experts).  Steps
cycle through 8 layers with distinct seeded weights (about 1.2 GB of expert
weights per layer at the Qwen3-30B-A3B shapes, far larger than the 126 MB
L2), so every step streams its activated experts from HBM.

Timed regions: exactly K steps back to back between a barrier +
synchronize on both sides and one CUDA event pair on the launching stream,
repeated until at least --min-seconds have been timed (so the clock sampler
sees the run); ms_per_step = total time / (reps * K).

value     = algorithmic bytes / device time of the headline routing run
            (whole job: summed over ranks, divided by the slowest rank's
            time).  Algorithmic bytes per layer = T * expert bytes (the
            activated experts, read once) + the router weights N*d*2 +
            activations (x read twice, scores, output).
modes     = every routing run of the headline workload.
sweep     = the rest of the metric ("vs B, OEA vs top-k"): the Zipf-routed
            30B workload at B = 1, 16, 64, the 235B workload at B = 64 and
            the mixed bf16/INT4 30B workload at B = 32, OEA and top-8 each.
router    = scoring + routing alone (moe_route back to back), its own
            microseconds and GB/s.
roofline  = the expert kernel alone: its algorithmic bytes per launch over
            its mean launch time (CUDA events on the launching stream
            around every expert launch, in a separate pass of the same
            steps), against the measured HBM copy bandwidth; `traffic` is
            ncu's DRAM bytes per launch from profiles/, when the capture
            matches the kernel source.
e2e       = the same metric through the public call with host buffers:
            every step's hidden states are copied in from pinned host
            memory and its output copied back, on a copy stream with double
            buffers (a step's input one step ahead, its output after an
            event), all inside the timed region.

python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                [--workload NAME] [--no-sweep] [--sweep-out FILE]
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import platform
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
SPEC_HBM_GBS = 8000.0   # the ~8 TB/s HBM3e figure the target is stated against
DEFAULT_WORKLOAD = "qwen3_30b_a3b_uniform_b16"
HEADLINE = {"qwen3_30b_a3b_uniform_b16": "oea_k0_3", "qwen3_30b_a3b_zipf_sweep": "oea_k0_5_p0.7",
            "qwen3_235b_a22b_zipf_b64": "oea_k0_5_p0.7", "qwen3_30b_a3b_mixed_int4_b32": "oea_k0_5"}
# the rest of the metric in the default line: (workload, batch sizes)
SWEEP = [("qwen3_30b_a3b_zipf_sweep", (1, 16, 64)), ("qwen3_235b_a22b_zipf_b64", (64,)),
         ("qwen3_30b_a3b_mixed_int4_b32", (32,))]
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


def router_bytes(w: synth.Workload, B: int) -> float:
    """Router weights once, hidden states in, scores out."""
    return w.N * w.d * 2 + B * w.d * 2 + B * w.N * 4


def layer_bytes(w: synth.Workload, B: int, T: float) -> float:
    return router_bytes(w, B) + expert_kernel_bytes(w, B, T)


def mixed_kernel_bytes(w: synth.Workload, B: int, n_hot_active: int, n_cold_active: int) -> float:
    """Expert-kernel bytes with bf16 hot and INT4 cold experts."""
    return (n_hot_active * w.expert_bytes + n_cold_active * synth.int4_expert_bytes(w.d, w.F)
            + 2 * B * w.d * 2)


def mixed_layer_bytes(w: synth.Workload, B: int, n_hot_active: int, n_cold_active: int) -> float:
    return router_bytes(w, B) + mixed_kernel_bytes(w, B, n_hot_active, n_cold_active)


def measured_peaks() -> dict:
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return {"hbm_gbs": float(d["hbm_gbs"]), "source": "measured"}
    return {"hbm_gbs": 6800.0, "source": "fallback"}


def strip_comments(src: str) -> str:
    """C/C++ source without its comments (string and character literals
    kept as they are), whitespace runs collapsed to one space."""
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
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_hash(source: str = "ffn_tc.cu") -> str:
    """Hash of the expert kernel's code (its source and common.cuh, comments
    and layout left out): an ncu record taken from other code is not used."""
    h = hashlib.sha256()
    for f in (source, "common.cuh"):
        with open(os.path.join(ROOT, "aware_expert_routing_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
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


def cpu_description() -> dict:
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.lower().startswith("model name"):
                model = line.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.TimeoutExpired):
        pass
    if not model:
        try:
            with open("/proc/cpuinfo") as f:
                for line in f:
                    if line.lower().startswith(("model name", "cpu part")):
                        model = line.split(":", 1)[1].strip()
                        break
        except OSError:
            pass
    return {"nproc": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine(),
            "arch": platform.machine()}


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
        self.windows = []
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
        """Samples taken between t0 and t1 (local wall clock) count."""
        self.windows.append((t0, t1))

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
                if not any(a <= ts <= b for a, b in self.windows):
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
    cpu = cpu_description()
    return {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": (f"{w.name} run {run[0]}: oracle router+routing on the full B={B} batch, then "
                       f"{o['pairs_timed']} single-token expert FFNs (8 experts cycled) timed for "
                       f"{budget_s:.0f} s and scaled to the layer's {o['pairs_per_layer']} (token, expert) "
                       f"pairs; {o['seconds_per_layer'] * 1e3:.1f} ms per layer, single thread on 1 of "
                       f"{cpu['nproc']} cores ({cpu['cpu_model']})"),
            "ms_per_layer": o["seconds_per_layer"] * 1e3, **cpu}


# ---------------------------------------------------------------------------
# our implementation
# ---------------------------------------------------------------------------
def build_mixed(moe, torch, w: synth.Workload, layer: int, D: dict, dev):
    """Hot set from a 200-step EMA trace of plain top-k on fresh seeded
    batches of 32 tokens; hot experts stay bf16 (device pool), cold experts
    are packed to INT4 on the device (moe_pack_int4)."""
    prm_t = moe.RouteParams(B=32, d=w.d, N=w.N, k=w.k)
    rt = moe.Routing(prm_t, dev)
    wst = moe.alloc_workspace(prm_t, 0, dev)
    xt = torch.empty(32, w.d, dtype=torch.bfloat16, device=dev)
    counts = []
    for step in range(200):
        moe.moe_synth_normal(xt, synth.trace_seed(w, layer, step), float(synth.scale_f32(1.0)))
        moe.moe_route(xt, D["w_router"], D["bias"], prm_t, rt, wst)
        counts.append(rt.counts.clone())
    hot = [int(e) for e in moe.ema_hot_set(torch.stack(counts).cpu().numpy(), w.hot_n)]
    cold = [e for e in range(w.N) if e not in hot]
    slot = np.empty(w.N, np.int32)
    for i, e in enumerate(hot):
        slot[e] = i
    for i, e in enumerate(cold):
        slot[e] = -1 - i
    hot_idx = torch.tensor(hot, device=dev)
    # W_gate's and W_up's pools as the two halves of one buffer (one tensor
    # map then reads both; see w_up in include/moe.h)
    gu = torch.empty((2, len(hot)) + tuple(D["w_gate"].shape[1:]), dtype=D["w_gate"].dtype, device=dev)
    torch.index_select(D["w_gate"], 0, hot_idx, out=gu[0])
    torch.index_select(D["w_up"], 0, hot_idx, out=gu[1])
    pools = {"w_gate": gu[0], "w_up": gu[1], "w_down": D["w_down"].index_select(0, hot_idx).contiguous()}
    u8 = dict(dtype=torch.uint8, device=dev)
    q = {"w_gate": torch.empty(len(cold), moe.int4_image_bytes(w.F, w.d), **u8),
         "w_up": torch.empty(len(cold), moe.int4_image_bytes(w.F, w.d), **u8),
         "w_down": torch.empty(len(cold), moe.int4_image_bytes(w.d, w.F), **u8)}
    for i, e in enumerate(cold):
        moe.moe_pack_int4(D["w_gate"][e], 64, out=q["w_gate"][i])
        moe.moe_pack_int4(D["w_up"][e], 64, out=q["w_up"][i])
        moe.moe_pack_int4(D["w_down"][e], 128, out=q["w_down"][i])
    mixed = moe.MixedExperts(torch.from_numpy(slot).to(dev), q["w_gate"], q["w_up"], q["w_down"],
                             len(hot), len(cold))
    for k in ("w_gate", "w_up", "w_down"):   # the full bf16 tensors are not needed any more
        D[k] = None
    D["hot"] = pools
    D["mixed"] = mixed
    D["is_hot"] = np.isin(np.arange(w.N), hot)


def build_weights(moe, torch, w: synth.Workload, dev, nl: int):
    """nl layers of router and expert weights, generated on the device."""
    bf = torch.bfloat16
    layers = []
    for l in range(nl):  # noqa: E741
        D = {}
        for name, tid in (("w_router", synth.T_ROUTER), ("w_gate", synth.T_GATE), ("w_up", synth.T_UP),
                          ("w_down", synth.T_DOWN)):
            t = torch.empty(synth.tensor_shape(w, tid), dtype=bf, device=dev)
            moe.moe_synth_normal(t, synth.tensor_seed(w.seed, l, tid),
                                 float(synth.scale_f32(synth.tensor_std(w, tid))))
            D[name] = t
        b = synth.make_bias(w, l)
        D["bias"] = torch.from_numpy(b).to(dev) if b is not None else None
        if w.int4_cold:
            build_mixed(moe, torch, w, l, D, dev)
            torch.cuda.empty_cache()
        layers.append(D)
    torch.cuda.synchronize(dev)
    return layers


def with_batch(moe, torch, w: synth.Workload, weights: list, B: int, dev):
    """The layers with hidden states of B tokens (seeded per layer)."""
    out = []
    for l, D in enumerate(weights):  # noqa: E741
        x = torch.empty((B, w.d), dtype=torch.bfloat16, device=dev)
        moe.moe_synth_normal(x, synth.tensor_seed(w.seed, l, synth.T_X), float(synth.scale_f32(1.0)))
        out.append(dict(D, x=x))
    torch.cuda.synchronize(dev)
    return out


def build_layers(moe, torch, w: synth.Workload, B: int, dev):
    return with_batch(moe, torch, w, build_weights(moe, torch, w, dev, N_LAYERS), B, dev)


def layer_call(moe, w, D, prm, routing, out, ws, stream, x=None):
    """One whole layer through the public one-call API."""
    x = D["x"] if x is None else x
    if "mixed" in D:
        h = D["hot"]
        moe.moe_decode_layer_mixed(x, D["w_router"], D["bias"], h["w_gate"], h["w_up"], h["w_down"], D["mixed"],
                                   w.F, prm, routing, out, ws, stream)
    else:
        moe.moe_decode_layer(x, D["w_router"], D["bias"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm,
                             routing, out, ws, stream)


def expert_call(moe, w, D, prm, routing, out, ws, stream):
    if "mixed" in D:
        h = D["hot"]
        moe.moe_expert_ffn_mixed(D["x"], h["w_gate"], h["w_up"], h["w_down"], D["mixed"], w.F, prm, routing, out,
                                 ws, stream)
    else:
        moe.moe_expert_ffn(D["x"], D["w_gate"], D["w_up"], D["w_down"], w.F, prm, routing, out, ws, stream)


def params_of(moe, w, B, run):
    label, mode, k0, p = run
    return moe.RouteParams(B=B, d=w.d, N=w.N, k=w.k, mode=moe.MODE_OEA if mode == "oea" else moe.MODE_TOPK,
                           k0=k0, p=p)


def timed_reps(torch, dev, stream, step, steps: int, min_seconds: float, first: int = 0,
               clocks=None, max_reps: int = 100000):
    """Exactly `steps` steps per timed region (barrier + synchronize on both
    sides, one CUDA event pair on the stream), repeated until min_seconds
    of device time; returns the per-region milliseconds and the steps
    issued."""
    reps_ms = []
    i = first
    total = 0.0
    while True:
        barrier(torch)
        torch.cuda.synchronize(dev)
        t0 = datetime.datetime.now()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps):
            step(i)
            i += 1
        b.record(stream)
        torch.cuda.synchronize(dev)
        t1 = datetime.datetime.now()
        barrier(torch)
        if clocks:
            clocks.window(t0, t1)
        ms = a.elapsed_time(b)
        reps_ms.append(ms)
        total += ms
        if total >= min_seconds * 1e3 or len(reps_ms) >= max_reps:
            return reps_ms, i


def run_mode(moe, torch, w, B, layers, run, steps, warmup, dev, stream, min_seconds, clocks=None,
             detail_steps=200):
    nl = len(layers)
    prm = params_of(moe, w, B, run)
    routing = moe.Routing(prm, dev)
    ws = moe.alloc_workspace(prm, w.F, dev)
    out = torch.empty((B, w.d), dtype=torch.bfloat16, device=dev)

    # T of each layer (routing is deterministic for fixed inputs), and for
    # mixed layers the active experts' formats
    Ts, kbytes, lbytes, nhot = [], [], [], []
    with torch.cuda.stream(stream):
        for D in layers:
            moe.moe_route(D["x"], D["w_router"], D["bias"], prm, routing, ws, stream)
            T = int(routing.T.item())
            Ts.append(T)
            if "mixed" in D:
                act = routing.active[:T].cpu().numpy()
                nh = int(D["is_hot"][act].sum())
                nhot.append(nh)
                kbytes.append(mixed_kernel_bytes(w, B, nh, T - nh))
                lbytes.append(mixed_layer_bytes(w, B, nh, T - nh))
            else:
                kbytes.append(expert_kernel_bytes(w, B, T))
                lbytes.append(layer_bytes(w, B, T))
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")

    def step(i):
        layer_call(moe, w, layers[i % nl], prm, routing, out, ws, stream)

    for i in range(warmup):
        step(i)
    torch.cuda.synchronize(dev)
    reps_ms, issued = timed_reps(torch, dev, stream, step, steps, min_seconds, first=warmup, clocks=clocks)
    n_steps = len(reps_ms) * steps
    total_ms = sum(reps_ms)
    layer_b = sum(lbytes[i % nl] for i in range(warmup, issued))

    # The expert kernel alone: events around every expert launch (moe_route,
    # then the expert call), in a separate pass.  An event between two
    # kernels keeps the second from starting early, so these steps are
    # slower than the timed regions'; only the expert kernel's duration is
    # taken from here.
    n2 = max(steps, detail_steps)
    ev_pre = [torch.cuda.Event(enable_timing=True) for _ in range(n2)]
    ev_post = [torch.cuda.Event(enable_timing=True) for _ in range(n2)]
    barrier(torch)
    torch.cuda.synchronize(dev)
    for i in range(n2):
        D = layers[i % nl]
        moe.moe_route(D["x"], D["w_router"], D["bias"], prm, routing, ws, stream)
        ev_pre[i].record(stream)
        expert_call(moe, w, D, prm, routing, out, ws, stream)
        ev_post[i].record(stream)
    torch.cuda.synchronize(dev)
    barrier(torch)
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")
    ffn_us = [ev_pre[i].elapsed_time(ev_post[i]) * 1e3 for i in range(n2)]
    ffn_b = sum(kbytes[i % nl] for i in range(n2))
    per_step_reps = [ms * 1e3 / steps for ms in reps_ms]
    return {
        "label": run[0], "T_mean": float(np.mean(Ts)), "T_per_layer": Ts, "layer_bytes": lbytes,
        "hot_active_mean": float(np.mean(nhot)) if nhot else None,
        "total_ms": total_ms, "bytes": layer_b, "reps": len(reps_ms), "steps_timed": n_steps,
        "us_per_layer": total_ms * 1e3 / n_steps,
        "us_per_layer_reps_p10_p50_p90": [float(np.percentile(per_step_reps, q)) for q in (10, 50, 90)],
        "gbs": layer_b / (total_ms * 1e-3) / 1e9,
        "tokens_per_s": B * n_steps / (total_ms * 1e-3),
        "ffn_us_mean": float(np.mean(ffn_us)),
        "ffn_gbs": ffn_b / (sum(ffn_us) * 1e-6) / 1e9,
        "ffn_bytes_per_launch": ffn_b / n2,
        "launches_per_region": moe.moe_layer_launches(prm, w.F) * steps,
    }


def run_router(moe, torch, w, B, layers, run, steps, warmup, dev, stream, min_seconds):
    """Scoring + routing alone (moe_route back to back)."""
    nl = len(layers)
    prm = params_of(moe, w, B, run)
    routing = moe.Routing(prm, dev)
    ws = moe.alloc_workspace(prm, 0, dev)

    def step(i):
        D = layers[i % nl]
        moe.moe_route(D["x"], D["w_router"], D["bias"], prm, routing, ws, stream)

    for i in range(warmup):
        step(i)
    reps_ms, _ = timed_reps(torch, dev, stream, step, steps, min_seconds)
    us = sum(reps_ms) * 1e3 / (len(reps_ms) * steps)
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")
    fused = moe.moe_layer_launches(prm, w.F) == 2
    return {"workload": w.name, "B": B, "run": run[0],
            "kernels": ["route_fused_kernel"] if fused else ["router_bf16_kernel", "route_kernel"],
            "us": round(us, 2), "bytes": router_bytes(w, B),
            "gbs": round(router_bytes(w, B) / (us * 1e-6) / 1e9, 1)}


def run_e2e(moe, torch, w, B, layers, run, steps, warmup, dev, stream, lbytes, min_seconds):
    """The public one-call layer with the hidden states copied in from
    pinned host memory and the output copied back, every step, inside the
    timed region.  The copies run on a copy stream with two device buffers
    each: a step's input is copied one step ahead, its output after an
    event, so they overlap the neighbouring layers."""
    nl = len(layers)
    prm = params_of(moe, w, B, run)
    routing = moe.Routing(prm, dev)
    ws = moe.alloc_workspace(prm, w.F, dev)
    cs = torch.cuda.Stream(dev)
    bf = torch.bfloat16
    x_host = [D["x"].cpu().pin_memory() for D in layers]
    out_host = [torch.empty((B, w.d), dtype=bf).pin_memory() for _ in range(2)]
    x_dev = [torch.empty((B, w.d), dtype=bf, device=dev) for _ in range(2)]
    out_dev = [torch.empty((B, w.d), dtype=bf, device=dev) for _ in range(2)]
    ev_h2d = [torch.cuda.Event() for _ in range(2)]
    ev_comp = [torch.cuda.Event() for _ in range(2)]
    ev_d2h = [torch.cuda.Event() for _ in range(2)]

    def h2d(i):   # step i's hidden states into x_dev[i % 2], once step i-2 has read that buffer
        b = i % 2
        cs.wait_event(ev_comp[b])
        with torch.cuda.stream(cs):
            x_dev[b].copy_(x_host[i % nl], non_blocking=True)
        ev_h2d[b].record(cs)

    def region(first: int, n: int):
        h2d(first)
        for i in range(first, first + n):
            b = i % 2
            if i + 1 < first + n:
                h2d(i + 1)
            stream.wait_event(ev_h2d[b])
            stream.wait_event(ev_d2h[b])           # out_dev[b] copied out (step i-2)
            layer_call(moe, w, layers[i % nl], prm, routing, out_dev[b], ws, stream, x=x_dev[b])
            ev_comp[b].record(stream)
            cs.wait_event(ev_comp[b])
            with torch.cuda.stream(cs):
                out_host[b].copy_(out_dev[b], non_blocking=True)
            ev_d2h[b].record(cs)
        stream.wait_event(ev_d2h[(first + n - 1) % 2])   # the last output is on the host

    region(0, warmup)
    torch.cuda.synchronize(dev)
    reps_ms = []
    i = warmup
    while True:
        barrier(torch)
        torch.cuda.synchronize(dev)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        cs.wait_event(a)
        region(i, steps)
        b.record(stream)
        torch.cuda.synchronize(dev)
        barrier(torch)
        reps_ms.append(a.elapsed_time(b))
        i += steps
        if sum(reps_ms) >= min_seconds * 1e3:
            break
    ms = sum(reps_ms)
    n_steps = len(reps_ms) * steps
    flags = moe.moe_device_status(ws, stream)
    if flags:
        raise RuntimeError(f"device flags {flags:#x}")
    byt = sum(lbytes[j % nl] for j in range(warmup, warmup + n_steps))
    return {"value": byt / (ms * 1e-3) / 1e9, "unit": UNIT, "h2d_bytes_per_step": B * w.d * 2,
            "d2h_bytes_per_step": B * w.d * 2, "us_per_layer": ms * 1e3 / n_steps,
            "call": "moe_decode_layer_mixed" if "mixed" in layers[0] else "moe_decode_layer",
            "_bytes": byt, "_ms": ms}


def config_of(w: synth.Workload, B: int, head: tuple, runs: dict, world: int) -> dict:
    """The workload named in the JSON line (the same for both arms)."""
    return {"workload": w.name, "B": B, "N": w.N, "k": w.k, "d": w.d, "d_ff": w.F,
            "routing": head[0], "layers_rotated": N_LAYERS, "runs": sorted(runs),
            "l2": "inputs larger than L2: %d-layer rotation, %.2f GB of expert weights per layer"
                  % (N_LAYERS, w.N * w.expert_bytes / 1e9),
            "parallelism": f"replicas x{world}"}


def mode_row(r: dict, peak: float) -> dict:
    return {"T": round(r["T_mean"], 2), "us_per_layer": round(r["us_per_layer"], 2),
            "us_reps_p10_p50_p90": [round(v, 2) for v in r["us_per_layer_reps_p10_p50_p90"]],
            "gbs": round(r["gbs"], 1), "tokens_per_s": round(r["tokens_per_s"]),
            "frac_of_measured_hbm": round(r["gbs"] / peak, 4),
            "ffn_us": round(r["ffn_us_mean"], 2), "ffn_gbs": round(r["ffn_gbs"], 1),
            "ffn_frac_of_measured_hbm": round(r["ffn_gbs"] / peak, 4),
            "ffn_frac_of_8tbs": round(r["ffn_gbs"] / SPEC_HBM_GBS, 4),
            **({"hot_active": round(r["hot_active_mean"], 2)} if r["hot_active_mean"] is not None else {})}


def add_vs_topk(rows: dict):
    if "topk" in rows:
        for label, r in rows.items():
            if label != "topk":
                r["latency_vs_topk"] = round(r["us_per_layer"] / rows["topk"]["us_per_layer"], 4)
                r["T_vs_topk"] = round(r["T"] / rows["topk"]["T"], 4)


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


def sweep_rows(moe, torch, args, dev, stream, peak):
    """The metric's other workloads and batch sizes, OEA against top-8."""
    rows = []
    for wname, batches in SWEEP:
        w = synth.WORKLOADS[wname]
        weights = build_weights(moe, torch, w, dev, N_LAYERS)
        for B in batches:
            layers = with_batch(moe, torch, w, weights, B, dev)
            res = {}
            for run in w.runs:
                r = run_mode(moe, torch, w, B, layers, run, args.steps, args.warmup, dev, stream,
                             args.sweep_seconds, detail_steps=100)
                res[run[0]] = dict(workload=wname, B=B, run=run[0], **mode_row(r, peak))
            add_vs_topk(res)
            rows += list(res.values())
            for r in res.values():
                log(json.dumps(r))
            del layers
        del weights
        torch.cuda.empty_cache()
    return rows


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
    if args.only_run:
        runs = {args.only_run: runs[args.only_run]}
        head = runs[args.only_run]
    stream = torch.cuda.Stream(dev)
    layers = build_layers(moe, torch, w, B, dev)
    peaks = measured_peaks()

    # the headline run first, with the clock sampler running
    results = {}
    clocks = Clocks(gpu_smi_id(torch, dev))
    time.sleep(0.5)          # nvidia-smi start-up
    results[head[0]] = run_mode(moe, torch, w, B, layers, head, args.steps, args.warmup, dev, stream,
                                args.min_seconds, clocks=clocks)
    time.sleep(0.2)
    clk = clocks.stop()
    for label, run in runs.items():
        if label != head[0]:
            results[label] = run_mode(moe, torch, w, B, layers, run, args.steps, args.warmup, dev, stream,
                                      args.min_seconds / 2)
    hr = results[head[0]]
    e2e = run_e2e(moe, torch, w, B, layers, head, args.steps, args.warmup, dev, stream, hr["layer_bytes"],
                  args.min_seconds / 2)
    router = [run_router(moe, torch, w, B, layers, head, args.steps, args.warmup, dev, stream, 0.2)]
    if B <= 32 and not args.no_sweep:   # the separate router and routing kernels (above 32 tokens)
        l64 = with_batch(moe, torch, w, [{k: v for k, v in D.items() if k != "x"} for D in layers], 64, dev)
        router.append(run_router(moe, torch, w, 64, l64, head, args.steps, args.warmup, dev, stream, 0.2))
        del l64

    # whole job: bytes of all ranks / slowest rank
    t_max = reduce_max(torch, dev, hr["total_ms"])
    b_all = reduce_sum(torch, dev, hr["bytes"])
    value = b_all / (t_max * 1e-3) / 1e9
    e2e_ms = reduce_max(torch, dev, e2e.pop("_ms"))
    e2e["value"] = round(reduce_sum(torch, dev, e2e.pop("_bytes")) / (e2e_ms * 1e-3) / 1e9, 1)
    e2e["us_per_layer"] = round(e2e["us_per_layer"], 2)

    del layers
    torch.cuda.empty_cache()
    sweep = [] if args.no_sweep else sweep_rows(moe, torch, args, dev, stream, peaks["hbm_gbs"])

    if rank != 0:
        return
    ach = hr["ffn_gbs"]
    roof = {"bound": "hbm", "achieved": round(ach, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
            "frac": round(ach / peaks["hbm_gbs"], 4), "frac_of_8tbs_spec": round(ach / SPEC_HBM_GBS, 4),
            "traffic": recorded_traffic(w.name, head[0], hr["ffn_bytes_per_launch"]),
            "kernel": "ffn_tc_kernel", "peak_source": peaks["source"],
            "algorithmic_bytes_per_launch": round(hr["ffn_bytes_per_launch"]),
            "mean_launch_us": round(hr["ffn_us_mean"], 2)}
    base = None
    if not args.no_cpu_baseline:
        mean_b = float(np.mean(hr["layer_bytes"]))
        base = cpu_baseline(w, B, head, args.cpu_budget,
                            (lambda T: mean_b) if w.int4_cold else (lambda T: layer_bytes(w, B, T)))
    modes = {label: mode_row(r, peaks["hbm_gbs"]) for label, r in results.items()}
    add_vs_topk(modes)
    line = {
        "metric": METRIC, "value": round(value, 1), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t_max / hr["steps_timed"], 5), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic: seeded SplitMix64/Irwin-Hall weights and hidden states, random init",
        "config": config_of(w, B, head, runs, world),
        "timed_regions": hr["reps"], "steps_per_region": args.steps,
        "modes": modes, "sweep": sweep, "router": router, "roofline": roof, "cpu_baseline": base, "e2e": e2e,
        "clocks": clk, "gpu_launches": hr["launches_per_region"],
    }
    print(json.dumps(line), flush=True)
    if args.sweep_out:
        full_sweep(moe, torch, w, dev, stream, args)
    if args.linearity_out:
        linearity(moe, torch, w, dev, stream, args)


def full_sweep(moe, torch, w, dev, stream, args):
    """Per-B rows for the workload's whole batch sweep (written to a file)."""
    rows = []
    peak = measured_peaks()["hbm_gbs"]
    weights = build_weights(moe, torch, w, dev, N_LAYERS)
    for B in (w.batch_sweep or (w.B,)):
        layers = with_batch(moe, torch, w, weights, B, dev)
        res = {}
        for run in w.runs:
            r = run_mode(moe, torch, w, B, layers, run, args.steps, args.warmup, dev, stream,
                         args.sweep_seconds)
            res[run[0]] = dict(workload=w.name, B=B, run=run[0], **mode_row(r, peak))
        add_vs_topk(res)
        rows += list(res.values())
        for r in res.values():
            log(json.dumps(r))
        del layers
    with open(args.sweep_out, "w") as f:
        json.dump(rows, f, indent=1)


def linear_fit(X: np.ndarray, y: np.ndarray) -> dict:
    """Least squares y = X beta; coefficients and R^2."""
    beta, *_ = np.linalg.lstsq(X, y, rcond=None)
    pred = X @ beta
    ss_res = float(np.sum((y - pred) ** 2))
    ss_tot = float(np.sum((y - y.mean()) ** 2))
    return {"coef": [float(b) for b in beta], "r2": 1.0 - ss_res / ss_tot if ss_tot > 0 else 1.0}


def linearity_points(k: int, N: int, B: int) -> list:
    """Forced union sizes T for one batch size: top-min(k, T) routing on T
    experts, so only T <= k is possible for a single token (distinct
    (B, k, T) points only)."""
    pts = []
    for Tt in (1, 2, 4, 8, 16, 24, 32, 48, 64, 96, 128):
        if Tt > N or (B == 1 and Tt > k):
            continue
        pts.append(Tt)
    return pts


def linearity(moe, torch, w, dev, stream, args):
    """Latency against T (distinct activated experts) and sum(cnt_e) (token-
    expert pairs), the OEA page's cost model (section 4: latency grows with
    the number of activated experts).  T is forced by a router bias of +20 on
    T experts drawn with a seeded generator (every token's top-k then lies
    among them) with top-min(k, T) routing, so sum(cnt_e) = B min(k, T);
    B in {1, 4, 16, 64} varies sum(cnt_e) independently of T.  Fits
    us = a sum(cnt_e) + b T + c for the whole layer and the expert kernel,
    over all points and per batch size; b is the cost of one more
    activated expert (a marginal cost, not a bandwidth).  32 distinct
    layers rotate (1.2 GB of experts each at the 30B shapes), so even T = 1
    streams 300 MB per rotation, above the 126 MB L2."""
    import dataclasses
    rows = []
    weights = build_weights(moe, torch, w, dev, 32)
    for B in (1, 4, 16, 64):
        base = with_batch(moe, torch, w, weights, B, dev)
        for Tt in linearity_points(w.k, w.N, B):
            k = min(w.k, Tt)
            wk = dataclasses.replace(w, k=k)
            bias = np.zeros(w.N, np.float32)
            bias[np.random.default_rng(1000 + Tt).choice(w.N, Tt, replace=False)] = 20.0
            bias_d = torch.from_numpy(bias).to(dev)
            layers = [dict(D, bias=bias_d) for D in base]
            r = run_mode(moe, torch, wk, B, layers, ("topk", "topk", k, 1.0), args.steps, args.warmup, dev,
                         stream, args.sweep_seconds, detail_steps=200)
            rows.append({"B": B, "k": k, "T_forced": Tt, "T": r["T_mean"], "sum_cnt": B * k,
                         "us_per_layer": r["us_per_layer"], "ffn_us": r["ffn_us_mean"]})
            log(json.dumps(rows[-1]))
        del base
    del weights
    torch.cuda.empty_cache()
    out = {"workload": w.name, "model": "us = a * sum_cnt + b * T + c", "layers_rotated": 32, "rows": rows}
    for key, col in (("fit_layer", "us_per_layer"), ("fit_expert_kernel", "ffn_us")):
        X = np.array([[r["sum_cnt"], r["T"], 1.0] for r in rows])
        f = linear_fit(X, np.array([r[col] for r in rows]))
        a, b, c = f["coef"]
        out[key] = {"a_us_per_pair": a, "b_us_per_expert": b, "c_us": c, "r2": f["r2"]}
        for Bq in (4, 16, 64):   # per batch size: us = b T + c (sum_cnt fixed for T >= k)
            sel = [r for r in rows if r["B"] == Bq and r["T_forced"] >= w.k]
            if len(sel) >= 3:
                fb = linear_fit(np.array([[r["T"], 1.0] for r in sel]), np.array([r[col] for r in sel]))
                out[key][f"B{Bq}_T_ge_k"] = {"b_us_per_expert": fb["coef"][0], "c_us": fb["coef"][1],
                                             "r2": fb["r2"], "points": len(sel)}
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
    cpu = cpu_description()
    sample = (f"per step: oracle router+routing on the full B={B} batch and single-token expert FFNs "
              f"(8 experts cycled, at least one, for {budget:.3f} s), scaled to one layer's "
              f"(token, expert) pairs; single thread on 1 of {cpu['nproc']} cores ({cpu['cpu_model']})")
    line = {"metric": METRIC, "value": value, "unit": UNIT, "n_gpus": int(os.environ.get("WORLD_SIZE", "1")),
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "impl": "reference",
            "config": config_of(w, B, head, runs, 1),
            "cpu_baseline": {"value": value, "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample, **cpu},
            "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20, help="steps per timed region")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(synth.WORKLOADS))
    ap.add_argument("--batch", type=int, default=0)
    ap.add_argument("--min-seconds", type=float, default=1.0,
                    help="device time the headline run's timed regions add up to at least")
    ap.add_argument("--sweep-seconds", type=float, default=0.25, help="the same for each sweep row")
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-sweep", action="store_true", help="only the headline workload")
    ap.add_argument("--sweep-out", default="", help="the workload's whole batch sweep, written to this file")
    ap.add_argument("--linearity-out", default="", help="latency-vs-T sweep and fit, written to this file")
    ap.add_argument("--layers", type=int, default=8, help="distinct layers rotated through")
    ap.add_argument("--only-run", default="", help="time only this routing run (profiling)")
    args = ap.parse_args()
    global N_LAYERS
    N_LAYERS = args.layers
    if args.warmup < 3:
        ap.error("--warmup must be at least 3")
    if args.steps < 1:
        ap.error("--steps must be at least 1")
    if args.impl == "reference":
        main_reference(args)
    else:
        main_ours(args)


if __name__ == "__main__":
    main()
