#!/usr/bin/env python3
"""Throughput bench of the quantized GEMV / routed-expert library on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Prints ONE JSON line (rank 0).  A step is one call of the hot path on one
batch of synthetic input of the named workload (default: the int4 group-32
GEMV, O = 16384, I = 6144, s = 1).  `value` is weight + scale bytes streamed
per second over the whole job (all ranks); the device timing replays a CUDA
graph of back-to-back calls with inputs resident in HBM, rotating over weight
copies that together exceed twice the L2 (or over fresh routings of the 6 GB
expert store), so no call finds its weights in L2.  `e2e` is the same metric
through the public API with pinned host buffers: each step copies its inputs
host->device and reads its result back.  With more than one rank (torchrun)
every rank runs an independent replica: the path has no exchange step.

--impl reference times the plain f64 CPU oracle on host cores, on bounded
samples of the same workload (rank 0 only).
"""
from __future__ import annotations

import argparse
import dataclasses
import glob
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from weight_only_quantized_qgemv_gb300 import synth  # noqa: E402

METRIC = "achieved weight-stream GB/s (% of GB300 HBM peak); µs per fused expert group"
DEFAULT_WORKLOAD = "int4_g32_16384x6144_s1"
FALLBACK_HBM_GBS = 6800.0
FALLBACK_TENSOR_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 8000.0
FMT_LABEL = {1: "int8-row", 2: "int4-row", 4: "int4-g", 5: "int3-g64", 7: "mxfp4-g32", 8: "mxfp4-e8m0-g32",
             13: "int8-g"}
GROUPED = (synth.INT4_G, synth.INT8_G)   # formats whose group size the caller passes


# ---------------------------------------------------------------------------
# ranks
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def reduce_max(value: float, world: int, device=None) -> float:
    """Max of a float over all ranks (identity for one rank)."""
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def reduce_sum(value: float, world: int, device=None) -> float:
    if world <= 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.SUM)
    return float(t.item())


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ---------------------------------------------------------------------------
# peaks, clocks, traffic record
# ---------------------------------------------------------------------------
def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak():
    """Dense f16 tensor peak for the prefill GEMM: the measured bf16 burst figure
    (f16 and bf16 run at the same nominal dense rate), else the fallback."""
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["bf16_tflops"])
        return v, "bf16_tflops of measured (f16 = bf16 dense rate)"
    except Exception:
        return FALLBACK_TENSOR_TFLOPS, "fallback 1.9 PFLOP/s bf16 (f16 = bf16 dense rate)"


class ClockSampler:
    """nvidia-smi clock/throttle samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"qgemv_clocks_{os.getpid()}.csv")

    def __enter__(self):
        try:
            self.out = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.out, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.out.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        sm, smax, reasons, power = [], [], set(), []
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            p = [c.strip() for c in line.split(",")]
            if len(p) < 9:
                continue
            try:
                sm.append(float(p[1]))
                smax.append(float(p[2]))
                power.append(float(p[3]))
            except ValueError:
                continue
            for n, v in zip(names, p[5:9]):
                if v.lower() == "active":
                    reasons.add(n)
        os.remove(self.path)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def source_hash() -> str:
    h = hashlib.sha256()
    for p in sorted(glob.glob(os.path.join(ROOT, "weight_only_quantized_qgemv_gb300", "csrc", "*"))):
        h.update(open(p, "rb").read())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch of the dominant kernel from the committed ncu
    summary for this workload, if it was taken on the current sources."""
    for path in glob.glob(os.path.join(ROOT, "profiles", "*.md")):
        text = open(path).read()
        if f"workload: {workload}\n" not in text:
            continue
        m = re.search(r"traffic_bytes_per_launch: (\d+)", text)
        hm = re.search(r"source_hash: (\w+)", text)
        if m and hm and hm.group(1) == source_hash():
            return int(m.group(1))
    return None


# ---------------------------------------------------------------------------
# workloads on the device
# ---------------------------------------------------------------------------
class GemvBench:
    def __init__(self, wl, device, l2_bytes):
        import torch
        self.wl = wl
        self.torch = torch
        self.step_bytes = wl.weight_bytes + wl.scale_bytes
        self.ncopies = max(2, -(-2 * l2_bytes // self.step_bytes) + 1)
        self.w, self.sc = [], []
        for c in range(self.ncopies):
            w, sc = wl.weights(copy=c)
            self.w.append(torch.from_numpy(w).to(device))
            self.sc.append(torch.from_numpy(sc).to(device))
        self.x_host = wl.x()
        self.x = torch.from_numpy(self.x_host).to(device)
        self.y = torch.empty(wl.s, wl.O, dtype=torch.float32, device=device)
        self.gs = wl.gs if wl.fmt in GROUPED else 0
        self.launches_per_step = 1
        if wl.gemm:     # prefill: the tensor-core GEMM, its x split and its workspace
            from weight_only_quantized_qgemv_gb300 import qgemm_workspace
            self.ws_bytes = qgemm_workspace(wl.I, wl.s)
            self.ws = torch.empty(self.ws_bytes, dtype=torch.uint8, device=device)
            self.launches_per_step = 2
        self.l2_note = f"rotates {self.ncopies} weight copies ({self.ncopies * self.step_bytes / 1e6:.0f} MB > 2x L2)"

    def call(self, c, stream):
        from weight_only_quantized_qgemv_gb300 import qgemm, qgemv
        wl = self.wl
        if wl.gemm:
            qgemm(wl.fmt, self.gs, self.w[c], self.sc[c], self.x, wl.O, wl.I, wl.s, self.y, self.ws, self.ws_bytes,
                  stream)
        else:
            qgemv(wl.fmt, self.gs, self.w[c], self.sc[c], self.x, wl.O, wl.I, wl.s, self.y, stream)

    def step(self, i, stream):
        self.call(i % self.ncopies, stream)

    def period(self):
        return self.ncopies

    def bytes_of(self, i):
        return self.step_bytes

    def e2e_setup(self):
        torch = self.torch
        self.x_pin = torch.from_numpy(self.x_host.copy()).pin_memory()
        self.y_pin = torch.empty(self.wl.s, self.wl.O, dtype=torch.float32).pin_memory()
        return self.x_pin.numel() * 4, self.y_pin.numel() * 4

    def e2e_step(self, i, stream):
        self.x.copy_(self.x_pin, non_blocking=True)
        self.call(i % self.ncopies, stream)
        self.y_pin.copy_(self.y, non_blocking=True)

    def config(self):
        cfg = gemv_config(self.wl)
        cfg["l2"] = self.l2_note
        return cfg


class ExpertBench:
    def __init__(self, wl, device, swiglu_limit=None, device_route=False):
        import torch
        from weight_only_quantized_qgemv_gb300 import QACT_SWIGLU, QACT_SWIGLU_CLAMPED, qexpert_group_workspace
        self.wl = wl
        # activation: SwiGLU, or clamped SwiGLU with the given limit
        self.act = QACT_SWIGLU if swiglu_limit is None else QACT_SWIGLU_CLAMPED
        self.limit = 0.0 if swiglu_limit is None else float(swiglu_limit)
        self.torch = torch
        self.d = {}
        for name, which in wl.MATRICES:
            nb, ns = wl.sizes(which)
            self.d[name] = torch.empty(wl.E * nb, dtype=torch.uint8, device=device)
            self.d[name + "_s"] = torch.empty(wl.E * ns, dtype=torch.uint8 if wl.fmt == synth.MXFP4_E8M0
                                              else torch.float32, device=device)

        def sink(name, slot, w, sc):
            self.d[name][slot * w.size:(slot + 1) * w.size].copy_(torch.from_numpy(w))
            self.d[name + "_s"][slot * sc.size:(slot + 1) * sc.size].copy_(torch.from_numpy(sc))

        wl.generate(range(wl.E), sink)
        torch.cuda.synchronize()
        self.nroutes = 64      # seeded routings the calls rotate over (each over a 6 GB store)
        ids, wts, xs = [], [], []
        for r in range(self.nroutes):
            i, w = wl.routing(step=r)
            ids.append(i)
            wts.append(w)
            xs.append(wl.x(step=r))
        self.ids_host = np.stack(ids).astype(np.int32)
        self.wts_host = np.stack(wts).astype(np.float32)
        self.x_host = np.stack(xs).astype(np.float32)
        self.ids = torch.from_numpy(self.ids_host).to(device)
        self.wts = torch.from_numpy(self.wts_host).to(device)
        self.x = torch.from_numpy(self.x_host).to(device)
        self.out = torch.empty(wl.s, wl.D, dtype=torch.float32, device=device)
        self.ws_bytes = qexpert_group_workspace(wl.E, wl.D, wl.F, wl.s, wl.k)
        self.ws = torch.zeros(self.ws_bytes, dtype=torch.uint8, device=device)   # zeroed before first use
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.gs = wl.gs if wl.fmt in GROUPED else 0
        self.expert_bytes = wl.expert_bytes()
        self.route_bytes = [len(np.unique(self.ids_host[r])) * self.expert_bytes for r in range(self.nroutes)]
        # the library says how many launches a call makes: one persistent
        # launch up to 256 (token, rank) pairs, else prep, gate/up, down, combine
        from weight_only_quantized_qgemv_gb300 import qexpert_group_launches
        self.launches_per_step = qexpert_group_launches(wl.fmt, self.gs, wl.E, wl.D, wl.F, wl.s, wl.k,
                                                        routed=device_route)
        self.fused = self.launches_per_step == 1
        self.device_route = device_route
        if device_route:
            # routing on the device from seeded logits: softmax top-k, renormalized
            self.logits_host = np.stack([wl.router_logits(step=r) for r in range(self.nroutes)])
            self.logits = torch.from_numpy(self.logits_host).to(device)
            self.ids_out = torch.empty(wl.s, wl.k, dtype=torch.int32, device=device)
            self.wts_out = torch.empty(wl.s, wl.k, dtype=torch.float32, device=device)
            top = np.argpartition(-self.logits_host, wl.k - 1, axis=2)[:, :, :wl.k]
            self.route_bytes = [len(np.unique(top[r])) * self.expert_bytes for r in range(self.nroutes)]

    def _call(self, r, x, ids, wts, stream, logits=None):
        from weight_only_quantized_qgemv_gb300 import QROUTE_SOFTMAX, qexpert_group_act, qexpert_group_routed
        wl, d = self.wl, self.d
        if self.device_route:
            qexpert_group_routed(wl.fmt, self.gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"],
                                 wl.E, wl.D, wl.F, x, wl.s, wl.k, QROUTE_SOFTMAX,
                                 self.logits[r] if logits is None else logits, None, 1, 1.0, self.act, self.limit,
                                 self.out, self.ids_out, self.wts_out, self.ws, self.ws_bytes, self.status, stream)
            return
        qexpert_group_act(wl.fmt, self.gs, d["gate"], d["gate_s"], d["up"], d["up_s"], d["down"], d["down_s"],
                          wl.E, wl.D, wl.F, x, wl.s, wl.k, ids, wts, self.act, self.limit, self.out, self.ws,
                          self.ws_bytes, self.status, stream)

    def step(self, i, stream):
        r = i % self.nroutes
        self._call(r, self.x[r], self.ids[r], self.wts[r], stream)

    def period(self):
        return self.nroutes

    def bytes_of(self, i):
        return self.route_bytes[i % self.nroutes]

    def e2e_setup(self):
        torch = self.torch
        self.x_pin = torch.from_numpy(self.x_host.copy()).pin_memory()
        self.ids_pin = torch.from_numpy(self.ids_host.copy()).pin_memory()
        self.wts_pin = torch.from_numpy(self.wts_host.copy()).pin_memory()
        self.out_pin = torch.empty(self.wl.s, self.wl.D, dtype=torch.float32).pin_memory()
        self.x1 = torch.empty_like(self.x[0])
        self.ids1 = torch.empty_like(self.ids[0])
        self.wts1 = torch.empty_like(self.wts[0])
        if self.device_route:
            self.logits_pin = torch.from_numpy(self.logits_host.copy()).pin_memory()
            self.logits1 = torch.empty_like(self.logits[0])
            return (self.x1.numel() + self.logits1.numel()) * 4, self.out_pin.numel() * 4
        h2d = (self.x1.numel() + self.ids1.numel() + self.wts1.numel()) * 4
        return h2d, self.out_pin.numel() * 4

    def e2e_step(self, i, stream):
        r = i % self.nroutes
        self.x1.copy_(self.x_pin[r], non_blocking=True)
        if self.device_route:
            self.logits1.copy_(self.logits_pin[r], non_blocking=True)
            self._call(r, self.x1, None, None, stream, logits=self.logits1)
            self.out_pin.copy_(self.out, non_blocking=True)
            return
        self.ids1.copy_(self.ids_pin[r], non_blocking=True)
        self.wts1.copy_(self.wts_pin[r], non_blocking=True)
        self._call(r, self.x1, self.ids1, self.wts1, stream)
        self.out_pin.copy_(self.out, non_blocking=True)

    def config(self):
        wl = self.wl
        cfg = expert_config(wl)
        cfg["l2"] = f"{self.nroutes} seeded routings over the {wl.E * self.expert_bytes / 1e9:.2f} GB store (> L2)"
        cfg["mean_experts_per_step"] = float(np.mean([len(np.unique(r)) for r in self.ids_host]))
        cfg["activation"] = "swiglu" if self.act == 0 else f"swiglu clamped at {self.limit:g}"
        if self.device_route:
            cfg["routing"] = "on the device: softmax top-k of seeded N(0,1) router logits, renormalized (qroute)"
            cfg["mean_experts_per_step"] = float(np.mean(self.route_bytes) / self.expert_bytes)
        else:
            cfg["routing"] = "host draws (k distinct experts, softmax of k N(0,1) logits)"
        return cfg


# ---------------------------------------------------------------------------
# CPU baseline: the oracle on a bounded sample
# ---------------------------------------------------------------------------
def oracle_sample_runner(wl, target_s: float, swiglu_limit=None):
    """A callable running the oracle on a sample of the workload, the bytes it
    covers, and a description.  Sized to ~target_s seconds."""
    from oracle import oracle as orc

    if isinstance(wl, synth.GemvWorkload):
        w, sc = wl.weights()
        x = wl.x()
        per_row = (wl.weight_bytes + wl.scale_bytes) // wl.O

        def run(nrows, start=0):
            rows = (np.arange(nrows) + start) % wl.O
            orc.qgemv_rows(wl.fmt, wl.gs, w, sc, x, wl.O, wl.I, rows)
            return nrows * per_row

        t = time.perf_counter()
        run(256)
        dt = max(time.perf_counter() - t, 1e-6) / 256
        nrows = int(max(16, target_s / dt))
        return ((lambda i=0: run(nrows, start=i * nrows)),
                f"{nrows} rows (cycling over the {wl.O} rows), all {wl.s} activation rows")

    # expert group: gate/up rows of the first routed expert of token 0 (the
    # oracle's fused gate/up arithmetic), sized to the target time
    ids, _ = wl.routing(step=0)
    x = wl.x(step=0)[:1]
    st = wl.store(ids[0, :1])
    per_row = 2 * (synth.packed_bytes(wl.fmt, 1, wl.D) + synth.scale_itemsize(wl.fmt) * (wl.D // wl.gs))

    def run_rows(nrows, start=0):
        rows = (np.arange(nrows) + start) % wl.F
        orc.qgate_up_rows(wl.fmt, wl.gs, st["gate"], st["gate_s"], st["up"], st["up_s"], x, wl.F, wl.D, rows,
                          act=0 if swiglu_limit is None else 1, limit=swiglu_limit or 0.0)
        return nrows * per_row

    t = time.perf_counter()
    run_rows(256)
    dt = max(time.perf_counter() - t, 1e-6) / 256
    nrows = int(max(16, target_s / dt))
    return ((lambda i=0: run_rows(nrows, start=i * nrows)),
            f"{nrows} gate/up rows (cycling over the {wl.F} rows) of expert {int(ids[0, 0])} (token 0, first routing)")


def _time_oracle(wl, target_s, swiglu_limit):
    """GB/s of the oracle over samples of about a second, repeated until about
    target_s seconds of CPU work, and a description of the sample."""
    run, desc = oracle_sample_runner(wl, min(1.0, target_s), swiglu_limit)
    t = time.perf_counter()
    nbytes, n = 0, 0
    while True:
        nbytes += run(n)
        n += 1
        dt = time.perf_counter() - t
        if dt >= target_s:
            break
    return nbytes / dt / 1e9, f"{n} samples of {desc}; {dt:.1f} s"


def cpu_baseline(wl, target_s=12.0, swiglu_limit=None):
    """The oracle on all the host cores (OpenMP over output rows), and on one
    core for about half as long."""
    from oracle import oracle as orc
    cores = orc.threads()
    value, sample = _time_oracle(wl, target_s, swiglu_limit)
    out = {"value": value, "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": sample}
    if cores > 1:
        orc.set_threads(1)
        try:
            v1, sample1 = _time_oracle(wl, target_s / 2, swiglu_limit)
        finally:
            orc.set_threads(cores)
        out["single_core"] = {"value": v1, "unit": "GB/s", "cores": 1, "sample": sample1}
    return out


def reference_arm(args, wl, world, rank):
    if rank != 0:
        return
    from oracle import oracle as orc
    orc.build()
    target = args.sample_seconds if args.sample_seconds else max(0.5, 60.0 / max(1, args.steps + args.warmup))
    run, desc = oracle_sample_runner(wl, target_s=target, swiglu_limit=args.swiglu_limit)
    for i in range(args.warmup):
        run(i)
    t = time.perf_counter()
    nbytes = 0
    for i in range(args.steps):
        nbytes += run(args.warmup + i)
    dt = time.perf_counter() - t
    value = nbytes / dt / 1e9
    cfg = gemv_config(wl) if isinstance(wl, synth.GemvWorkload) else expert_config(wl)
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": cfg,
            "cpu_baseline": {"value": value, "unit": "GB/s", "cores": orc.threads(), "kind": "oracle",
                             "sample": desc + " per step"},
            "e2e": {"value": value, "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)


def percentiles(us):
    a = np.asarray(us, dtype=np.float64)
    return {"p10": float(np.percentile(a, 10)), "p50": float(np.percentile(a, 50)),
            "p90": float(np.percentile(a, 90))}


def largest_divisor_at_most(n: int, cap: int) -> int:
    for g in range(min(n, cap), 0, -1):
        if n % g == 0:
            return g
    return 1


class GraphSet:
    """CUDA graphs of G back-to-back calls whose replays, taken in order, continue
    the rotation over the workload's weight copies (or routings): graph j holds
    calls j*G .. j*G + G - 1 of an endless sequence, modulo the rotation period,
    so no replay boundary brings a copy back sooner than the period does."""

    def __init__(self, bench, G, stream, torch, max_graphs=64):
        self.G = G
        period = bench.period()
        self.n = max(1, min(math.lcm(G, period) // G, max_graphs))
        self.graphs = []
        self.bytes = []
        for gi in range(self.n):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream):
                for j in range(G):
                    bench.step(gi * G + j, torch.cuda.current_stream().cuda_stream)
            self.graphs.append(g)
            self.bytes.append(sum(bench.bytes_of(gi * G + j) for j in range(G)))
        self.next = 0
        with torch.cuda.stream(stream):        # warm: every graph once
            for g in self.graphs:
                g.replay()
        stream.synchronize()

    def replay(self):
        """Replays the next graph of the rotation; returns the bytes its calls stream."""
        i = self.next
        self.graphs[i].replay()
        self.next = (i + 1) % self.n
        return self.bytes[i]


def timed_regions(gs, K, stream, torch, min_regions=200, min_seconds=1.0, est_call_s=1e-5):
    """Times regions of exactly K calls (K / G graph replays) with CUDA events on
    the launching stream, back to back, at least min_regions of them and about
    min_seconds in all.  Returns [(seconds, bytes)] per region."""
    per_region = K // gs.G
    n = max(min_regions, int(math.ceil(min_seconds / max(est_call_s * K, 1e-9))))
    n = min(n, 200000)
    evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
    nbytes = []
    with torch.cuda.stream(stream):
        for a, b in evs:
            a.record(stream)
            tot = 0
            for _ in range(per_region):
                tot += gs.replay()
            b.record(stream)
            nbytes.append(tot)
    torch.cuda.synchronize()
    return [(a.elapsed_time(b) / 1e3, nb) for (a, b), nb in zip(evs, nbytes)]


def eager_distribution(bench, stream, torch, per_call_s, gs, n_eager=200):
    """Single calls, each alone between two events, enqueued behind tens of
    milliseconds of graph replays so the device never waits on the host; the
    event between two calls keeps one call from starting under the previous."""
    lead = max(1, int(-(-(20e-3 + 60e-6 * n_eager) // max(per_call_s * gs.G, 1e-9))))
    calls = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n_eager)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for _ in range(lead):
            gs.replay()
        for i, (a, b) in enumerate(calls):
            a.record(stream)
            bench.step(i, stream.cuda_stream)
            b.record(stream)
    torch.cuda.synchronize()
    return percentiles([a.elapsed_time(b) * 1e3 for a, b in calls])


def e2e_rate(bench, stream, torch, steps, world, device):
    """The metric through the public API from pinned host buffers: every step
    copies its inputs host -> device, calls, and reads its result back, then
    synchronizes.  Returns (GB/s over all ranks, us per step, h2d, d2h, steps)."""
    h2d, d2h = bench.e2e_setup()
    barrier(world)
    torch.cuda.synchronize()
    nbytes = 0
    t = time.perf_counter()
    with torch.cuda.stream(stream):
        for i in range(steps):
            bench.e2e_step(i, stream.cuda_stream)
            stream.synchronize()
            nbytes += bench.bytes_of(i)
    dt = reduce_max(time.perf_counter() - t, world, device)
    return reduce_sum(float(nbytes), world, device) / dt / 1e9, dt / steps * 1e6, h2d, d2h, steps


def gemv_kernel_name(wl, sms=152):
    """The kernel one qgemv call of this workload runs (the library's automatic choice):
    the tile kernel for int3 and several activation rows, and for one row when
    lanes share scales (per-row scales, ue8m0 words, groups longer than a
    chunk) on a matrix with at least 64 rows per SM and a tile plan that fits.
    Prefill workloads run qgemm."""
    if wl.gemm:
        return "whole qgemm call (k_gemm_split_x + k_gemm, tcgen05)"
    if wl.s > 1 or wl.fmt == synth.INT3_G64:
        return "k_tile"
    int8 = wl.fmt in (synth.INT8_ROW, synth.INT8_G)
    codes_per_chunk, codes_per_slice = (16, 512) if int8 else (32, 1024)
    if wl.fmt in (synth.INT8_ROW, synth.INT4_ROW):
        shares, fits = True, True
    elif wl.fmt == synth.MXFP4_E8M0:
        shares, fits = True, wl.I % 512 == 0
    elif wl.fmt in GROUPED:
        shares = wl.gs > codes_per_chunk
        fits = codes_per_slice % wl.gs == 0 and 4 * codes_per_slice // wl.gs >= 16 and (4 * wl.I // wl.gs) % 16 == 0
    else:
        shares, fits = False, False
    short = -(-wl.O // sms) < 64
    return "k_tile" if (shares and fits and not short) else "k_stream"


def expert_kernel_name(bench):
    """The launches one qexpert_group call of this workload runs."""
    if bench.fused:
        return "k_moe (the whole expert group in one launch)"
    return "whole qexpert_group call (k_expert_prep + k_tile gate/up + k_tile down + k_expert_combine)"


def gemv_config(wl):
    return {"workload": wl.name, "kind": "qgemv", "fmt": FMT_LABEL[wl.fmt] + (str(wl.gs) if wl.fmt in GROUPED else ""),
            "O": wl.O, "I": wl.I, "s": wl.s, "gs": wl.gs, "parallelism": "replicas"}


def expert_config(wl):
    return {"workload": wl.name, "kind": "qexpert_group", "fmt": FMT_LABEL[wl.fmt] + (str(wl.gs) if wl.fmt in GROUPED else ""),
            "E": wl.E, "D": wl.D, "F": wl.F, "s": wl.s, "k": wl.k, "gs": wl.gs, "parallelism": "replicas"}


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------
def make_bench(wl, device, l2, swiglu_limit=None, device_route=False):
    if isinstance(wl, synth.GemvWorkload):
        return GemvBench(wl, device, l2)
    return ExpertBench(wl, device, swiglu_limit, device_route)


def est_call_seconds(wl):
    """A rough duration of one call, to size the timed regions."""
    if isinstance(wl, synth.GemvWorkload) and wl.gemm:
        return 2.0 * wl.O * wl.I * wl.s / 3e14 + 30e-6
    if isinstance(wl, synth.GemvWorkload):
        return (wl.weight_bytes + wl.scale_bytes) / 5e12 + 2e-6
    return 0.9 * wl.s * wl.k * wl.expert_bytes() / 5e12 + 10e-6


def kernel_name(bench):
    if isinstance(bench, GemvBench):
        return gemv_kernel_name(bench.wl)
    return expert_kernel_name(bench)


def workload_line(name, args, device, l2, stream, torch, peak, e2e_steps=200):
    """One workload of the configs block: us per call over >= 200 timed graph
    replays of 64 back-to-back calls, GB/s, roofline fractions, traffic and
    the kernel, plus the same calls end to end from host buffers."""
    wl = synth.workload(name)
    bench = make_bench(wl, device, l2, None if isinstance(wl, synth.GemvWorkload) else args.swiglu_limit)
    with torch.cuda.stream(stream):
        for i in range(3):
            bench.step(i, stream.cuda_stream)
    stream.synchronize()
    gs = GraphSet(bench, 64, stream, torch)
    res = timed_regions(gs, 64, stream, torch, min_regions=200, min_seconds=0.5, est_call_s=est_call_seconds(wl))
    us = [t / 64 * 1e6 for t, _ in res]
    gbs = [nb / t / 1e9 for t, nb in res]
    p = percentiles(us)
    g50 = float(np.median(gbs))
    e2e_gbs, e2e_us, h2d, d2h, n = e2e_rate(bench, stream, torch, e2e_steps, 1, device)
    line = {"us_per_call": p, "GBps": g50, "frac": g50 / peak, "frac_of_8000": g50 / NOMINAL_HBM_GBS,
            "bytes_per_call": float(np.mean([nb / 64 for _, nb in res])), "traffic": recorded_traffic(name),
            "kernel": kernel_name(bench), "launches_per_call": bench.launches_per_step, "replays": len(res),
            "calls_per_replay": 64,
            "e2e": {"GBps": e2e_gbs, "us_per_call": e2e_us, "h2d_bytes": h2d, "d2h_bytes": d2h, "steps": n}}
    if isinstance(wl, synth.GemvWorkload) and wl.gemm:
        tpeak, _ = tensor_peak()
        tf = 2.0 * wl.O * wl.I * wl.s / (p["p50"] * 1e-6) / 1e12
        line.update({"bound": "tensor", "TFLOPs": tf, "frac": tf / tpeak, "frac_of_8000": None})
    elif isinstance(wl, synth.ExpertWorkload):
        line["us_per_fused_expert_group"] = p
        line["mean_experts_per_call"] = float(np.mean(bench.route_bytes) / bench.expert_bytes)
    del gs, bench
    torch.cuda.empty_cache()
    return line


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=64)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD,
                    choices=synth.WORKLOADS + synth.VARIANT_WORKLOADS + synth.PREFILL_WORKLOADS)
    ap.add_argument("--impl", default="native", choices=["native", "reference"])
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-configs", action="store_true", help="skip the per-workload configs block")
    ap.add_argument("--all-workloads", action="store_true",
                    help="configs block over the variant and prefill workloads too")
    ap.add_argument("--min-regions", type=int, default=200, help="timed regions of --steps calls (median taken)")
    ap.add_argument("--sample-seconds", type=float, default=None,
                    help="CPU seconds per oracle sample (reference arm / CPU baseline)")
    ap.add_argument("--device-route", action="store_true",
                    help="expert workloads: route on the device from seeded router logits (qexpert_group_routed)")
    ap.add_argument("--swiglu-limit", type=float, default=None,
                    help="expert workloads: clamped SwiGLU with this limit instead of SwiGLU")
    ap.add_argument("--experts", type=int, default=None,
                    help="expert workloads, for profiler captures: a store of this many experts instead of the "
                         "workload's (each call still routes every token to k distinct experts, so a call's "
                         "work is unchanged; the store, and so the device memory, shrinks)")
    args = ap.parse_args()
    wl = synth.workload(args.workload)
    if args.experts is not None:
        if not isinstance(wl, synth.ExpertWorkload) or not (wl.k <= args.experts <= wl.E):
            raise SystemExit("--experts applies to expert workloads, between k and the workload's E")
        wl = dataclasses.replace(wl, E=args.experts, _cache={})
    world, rank, local = dist_env()
    args.steps = max(1, args.steps)
    args.warmup = max(3, args.warmup)

    if args.impl == "reference":
        reference_arm(args, wl, world, rank)
        return

    import torch
    if not torch.cuda.is_available():
        raise SystemExit("bench.py needs a CUDA GPU (the library has no CPU path)")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=device)
    from weight_only_quantized_qgemv_gb300 import _build, _lib
    if rank == 0 or not _build.up_to_date():
        _build.build()
    barrier(world)
    _lib.lib()

    props = torch.cuda.get_device_properties(device)
    l2 = getattr(props, "L2_cache_size", 0) or 132 * 1024 * 1024
    peak, peak_src = hbm_peak()
    stream = torch.cuda.Stream(device)
    bench = make_bench(wl, device, l2, args.swiglu_limit, args.device_route)

    # warm-up: W eager steps, then the graphs (their capture and first replay warm up too)
    with torch.cuda.stream(stream):
        for i in range(args.warmup):
            bench.step(i, stream.cuda_stream)
    stream.synchronize()
    K = args.steps
    G = largest_divisor_at_most(K, 64)
    gs = GraphSet(bench, G, stream, torch)

    # timed: regions of exactly K calls, at least --min-regions of them (about a
    # second in all, so the clock samples see the load); the median region
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize()
        res = timed_regions(gs, K, stream, torch, min_regions=args.min_regions, min_seconds=1.0,
                            est_call_s=est_call_seconds(wl))
        torch.cuda.synchronize()
        barrier(world)
    clocks = clk.summary()
    times = np.array([t for t, _ in res])
    region_bytes = np.array([nb for _, nb in res], dtype=np.float64)
    i_med = int(np.argsort(times)[len(times) // 2])
    t_med = float(times[i_med])
    t_max = reduce_max(t_med, world, device)
    total_bytes = reduce_sum(float(region_bytes[i_med]), world, device)
    value = total_bytes / t_max / 1e9
    per_launch_s = t_med / K
    achieved = region_bytes[i_med] / K / per_launch_s / 1e9
    timing = {"regions": len(res), "steps_per_region": K, "graph_calls_per_replay": G,
              "us_per_call": percentiles(times / K * 1e6),
              "timed_seconds": float(times.sum()),
              "eager_us_per_call": eager_distribution(bench, stream, torch, per_launch_s, gs)}

    # end to end through the public API, host buffers, copies inside the timed region
    e2e_value, e2e_us, h2d, d2h, k_e2e = e2e_rate(bench, stream, torch, min(max(K, 200), 2000), world, device)
    barrier(world)
    launches = bench.launches_per_step
    kname = kernel_name(bench)
    cfg = bench.config()
    del gs, bench
    torch.cuda.empty_cache()

    if rank != 0:
        if world > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    configs = None
    if not args.no_configs:
        names = list(synth.WORKLOADS) + (synth.VARIANT_WORKLOADS + synth.PREFILL_WORKLOADS
                                         if args.all_workloads else [])
        configs = {n: workload_line(n, args, device, l2, stream, torch, peak) for n in names}
    cpu = None
    if not args.no_cpu_baseline:
        cpu = cpu_baseline(wl, args.sample_seconds or 12.0, args.swiglu_limit)
    cfg["graph_calls_per_replay"] = G
    roof = {"bound": "hbm", "achieved": achieved, "peak": peak, "unit": "GB/s",
            "frac": achieved / peak, "peak_source": f"hbm_gbs of {peak_src}",
            "frac_of_8000": achieved / NOMINAL_HBM_GBS,
            "traffic": recorded_traffic(wl.name),
            "algorithmic_bytes_per_launch": float(region_bytes[i_med] / K), "kernel": kname}
    if isinstance(wl, synth.GemvWorkload) and wl.gemm:
        # a prefill batch is a dense contraction: the tensor roofline, on the
        # algorithmic 2 O I s flops (the two-part split of x doubles the MMAs)
        tpeak, tsrc = tensor_peak()
        flops = 2.0 * wl.O * wl.I * wl.s
        roof = {"bound": "tensor", "achieved": flops / per_launch_s / 1e12, "peak": tpeak, "unit": "TFLOP/s",
                "frac": flops / per_launch_s / 1e12 / tpeak, "peak_source": tsrc,
                "traffic": recorded_traffic(wl.name), "algorithmic_flops_per_launch": flops,
                "mma_flops_per_launch": 2 * flops, "weight_stream_gbs": achieved, "kernel": kname}
    line = {
        "metric": METRIC, "value": value, "unit": "GB/s", "n_gpus": world, "steps": K,
        "warmup": args.warmup, "ms_per_step": t_max / K * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic", "config": cfg,
        "us_per_call": per_launch_s * 1e6,
        "timing": timing,
        "roofline": roof,
        "clocks": clocks,
        "e2e": {"value": e2e_value, "unit": "GB/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": k_e2e, "us_per_step": e2e_us},
        "gpu_launches": K * launches,
        "gpu_launches_all_regions": K * launches * len(res),
        "configs": configs,
        "cpu_baseline": cpu,
    }
    print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
