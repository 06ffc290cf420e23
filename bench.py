#!/usr/bin/env python3
"""Benchmark of the GGUF block-quantized matmul library on one GB300.

A step is one pass of the Q4_0 decode-layer GEMV set at M = 1 (seven
projections with hidden size 2048: q 2048->2048, k 2048->512, v 2048->512,
o 2048->2048, gate 2048->8192, up 2048->8192, down 8192->2048), i.e. the
Q4_0 dispatches of a Gemma4-style decode layer whose count per token is given
in "Add generated quant-kernel JIT and accelerate Gemma4, BGE-M3, and
GLiNER2", section "Validation".  The metric is weight GB/s: the Q4_0 bytes a
step streams (34,209,792) times steps, over the device time.

Timing: inputs are resident in HBM; R weight replicas (footprint >= 4x L2)
rotate so that no step finds its weights in L2; the steps are replayed from
CUDA graphs and timed with CUDA events on the launching stream, with a
barrier and a device synchronise on both sides, max over ranks.  SM clocks
and throttle reasons are sampled with nvidia-smi during the timed region.

`e2e` repeats the step through the public API with host buffers: each step
copies its activations from pinned host memory, runs the step's calls and
copies the outputs back (weights stay resident: they are the model).

`--impl reference` times the CPU oracle (the plain C definition) on the
box's host cores, on a bounded sample of the same workload.

Other workloads (single small GEMV, batched GEMV, Q8_0 LM head, dequant,
prefill GEMM) are measured the same way and reported under "secondary".

Under torchrun each rank runs an independent replica of the workload on its
own GPU (replicas only: the path has no exchange step).
"""
from __future__ import annotations

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

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

from block_quantized_matmul_gguf_gb300 import synth  # noqa: E402

METRIC = "quant GEMV weight GB/s (% of HBM peak); Q4_0 prefill GEMM TFLOP/s"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}
# Non-tensor FP32 FMA peak from unit counts and clock (no measured figure is
# available): 152 SMs x 128 FMA lanes x 2 flop per cycle at the maximum SM clock.
GB300_SMS = 152
FP32_LANES_PER_SM = 128


def fp32_peak_tflops(peaks) -> float:
    return GB300_SMS * FP32_LANES_PER_SM * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32000)
    ap.add_argument("--warmup", type=int, default=320)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary workloads (headline only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--profile", default=None, metavar="CASE",
                    help="no timing: run CASE a few times for a profiler and exit. CASE is "
                         "decode_grouped (the timed decode step), decode (seven separate calls), "
                         "gemv:FMT:M:N:K, geglu:M:N:K, gemm_geglu:M:N:K, dequant:FMT:N:K "
                         "gemm:M:N:K, gemm_ws:M:N:K (two-phase) or gemm_q8_0:M:N:K")
    ap.add_argument("--profile-launches", type=int, default=3)
    return ap.parse_args(argv)


def run_profile(args):
    """Launch one small case a few times (for ncu), untimed."""
    import torch
    from block_quantized_matmul_gguf_gb300 import qmm
    torch.cuda.set_device(0)
    dev = torch.device("cuda:0")
    parts = args.profile.split(":")
    reps = args.profile_launches
    if parts[0] == "decode_grouped":
        # the timed step: q+k+v (shared x), o, gate+up (shared x), down
        cases = [synth.gemv_case("q4_0", 1, p.n, p.k, seed=0, stream=10 + i)
                 for i, p in enumerate(synth.DECODE_LAYER)]
        names = [p.name for p in synth.DECODE_LAYER]
        W = [torch.from_numpy(c.w).to(dev) for c in cases]
        Y = [torch.empty((1, c.n), dtype=torch.float32, device=dev) for c in cases]
        groups = [[names.index(nm) for nm in g] for g in DECODE_GROUPS]
        X = [torch.from_numpy(cases[g[0]].x).to(dev) for g in groups]
        for _ in range(reps):
            for g, x in zip(groups, X):
                qmm.qmm_gemv_q4_0_multi([(W[i], Y[i], cases[i].n) for i in g], x, 1,
                                        cases[g[0]].k)
    elif parts[0] == "geglu":
        m, n, k = int(parts[1]), int(parts[2]), int(parts[3])
        wg = torch.from_numpy(synth.q4_0_weights(n, k, seed=0, stream=14)).to(dev)
        wu = torch.from_numpy(synth.q4_0_weights(n, k, seed=0, stream=15)).to(dev)
        x = torch.from_numpy(synth.activations_f32(m, k, seed=0, stream=16)).to(dev)
        for _ in range(reps):
            qmm.geglu_q4_0(wg, wu, x, n, k)
    elif parts[0] == "gemm_geglu":
        m, n, k = int(parts[1]), int(parts[2]), int(parts[3])
        wg, xb = synth.gemm_case(m, n, k, seed=0, stream=80)
        wu = synth.q4_0_weights(n, k, seed=0, stream=81)
        WG, WU = torch.from_numpy(wg).to(dev), torch.from_numpy(wu).to(dev)
        X = torch.from_numpy(xb.astype(np.int16)).to(dev)
        for _ in range(reps):
            qmm.gemm_geglu_q4_0(WG, WU, X, n, k)
    elif parts[0] == "decode":
        cases = [synth.gemv_case("q4_0", 1, p.n, p.k, seed=0, stream=10 + i)
                 for i, p in enumerate(synth.DECODE_LAYER)]
        W = [torch.from_numpy(c.w).to(dev) for c in cases]
        X = [torch.from_numpy(c.x).to(dev) for c in cases]
        for _ in range(reps):
            for c, w, x in zip(cases, W, X):
                qmm.gemv("q4_0", w, x, c.n, c.k)
    elif parts[0] == "gemv":
        fmt, m, n, k = parts[1], int(parts[2]), int(parts[3]), int(parts[4])
        c = synth.gemv_case(fmt, m, n, k, seed=0, stream=1)
        w, x = torch.from_numpy(c.w).to(dev), torch.from_numpy(c.x).to(dev)
        for _ in range(reps):
            qmm.gemv(fmt, w, x, n, k)
    elif parts[0] == "dequant":
        fmt, n, k = parts[1], int(parts[2]), int(parts[3])
        c = synth.gemv_case(fmt, 1, n, k, seed=0, stream=1)
        w = torch.from_numpy(c.w).to(dev)
        for _ in range(reps):
            qmm.dequant(fmt, w, n, k)
    elif parts[0] == "gemm":
        m, n, k = int(parts[1]), int(parts[2]), int(parts[3])
        w, xb = synth.gemm_case(m, n, k, seed=0, stream=1)
        W = torch.from_numpy(w).to(dev)
        X = torch.from_numpy(xb.astype(np.int16)).to(dev)
        for _ in range(reps):
            qmm.gemm_q4_0(W, X, n, k)
    elif parts[0] == "gemm_ws":
        m, n, k = int(parts[1]), int(parts[2]), int(parts[3])
        w, xb = synth.gemm_case(m, n, k, seed=0, stream=1)
        W = torch.from_numpy(w).to(dev)
        X = torch.from_numpy(xb.astype(np.int16)).to(dev)
        WS = torch.empty(qmm.qmm_gemm_workspace_bytes(n, k), dtype=torch.uint8, device=dev)
        for _ in range(reps):
            qmm.gemm("q4_0", W, X, n, k, workspace=WS)
    elif parts[0] == "gemm_q8_0":
        m, n, k = int(parts[1]), int(parts[2]), int(parts[3])
        W = torch.from_numpy(synth.q8_0_weights(n, k, seed=0, stream=75)).to(dev)
        X = torch.from_numpy(synth.activations_bf16(m, k, seed=0, stream=76).astype(np.int16)).to(dev)
        for _ in range(reps):
            qmm.gemm("q8_0", W, X, n, k)
    else:
        raise SystemExit(f"unknown profile case {args.profile}")
    torch.cuda.synchronize()
    err = qmm.qmm_get_device_error()
    print(json.dumps({"profile": args.profile, "launches": reps, "device_error": err}))
    if err:
        raise SystemExit(1)


# ----------------------------------------------------------------- distributed

class Dist:
    def __init__(self):
        self.world = int(os.environ.get("WORLD_SIZE", "1"))
        self.rank = int(os.environ.get("RANK", "0"))
        self.local_rank = int(os.environ.get("LOCAL_RANK", "0"))
        self.pg = None
        if self.world > 1:
            import torch.distributed as dist
            os.environ.setdefault("MASTER_ADDR", "127.0.0.1")
            dist.init_process_group("gloo", rank=self.rank, world_size=self.world)
            self.pg = dist

    def barrier(self):
        if self.pg:
            self.pg.barrier()

    def max(self, v: float) -> float:
        if not self.pg:
            return v
        import torch
        t = torch.tensor([v], dtype=torch.float64)
        self.pg.all_reduce(t, op=self.pg.ReduceOp.MAX)
        return float(t.item())

    def close(self):
        if self.pg:
            self.pg.destroy_process_group()


def aggregate(per_rank_units: float, elapsed_s_max: float, world: int) -> float:
    """Whole-job throughput: units every rank processed over the slowest rank's time."""
    return per_rank_units * world / elapsed_s_max


# ----------------------------------------------------------------- clocks

class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(prefix="clocks", suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.25)
        except OSError:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.15)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        for line in open(self.path):
            parts = [p.strip() for p in line.split(",")]
            if len(parts) >= 9:
                rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        smax = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(smax) if smax else None,
                "reasons": reasons, "samples": len(rows)}


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return dict(FALLBACK_PEAKS), "fallback"


def read_profile_traffic(name: str):
    """Per-launch DRAM bytes of a kernel from its committed ncu summary, if the
    summary was taken on the current kernel source (source hash matches)."""
    import hashlib
    path = os.path.join(ROOT, "profiles", name)
    if not os.path.exists(path):
        return None
    fields = {}
    for line in open(path):
        if ":" in line and line.startswith("- "):
            k, v = line[2:].split(":", 1)
            fields[k.strip()] = v.strip().strip("`")
    src = fields.get("source_files", "")
    want = fields.get("source_sha256", "")
    h = hashlib.sha256()
    for rel in src.split(","):
        rel = rel.strip()
        if not rel:
            continue
        p = os.path.join(ROOT, rel)
        if not os.path.exists(p):
            return None
        h.update(open(p, "rb").read())
    if not want or h.hexdigest() != want:
        return None
    try:
        return float(fields["dram_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


# ----------------------------------------------------------------- GPU workloads

class Timer:
    """CUDA-event timing of graph replays on one stream."""

    def __init__(self, torch, stream):
        self.torch = torch
        self.stream = stream

    def run(self, fn, dist=None):
        torch = self.torch
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            a.record(self.stream)
            fn()
            b.record(self.stream)
        torch.cuda.synchronize()
        if dist:
            dist.barrier()
        return a.elapsed_time(b) / 1e3


def replicas_for(bytes_per_rep: int, l2: int, cap: int = 64) -> int:
    return max(1, min(cap, math.ceil(4 * l2 / max(1, bytes_per_rep))))


def capture(torch, stream, body):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(stream):
        body()  # warm-up outside capture (sets kernel attributes)
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=stream):
        body()
    torch.cuda.synchronize()
    return g


# The decode layer's GEMV calls in dependency order: q, k and v read the
# same normed hidden state (one grouped call), o reads the attention output,
# gate and up read the same FFN input (one grouped call), down reads their
# activation.  Each group is one launch.
DECODE_GROUPS = (("q", "k", "v"), ("o",), ("gate", "up"), ("down",))


class DecodeLayer:
    """GEMV groups over R rotating weight replicas; a group's projections
    share one activation matrix and run as one call."""

    def __init__(self, torch, qmm, l2_bytes, stream, m=1, projections=synth.DECODE_LAYER,
                 stream_base=10, fmt="q4_0", weights=None, groups=None):
        self.torch, self.qmm, self.m, self.fmt = torch, qmm, m, fmt
        self.projs = projections
        self.cases = [synth.gemv_case(fmt, m, p.n, p.k, seed=0, stream=stream_base + i,
                                      weights=None if weights is None else weights[i])
                      for i, p in enumerate(projections)]
        names = [p.name for p in projections]
        if groups is None:
            groups = tuple((nm,) for nm in names)
        self.groups = [[names.index(nm) for nm in g] for g in groups]
        bb = 18 if fmt == "q4_0" else 34
        self.step_bytes = sum(p.n * (p.k // 32) * bb for p in projections)
        self.launches_per_step = len(self.groups)
        self.R = replicas_for(self.step_bytes, l2_bytes)
        dev = torch.device("cuda")
        base = [torch.from_numpy(c.w.reshape(-1)).to(dev) for c in self.cases]
        self.W = [[b.clone() for b in base] for _ in range(self.R)]
        del base
        # one activation matrix per group (the first member's synthetic x) and
        # one output per projection, each a view of one flat buffer, so that a
        # step's inputs and outputs move host<->device in one copy each; every
        # view starts on a multiple of 256 floats (16-byte aligned)
        xs = [self.cases[g[0]].x for g in self.groups]
        self.X_flat = torch.from_numpy(np.concatenate([a.reshape(-1) for a in xs])).to(dev)
        self.X, off = [], 0
        for a in xs:
            self.X.append(self.X_flat[off:off + a.size].view(a.shape))
            off += a.size
        self.Y_flat = torch.empty(sum(m * p.n for p in projections), dtype=torch.float32, device=dev)
        self.Y, off = [], 0
        for p in projections:
            self.Y.append(self.Y_flat[off:off + m * p.n].view(m, p.n))
            off += m * p.n
        self.stream = stream
        self.fn = qmm.qmm_gemv_q4_0 if fmt == "q4_0" else qmm.qmm_gemv_q8_0
        self.fn_multi = qmm.qmm_gemv_q4_0_multi if fmt == "q4_0" else qmm.qmm_gemv_q8_0_multi
        self.full = capture(torch, stream, lambda: [self.step(r) for r in range(self.R)])
        self.single = [None] * self.R

    def step(self, r):
        s = self.stream.cuda_stream
        for gi, g in enumerate(self.groups):
            k = self.projs[g[0]].k
            if len(g) == 1:
                i = g[0]
                self.fn(self.W[r][i], self.X[gi], self.Y[i], self.m, self.projs[i].n, k, s)
            else:
                self.fn_multi([(self.W[r][i], self.Y[i], self.projs[i].n) for i in g],
                              self.X[gi], self.m, k, s)

    def run_steps(self, k):
        """Exactly k steps, rotating replicas from replica 0."""
        for _ in range(k // self.R):
            self.full.replay()
        for r in range(k % self.R):
            if self.single[r] is None:
                self.single[r] = capture(self.torch, self.stream, lambda r=r: self.step(r))
            self.single[r].replay()


def measure_e2e(torch, qmm, layer: DecodeLayer, steps: int, dist):
    """Same step through the public API with host buffers: pinned host x ->
    device, the step's calls, device y -> pinned host, every step.  The
    step's activations (and outputs) sit in one flat buffer, so each
    direction is one copy."""
    x_host = layer.X_flat.cpu().pin_memory()
    y_host = torch.empty(layer.Y_flat.shape, dtype=torch.float32).pin_memory()
    h2d = x_host.numel() * 4
    d2h = y_host.numel() * 4
    s = layer.stream

    def one(r):
        with torch.cuda.stream(s):
            layer.X_flat.copy_(x_host, non_blocking=True)
            layer.step(r)
            y_host.copy_(layer.Y_flat, non_blocking=True)

    for r in range(min(8, steps)):
        one(r % layer.R)
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        one(i % layer.R)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    if dist:
        dist.barrier()
    return el, h2d, d2h


def run_secondary(torch, qmm, l2, stream, timer, peaks):
    """Other workloads, each as GB/s or TFLOP/s per GPU (rank 0)."""
    out = {}
    hbm = peaks["hbm_gbs"]

    weight_cache = {}

    def gemv_entry(name, fmt, m, projs, base, grouped=False):
        key = (fmt, base, tuple((p.n, p.k) for p in projs))
        if key not in weight_cache:
            weight_cache.clear()
            weight_cache[key] = [synth.gemv_case(fmt, 1, p.n, p.k, seed=0, stream=base + i).w
                                 for i, p in enumerate(projs)]
        layer = DecodeLayer(torch, qmm, l2, stream, m=m, projections=projs, stream_base=base,
                            fmt=fmt, weights=weight_cache[key],
                            groups=(tuple(p.name for p in projs),) if grouped else None)
        steps = max(layer.R, (2000 // layer.R) * layer.R)
        layer.run_steps(layer.R)
        el = timer.run(lambda: layer.run_steps(steps))
        gbs = layer.step_bytes * steps / el / 1e9
        resident = layer.R * layer.step_bytes
        # at M rows each weight takes M FMAs (2M flop) per 18/32 (Q4_0) or
        # 34/32 (Q8_0) bytes: the FP32-issue ceiling in weight bytes per second
        bpw = (18 if fmt == "q4_0" else 34) / 32.0
        fp32_ceiling = fp32_peak_tflops(peaks) * 1e12 * bpw / (2 * m) / 1e9
        out[name] = {"gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
                     "fp32_ceiling_gbs": round(fp32_ceiling, 1),
                     "frac_of_min_ceiling": round(gbs / min(hbm, fp32_ceiling), 4),
                     "us_per_call": round(el / steps / layer.launches_per_step * 1e6, 3),
                     "replicas": layer.R,
                     "l2": ("weights rotate through %d replicas (%.0f MB, %s)"
                            % (layer.R, resident / 1e6, "larger than L2" if resident > l2 else
                               "smaller than L2: L2-resident, not an HBM figure"))}
        del layer
        torch.cuda.empty_cache()

    gemv_entry("q4_0_gemv_256x1024_m1", "q4_0", 1, (synth.SINGLE_SMALL,), 90)
    # the decode step's projections one at a time (separate dependent calls)
    for i, p in enumerate(synth.DECODE_LAYER):
        gemv_entry(f"q4_0_decode_{p.name}_{p.n}x{p.k}_m1", "q4_0", 1, (p,), 10 + i)
    for m in synth.BATCHED_M:
        for i, p in enumerate(synth.BATCHED_SHAPES):
            gemv_entry(f"q4_0_gemv_{p.n}x{p.k}_m{m}", "q4_0", m, (p,), 30 + i)
    for m in synth.LM_HEAD_M:
        gemv_entry(f"q8_0_lm_head_262144x2048_m{m}", "q8_0", m, (synth.LM_HEAD,), 50)
    # the feed-forward input: gate and up as one grouped call (two outputs
    # written) against the fused GeGLU call (h = gelu(g) * u written)
    ffn = tuple(p for p in synth.DECODE_LAYER if p.name in ("gate", "up"))
    for m in (1, 8):
        gemv_entry(f"q4_0_decode_gate_up_grouped_m{m}", "q4_0", m, ffn, 14, grouped=True)
        try:
            out.update(measure_geglu(torch, qmm, l2, stream, timer, hbm, ffn, m))
        except Exception as e:  # noqa: BLE001 - reported, not hidden
            out[f"q4_0_decode_ffn_geglu_m{m}"] = {"error": str(e)[:200]}
    try:
        out.update(measure_gemm(torch, qmm, l2, stream, timer, peaks))
    except Exception as e:  # noqa: BLE001 - reported, not hidden
        out["q4_0_gemm"] = {"error": str(e)[:200]}
    return out


def measure_geglu(torch, qmm, l2, stream, timer, hbm, ffn, m):
    """Fused GeGLU decode call over rotating replicas of the gate/up pair."""
    gate, up = ffn
    n, k = gate.n, gate.k
    dev = torch.device("cuda")
    wg = torch.from_numpy(synth.q4_0_weights(n, k, seed=0, stream=14)).to(dev)
    wu = torch.from_numpy(synth.q4_0_weights(n, k, seed=0, stream=15)).to(dev)
    pair_bytes = 2 * wg.numel()
    R = replicas_for(pair_bytes, l2)
    WG = [wg.clone() for _ in range(R)]
    WU = [wu.clone() for _ in range(R)]
    del wg, wu
    x = torch.from_numpy(synth.activations_f32(m, k, seed=0, stream=16)).to(dev)
    h = torch.empty((m, n), dtype=torch.float32, device=dev)
    s = stream.cuda_stream

    def body():
        for r in range(R):
            qmm.qmm_gemv_q4_0_geglu(WG[r], WU[r], x, h, m, n, k, s)

    g = capture(torch, stream, body)
    reps = max(1, 2000 // R)
    g.replay()
    el = timer.run(lambda: [g.replay() for _ in range(reps)])
    calls = reps * R
    gbs = pair_bytes * calls / el / 1e9
    return {f"q4_0_decode_ffn_geglu_m{m}": {
        "gbs": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4),
        "us_per_call": round(el / calls * 1e6, 3), "replicas": R,
        "what": "h = gelu_tanh(x.Wg^T) * (x.Wu^T), gate and up %dx%d Q4_0, one launch" % (n, k),
        "l2": "weights rotate through %d replicas (%.0f MB, larger than L2)"
              % (R, R * pair_bytes / 1e6)}}


def measure_gemm(torch, qmm, l2, stream, timer, peaks):
    """Prefill GEMMs: median of 20 launches, L2 flushed before each.  Each
    product is timed fused (one kernel, no workspace) and two-phase (weights
    dequantised once into a bf16 workspace, then the shared-memory-operand
    GEMM; both kernels inside the timed region)."""
    res = {}
    dev = torch.device("cuda")
    flush = torch.empty(2 * l2 // 4, dtype=torch.float32, device=dev)
    gf = capture(torch, stream, lambda: flush.add_(1.0))
    s = stream.cuda_stream
    peak = peaks["bf16_tflops"]

    def timed(call):
        g = capture(torch, stream, call)
        times = []
        for _ in range(20):
            gf.replay()
            times.append(timer.run(g.replay))
        return statistics.median(times), statistics.quantiles(times, n=10)

    def entry(name, flops, t, q=None, **extra):
        e = {"tflops": round(flops / t / 1e12, 1), "frac_bf16_peak": round(flops / t / 1e12 / peak, 4),
             "us": round(t * 1e6, 2)}
        if q is not None:
            e.update(us_p10=round(q[0] * 1e6, 2), us_p90=round(q[-1] * 1e6, 2))
        e.update(extra)
        e.setdefault("l2", "flushed (2x L2 write) before each timed launch")
        res[name] = e

    m = synth.PREFILL_M
    for i, p in enumerate(synth.PREFILL_SHAPES):
        w, xb = synth.gemm_case(m, p.n, p.k, seed=0, stream=70 + i)
        W = torch.from_numpy(w.reshape(-1)).to(dev)
        X = torch.from_numpy(xb.astype(np.int16)).to(dev)
        Y = torch.empty((m, p.n), dtype=torch.float32, device=dev)
        WS = torch.empty(qmm.qmm_gemm_workspace_bytes(p.n, p.k), dtype=torch.uint8, device=dev)
        flops = 2.0 * m * p.n * p.k
        t, q = timed(lambda: qmm.qmm_gemm_q4_0(W, X, Y, m, p.n, p.k, s))
        entry(f"q4_0_gemm_{m}x{p.n}x{p.k}", flops, t, q, path="fused")
        t, q = timed(lambda: qmm.qmm_gemm_q4_0_ws(W, X, Y, m, p.n, p.k, WS, WS.numel(), s))
        entry(f"q4_0_gemm_two_phase_{m}x{p.n}x{p.k}", flops, t, q,
              path="dequant to bf16 workspace + shared-memory-operand GEMM")
        # practical ceiling of the same contraction: cuBLAS bf16 with the
        # weights already dense bf16 (no dequantization), same flush and timing
        Wd = torch.randn((p.n, p.k), device=dev).to(torch.bfloat16)
        Xd = torch.randn((m, p.k), device=dev).to(torch.bfloat16)
        t, _ = timed(lambda: torch.matmul(Xd, Wd.t()))
        entry(f"cublas_bf16_dense_{m}x{p.n}x{p.k}", flops, t,
              what="torch.matmul bf16 x bf16 -> bf16 of dense weights: a practical ceiling, not this library")
        del Wd, Xd, W, Y, WS
    # Q8_0 weights (the 8192 x 2048 shape)
    p = synth.PREFILL_SHAPES[0]
    W8 = torch.from_numpy(synth.q8_0_weights(p.n, p.k, seed=0, stream=75).reshape(-1)).to(dev)
    X = torch.from_numpy(synth.activations_bf16(m, p.k, seed=0, stream=76).astype(np.int16)).to(dev)
    Y = torch.empty((m, p.n), dtype=torch.float32, device=dev)
    WS = torch.empty(qmm.qmm_gemm_workspace_bytes(p.n, p.k), dtype=torch.uint8, device=dev)
    flops = 2.0 * m * p.n * p.k
    t, _ = timed(lambda: qmm.qmm_gemm_q8_0(W8, X, Y, m, p.n, p.k, s))
    entry(f"q8_0_gemm_{m}x{p.n}x{p.k}", flops, t, path="fused")
    t, _ = timed(lambda: qmm.qmm_gemm_q8_0_ws(W8, X, Y, m, p.n, p.k, WS, WS.numel(), s))
    entry(f"q8_0_gemm_two_phase_{m}x{p.n}x{p.k}", flops, t,
          path="dequant to bf16 workspace + shared-memory-operand GEMM")
    del W8, Y, WS
    # prefill GeGLU: the 8192 x 2048 gate/up pair over the same prompt, h bf16
    gate = next(p for p in synth.DECODE_LAYER if p.name == "gate")
    n, k = gate.n, gate.k
    wg, xb = synth.gemm_case(m, n, k, seed=0, stream=80)
    wu = synth.q4_0_weights(n, k, seed=0, stream=81)
    WG, WU = torch.from_numpy(wg.reshape(-1)).to(dev), torch.from_numpy(wu.reshape(-1)).to(dev)
    X = torch.from_numpy(xb.astype(np.int16)).to(dev)
    H = torch.empty((m, n), dtype=torch.int16, device=dev)
    WS = torch.empty(qmm.qmm_gemm_workspace_bytes(n, k, geglu=True), dtype=torch.uint8, device=dev)
    flops = 2.0 * m * (2 * n) * k
    what = ("h = bf16(gelu_tanh(X.Wg^T) * (X.Wu^T)), gate and up %dx%d Q4_0; flops count both "
            "products" % (n, k))
    t, _ = timed(lambda: qmm.qmm_gemm_q4_0_geglu(WG, WU, X, H, m, n, k, s))
    entry(f"q4_0_gemm_geglu_{m}x{n}x{k}", flops, t, what=what, path="fused")
    t, _ = timed(lambda: qmm.qmm_gemm_q4_0_geglu_ws(WG, WU, X, H, m, n, k, WS, WS.numel(), s))
    entry(f"q4_0_gemm_geglu_two_phase_{m}x{n}x{k}", flops, t, what=what,
          path="dequant to bf16 workspace + shared-memory-operand GEMM")
    return res


def cpu_baseline(seconds: float):
    """The oracle, as it stands, on the host cores: full decode-layer passes
    repeated for about `seconds`."""
    import oracle
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    cases = [synth.gemv_case("q4_0", 1, p.n, p.k, seed=0, stream=10 + i)
             for i, p in enumerate(synth.DECODE_LAYER)]
    step_bytes = sum(synth.q4_0_bytes(p.n, p.k) for p in synth.DECODE_LAYER)
    passes = 0
    t0 = time.perf_counter()
    while True:
        for c in cases:
            oracle.gemv_q4_0(c.w, c.x, c.m, c.n, c.k)
        passes += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    value = step_bytes * passes / el / 1e9
    # the same oracle on one thread, a shorter sample
    oracle.set_threads(1)
    passes1 = 0
    t0 = time.perf_counter()
    while True:
        for c in cases:
            oracle.gemv_q4_0(c.w, c.x, c.m, c.n, c.k)
        passes1 += 1
        el1 = time.perf_counter() - t0
        if el1 >= seconds / 4:
            break
    oracle.set_threads(cores)
    # the prefill GEMM oracle on a slice of its workload: 16 of the 2048 tokens
    # of the 2048 x 8192 x 2048 product
    gp = synth.PREFILL_SHAPES[0]
    gw, gx = synth.gemm_case(16, gp.n, gp.k, seed=0, stream=70)
    t0 = time.perf_counter()
    reps = 0
    while True:
        oracle.gemm_q4_0(gw, gx, 16, gp.n, gp.k)
        reps += 1
        elg = time.perf_counter() - t0
        if elg >= min(3.0, seconds / 4):
            break
    gemm_gflops = 2.0 * 16 * gp.n * gp.k * reps / elg / 1e9
    return {"value": round(value, 4), "unit": "GB/s", "cores": cores,
            "kind": "oracle",
            "sample": f"{passes} full passes of the decode-layer set (M=1, 7 Q4_0 projections) "
                      f"in {el:.1f} s, binary64 C oracle, {cores} OpenMP threads",
            "single_thread": {"value": round(step_bytes * passes1 / el1 / 1e9, 4), "unit": "GB/s",
                              "sample": f"{passes1} passes in {el1:.1f} s on 1 thread"},
            "gemm": {"value": round(gemm_gflops, 3), "unit": "GFLOP/s",
                     "sample": f"{reps} passes of 16 tokens x {gp.n} x {gp.k} (Q4_0, bf16 X) in "
                               f"{elg:.1f} s, binary64 C oracle, {cores} OpenMP threads"}}


# ----------------------------------------------------------------- arms

def run_ours(args, dist):
    import torch
    from block_quantized_matmul_gguf_gb300 import qmm

    torch.cuda.set_device(dist.local_rank)
    qmm.load()
    props = torch.cuda.get_device_properties(dist.local_rank)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    timer = Timer(torch, stream)

    layer = DecodeLayer(torch, qmm, l2, stream, groups=DECODE_GROUPS)
    warm = max(3, args.warmup)
    layer.run_steps(warm)
    torch.cuda.synchronize()

    clocks = ClockSampler(dist.local_rank)
    clocks.start()
    el = timer.run(lambda: layer.run_steps(args.steps), dist)
    clk = clocks.stop()
    el_max = dist.max(el)
    err = qmm.qmm_get_device_error(stream)
    if err != 0:
        raise RuntimeError(f"device error word after the timed region: {err}")

    value = aggregate(layer.step_bytes * args.steps, el_max, dist.world) / 1e9
    per_launch_s = el_max / (args.steps * layer.launches_per_step)
    bytes_per_launch = layer.step_bytes / layer.launches_per_step
    achieved = bytes_per_launch / per_launch_s / 1e9
    traffic = read_profile_traffic("gemv_q4_0_decode_layer_m1.md")

    e2e_el, h2d, d2h = measure_e2e(torch, qmm, layer, max(200, args.steps // 20), dist)
    e2e_steps = max(200, args.steps // 20)
    e2e_value = aggregate(layer.step_bytes * e2e_steps, dist.max(e2e_el), dist.world) / 1e9

    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": dist.world,
        "steps": args.steps,
        "warmup": warm,
        "ms_per_step": round(el_max / args.steps * 1e3, 6),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32",
        "data": "synthetic (SplitMix64 seed 0: d ~ U[0.001,0.02] binary16, uniform nibbles, "
                "x ~ N(0,1) fp32)",
        "config": {
            "workload": "Q4_0 decode-layer GEMV set, M=1: q 2048->2048, k 2048->512, "
                        "v 2048->512, o 2048->2048, gate 2048->8192, up 2048->8192, "
                        "down 8192->2048 (34,209,792 weight bytes per step), as 4 dependent "
                        "calls: q+k+v grouped (shared x), o, gate+up grouped, down",
            "weight_bytes_per_step": layer.step_bytes,
            "launches_per_step": layer.launches_per_step,
            "replicas": layer.R,
            "l2": f"inputs larger than L2: {layer.R} rotating weight replicas "
                  f"({layer.R * layer.step_bytes / 1e6:.0f} MB) vs {l2 / 1e6:.0f} MB L2",
            "timing": "CUDA graphs of the steps, CUDA events on the launching stream",
            "parallelism": f"replicas x{dist.world}",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic,
            "kernel": "gemv_stream_kernel<Q4_0, M=1>",
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
            if peak_src == "measured" else "fallback 6.8 TB/s",
            "bytes_per_launch": bytes_per_launch,
        },
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "path": "pinned host x (the step's activations, one buffer) -> device in one "
                        "copy, the step's 4 C-ABI calls via ctypes, the 7 outputs -> pinned host "
                        "in one copy, per step; host wall clock"},
        "gpu_launches": args.steps * layer.launches_per_step,
    }
    del layer
    torch.cuda.empty_cache()
    if not args.no_secondary and dist.rank == 0:
        result["secondary"] = run_secondary(torch, qmm, l2, stream, timer, peaks)
    if dist.rank == 0 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(args.cpu_seconds)
    return result


def run_reference(args, dist):
    """The oracle on the host cores, same workload and metric, each step a
    bounded sample of the decode-layer set's rows."""
    if dist.rank != 0:
        return None
    import oracle
    cores = os.cpu_count() or 1
    oracle.set_threads(cores)
    cases = [synth.gemv_case("q4_0", 1, p.n, p.k, seed=0, stream=10 + i)
             for i, p in enumerate(synth.DECODE_LAYER)]
    t0 = time.perf_counter()
    for c in cases:
        oracle.gemv_q4_0(c.w, c.x, c.m, c.n, c.k)
    t_full = time.perf_counter() - t0
    budget = 90.0
    frac = min(1.0, budget / max(1e-9, (args.steps + args.warmup) * t_full))
    rows = [max(1, int(round(frac * c.n))) for c in cases]
    sub = [(c.w[:r], c.x, r, c.k) for c, r in zip(cases, rows)]
    sample_bytes = sum(r * (k // 32) * 18 for (_, _, r, k) in sub)

    def step():
        for w, x, r, k in sub:
            oracle.gemv_q4_0(w, x, 1, r, k)

    for _ in range(max(3, args.warmup)):
        step()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        step()
    el = time.perf_counter() - t0
    value = sample_bytes * args.steps / el / 1e9
    sample = (f"first {frac * 100:.3g}% of the rows of each of the 7 projections "
              f"({sample_bytes} weight bytes) per step, binary64 C oracle, {cores} threads")
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s",
        "n_gpus": dist.world, "steps": args.steps, "warmup": max(3, args.warmup),
        "ms_per_step": round(el / args.steps * 1e3, 4), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": "Q4_0 decode-layer GEMV set, M=1 (same as ours)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main(argv=None):
    args = parse_args(argv)
    if args.profile:
        run_profile(args)
        return
    dist = Dist()
    try:
        res = run_reference(args, dist) if args.impl == "reference" else run_ours(args, dist)
        if res is not None and dist.rank == 0:
            print(json.dumps(res), flush=True)
    finally:
        dist.close()


if __name__ == "__main__":
    main()
