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
copies the outputs back (weights stay resident: they are the model).  The
copies are the library's qmm_copy launches; the same with cudaMemcpyAsync
copies is reported beside it.

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
# available): SMs (queried from the device) x 128 FMA lanes x 2 flop per cycle
# at the maximum SM clock.
FP32_LANES_PER_SM = 128


def fp32_peak_tflops(peaks, sms: int) -> float:
    return sms * FP32_LANES_PER_SM * 2 * float(peaks.get("sm_max_mhz", 2070.0)) * 1e6 / 1e12


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=32000)
    ap.add_argument("--warmup", type=int, default=320)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-secondary", action="store_true",
                    help="skip the secondary workloads (headline only)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--only", default=None, metavar="REGEX",
                    help="secondary workloads: run only those whose name matches REGEX")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle baseline sample")
    ap.add_argument("--profile", default=None, metavar="CASE",
                    help="no timing: run CASE a few times for a profiler and exit. CASE is "
                         "decode_grouped (the timed decode step), decode (seven separate calls), "
                         "gate_up:M (the step's gate+up launch), "
                         "gemv:FMT:M:N:K, gemv_tc:M:N:K, geglu:M:N:K, gemm_geglu:M:N:K, dequant:FMT:N:K "
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
    elif parts[0] == "gate_up":
        # the decode step's gate+up launch: two 8192 x 2048 Q4_0 matrices sharing x
        m = int(parts[1]) if len(parts) > 1 else 1
        projs = [p for p in synth.DECODE_LAYER if p.name in ("gate", "up")]
        W = [torch.from_numpy(synth.q4_0_weights(p.n, p.k, seed=0, stream=14 + i)).to(dev)
             for i, p in enumerate(projs)]
        Y = [torch.empty((m, p.n), dtype=torch.float32, device=dev) for p in projs]
        x = torch.from_numpy(synth.activations_f32(m, projs[0].k, seed=0, stream=16)).to(dev)
        for _ in range(reps):
            qmm.qmm_gemv_q4_0_multi([(w, y, p.n) for w, y, p in zip(W, Y, projs)], x, m, projs[0].k)
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
    elif parts[0] == "gemv_tc":
        m, n, k = int(parts[1]), int(parts[2]), int(parts[3])
        c = synth.gemv_case("q4_0", m, n, k, seed=0, stream=1)
        w, x = torch.from_numpy(c.w).to(dev), torch.from_numpy(c.x).to(dev)
        for _ in range(reps):
            qmm.gemv_tc_q4_0(w, x, n, k)
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

    # cycles of a spin kernel queued ahead of the start event (about 2 ms):
    # while the GPU spins, the host enqueues the timed launches, so that no
    # host launch latency falls between the two events
    PREQUEUE_CYCLES = 4_000_000

    def run(self, fn, dist=None, prequeue=True):
        torch = self.torch
        if dist:
            dist.barrier()
        torch.cuda.synchronize()
        a = torch.cuda.Event(enable_timing=True)
        b = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(self.stream):
            if prequeue:
                torch.cuda._sleep(self.PREQUEUE_CYCLES)
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
                 stream_base=10, fmt="q4_0", weights=None, groups=None, tensor_cores=False):
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
        if tensor_cores:  # the tensor-core GEMV (single projections only)
            self.fn = qmm.qmm_gemv_q4_0_tc
        self.fn_multi = qmm.qmm_gemv_q4_0_multi if fmt == "q4_0" else qmm.qmm_gemv_q8_0_multi
        # one graph for a whole rotation and one per single step, all captured
        # (and replayed once, which uploads them) before anything is timed
        self.full = capture(torch, stream, lambda: [self.step(r) for r in range(self.R)])
        self.single = [capture(torch, stream, lambda r=r: self.step(r)) for r in range(self.R)]
        self.pos = 0  # replica of the next step: the rotation continues across calls
        self.timed_graphs = {}

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

    def warm_graphs(self):
        """Replay every graph once (outside any timed region): the first replay
        of a CUDA graph uploads it.  Ends at the rotation's start."""
        self.full.replay()
        for g in self.single:
            g.replay()
        self.pos = 0

    def run_steps(self, k):
        """Exactly k untimed steps.  They continue the replica rotation where
        the previous call left it."""
        done = 0
        while done < k and self.pos != 0:
            self.single[self.pos].replay()
            self.pos = (self.pos + 1) % self.R
            done += 1
        while k - done >= self.R:
            self.full.replay()
            done += self.R
        while done < k:
            self.single[self.pos].replay()
            self.pos = (self.pos + 1) % self.R
            done += 1

    # timed runs: graphs of many consecutive steps from replica 0, so that
    # the steps follow one another with programmatic dependent launch (a
    # graph boundary, as between single-step graphs, ends that overlap)
    BIG_ROTATIONS = 8

    def _timed_plan(self, k):
        big = self.BIG_ROTATIONS * self.R
        n_big, rem = divmod(k, big)
        return n_big, rem

    def prepare_timed(self, k):
        """Capture and upload the graphs that time_steps(k) replays, then leave
        the rotation at replica 0 with every replica last read in replica
        order (replica 0 R steps before the next step).  Untimed steps."""
        n_big, rem = self._timed_plan(k)
        big = self.BIG_ROTATIONS * self.R
        if n_big and big not in self.timed_graphs:
            self.timed_graphs[big] = capture(
                self.torch, self.stream, lambda: [self.step(i % self.R) for i in range(big)])
        if rem and rem not in self.timed_graphs:
            self.timed_graphs[rem] = capture(
                self.torch, self.stream, lambda: [self.step(i % self.R) for i in range(rem)])
        for key in ({big} if n_big else set()) | ({rem} if rem else set()):
            self.timed_graphs[key].replay()
        self.pos = (rem % self.R) if rem else 0
        self.run_steps((self.R - self.pos) % self.R)  # back to replica 0
        self.full.replay()

    def time_steps(self, k):
        """Exactly k steps from replica 0 (call prepare_timed(k) first)."""
        n_big, rem = self._timed_plan(k)
        big = self.BIG_ROTATIONS * self.R
        for _ in range(n_big):
            self.timed_graphs[big].replay()
        if rem:
            self.timed_graphs[rem].replay()
        self.pos = k % self.R


def measure_e2e(torch, qmm, layer: DecodeLayer, steps: int, dist, graphs: bool,
                copy_engine: bool = False, rotation_graph: bool = False):
    """The step through the public C ABI with host buffers: pinned host x ->
    device, the step's four calls, device y -> pinned host, every step; the
    weights stay resident (they are the model).  The step's activations (and
    outputs) sit in one flat buffer, so each direction is one copy.

    graphs=False: every step makes its copies and the four ctypes calls from
    Python.  graphs=True: each step replays a CUDA graph captured from those
    same copies and calls (one graph per weight replica), as a decode loop
    that captures its layer once would run it.  Host wall clock over all
    steps, synchronised at both ends.

    The copies are the library's qmm_copy launches (the SMs read and write
    the pinned host buffers); copy_engine=True makes them cudaMemcpyAsync
    transfers instead (torch's non-blocking copy_), for comparison.

    rotation_graph=True (with graphs): one graph holds a whole rotation of R
    consecutive steps, each still with its own copies in and out, as a decode
    loop that captures all of a token's layers together would run them;
    steps is rounded up to whole rotations."""
    x_host = layer.X_flat.cpu().pin_memory()
    y_host = torch.empty(layer.Y_flat.shape, dtype=torch.float32).pin_memory()
    h2d = x_host.numel() * 4
    d2h = y_host.numel() * 4
    s = layer.stream

    def one(r):
        with torch.cuda.stream(s):
            if copy_engine:
                layer.X_flat.copy_(x_host, non_blocking=True)
            else:
                qmm.qmm_copy(layer.X_flat, x_host, h2d, s)
            layer.step(r)
            if copy_engine:
                y_host.copy_(layer.Y_flat, non_blocking=True)
            else:
                qmm.qmm_copy(y_host, layer.Y_flat, d2h, s)

    if graphs and rotation_graph:
        steps = -(-steps // layer.R) * layer.R
        g_rot = capture(torch, s, lambda: [one(r) for r in range(layer.R)])
        g_rot.replay()

        def run(i):
            if i % layer.R == 0:
                g_rot.replay()
    elif graphs:
        gs = [capture(torch, s, lambda r=r: one(r)) for r in range(layer.R)]
        for g in gs:
            g.replay()

        def run(i):
            gs[i % layer.R].replay()
    else:
        for r in range(min(8, steps)):
            one(r % layer.R)
        run = lambda i: one(i % layer.R)  # noqa: E731
    torch.cuda.synchronize()
    if dist:
        dist.barrier()
    t0 = time.perf_counter()
    for i in range(steps):
        run(i)
    torch.cuda.synchronize()
    el = time.perf_counter() - t0
    if dist:
        dist.barrier()
    return el, h2d, d2h, steps


def run_secondary(torch, qmm, l2, stream, timer, peaks, sms, only=None):
    """Other workloads, each as GB/s or TFLOP/s per GPU (rank 0).  only: a
    regular expression; workloads whose names do not match are skipped."""
    import re
    out = {}
    hbm = peaks["hbm_gbs"]
    wanted = (lambda name: re.search(only, name) is not None) if only else (lambda name: True)

    weight_cache = {}

    def gemv_entry(name, fmt, m, projs, base, grouped=False, tensor_cores=False):
        if not wanted(name):
            return
        key = (fmt, base, tuple((p.n, p.k) for p in projs))
        if key not in weight_cache:
            weight_cache.clear()
            weight_cache[key] = [synth.gemv_case(fmt, 1, p.n, p.k, seed=0, stream=base + i).w
                                 for i, p in enumerate(projs)]
        layer = DecodeLayer(torch, qmm, l2, stream, m=m, projections=projs, stream_base=base,
                            fmt=fmt, weights=weight_cache[key],
                            groups=(tuple(p.name for p in projs),) if grouped else None,
                            tensor_cores=tensor_cores)
        steps = max(layer.R, (2000 // layer.R) * layer.R)
        layer.warm_graphs()
        layer.prepare_timed(steps)
        el = timer.run(lambda: layer.time_steps(steps))
        gbs = layer.step_bytes * steps / el / 1e9
        resident = layer.R * layer.step_bytes
        # at M rows each weight takes M FMAs (2M flop) per 18/32 (Q4_0) or
        # 34/32 (Q8_0) bytes: the FP32-issue ceiling in weight bytes per second
        bpw = (18 if fmt == "q4_0" else 34) / 32.0
        fp32_ceiling = fp32_peak_tflops(peaks, sms) * 1e12 * bpw / (2 * m) / 1e9
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
    # the same batched products on the tensor cores (qmm_gemv_q4_0_tc)
    for m in (1,) + tuple(synth.BATCHED_M):
        for i, p in enumerate(synth.BATCHED_SHAPES):
            gemv_entry(f"q4_0_gemv_tc_{p.n}x{p.k}_m{m}", "q4_0", m, (p,), 30 + i, tensor_cores=True)
    for m in synth.LM_HEAD_M:
        gemv_entry(f"q8_0_lm_head_262144x2048_m{m}", "q8_0", m, (synth.LM_HEAD,), 50)
    # the same 262144 x 2048 matrix in Q4_0 (302 MB), one token
    gemv_entry("q4_0_gemv_262144x2048_m1", "q4_0", 1, (synth.LM_HEAD,), 52)
    # the feed-forward input: gate and up as one grouped call (two outputs
    # written) against the fused GeGLU call (h = gelu(g) * u written)
    ffn = tuple(p for p in synth.DECODE_LAYER if p.name in ("gate", "up"))
    for m in (1, 8):
        gemv_entry(f"q4_0_decode_gate_up_grouped_m{m}", "q4_0", m, ffn, 14, grouped=True)
        if not wanted(f"q4_0_decode_ffn_geglu_m{m}"):
            continue
        try:
            out.update(measure_geglu(torch, qmm, l2, stream, timer, hbm, ffn, m))
        except Exception as e:  # noqa: BLE001 - reported, not hidden
            out[f"q4_0_decode_ffn_geglu_m{m}"] = {"error": str(e)[:200]}
    if wanted("q4_0_gemm_2048x8192x2048"):
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
    """Prefill GEMMs.  Each product runs over R rotating replicas of its
    inputs and output (footprint >= 2x L2, so every launch finds its operands
    in HBM), captured as one graph of R back-to-back launches; a sample times
    several replays of that graph (K = R x replays launches) with CUDA events,
    and the figure is the median over samples of time per launch.  Each
    product is timed fused (one kernel, no workspace) and two-phase (weights
    dequantised once into a bf16 workspace, then the shared-memory-operand
    GEMM; both kernels in the timed region)."""
    res = {}
    dev = torch.device("cuda")
    s = stream.cuda_stream
    peak = peaks["bf16_tflops"]

    def timed(calls, samples=7, min_launches=64):
        """calls: one callable per replica.  Returns (median s/launch, p10, p90, K)."""
        g = capture(torch, stream, lambda: [c() for c in calls])
        g.replay()
        g.replay()
        reps = max(1, -(-min_launches // len(calls)))
        times = []
        for _ in range(samples):
            t = timer.run(lambda: [g.replay() for _ in range(reps)])
            times.append(t / (reps * len(calls)))
        times.sort()
        return statistics.median(times), times[0], times[-1], reps * len(calls)

    def entry(name, flops, tq, **extra):
        t, lo, hi, launches = tq
        e = {"tflops": round(flops / t / 1e12, 1), "frac_bf16_peak": round(flops / t / 1e12 / peak, 4),
             "us": round(t * 1e6, 2), "us_min": round(lo * 1e6, 2), "us_max": round(hi * 1e6, 2),
             "launches_per_sample": launches}
        e.update(extra)
        e.setdefault("l2", "operands rotate through replicas larger than 2x L2 (inputs cold in HBM)")
        res[name] = e

    def replicas(nbytes):
        return max(2, min(16, math.ceil(2 * l2 / max(1, nbytes))))

    m = synth.PREFILL_M
    for i, p in enumerate(synth.PREFILL_SHAPES):
        w, xb = synth.gemm_case(m, p.n, p.k, seed=0, stream=70 + i)
        W0 = torch.from_numpy(w.reshape(-1)).to(dev)
        X0 = torch.from_numpy(xb.astype(np.int16)).to(dev)
        R = replicas(W0.numel() + 2 * X0.numel() + 4 * m * p.n)
        W = [W0.clone() for _ in range(R)]
        X = [X0.clone() for _ in range(R)]
        Y = [torch.empty((m, p.n), dtype=torch.float32, device=dev) for _ in range(R)]
        WS = torch.empty(qmm.qmm_gemm_workspace_bytes(p.n, p.k), dtype=torch.uint8, device=dev)
        del W0, X0
        flops = 2.0 * m * p.n * p.k
        entry(f"q4_0_gemm_{m}x{p.n}x{p.k}", flops,
              timed([lambda r=r: qmm.qmm_gemm_q4_0(W[r], X[r], Y[r], m, p.n, p.k, s) for r in range(R)]),
              path="fused", replicas=R)
        entry(f"q4_0_gemm_two_phase_{m}x{p.n}x{p.k}", flops,
              timed([lambda r=r: qmm.qmm_gemm_q4_0_ws(W[r], X[r], Y[r], m, p.n, p.k, WS, WS.numel(), s)
                     for r in range(R)]),
              path="dequant to bf16 workspace + shared-memory-operand GEMM", replicas=R)
        entry(f"q4_0_gemm_prefill_static_scratch_{m}x{p.n}x{p.k}", flops,
              timed([lambda r=r: qmm.qmm_gemm_q4_0_prefill(W[r], X[r], Y[r], m, p.n, p.k, s)
                     for r in range(R)]),
              path="two-phase on the library's own scratch (no workspace argument)", replicas=R)
        del W, X, Y, WS
        # a short prompt (256 tokens) with the same weights: fused alone, and
        # with a workspace, where the fused kernel splits K through it
        ms = synth.SHORT_PROMPT_M
        w, xb = synth.gemm_case(ms, p.n, p.k, seed=0, stream=74 + i)
        W0 = torch.from_numpy(w.reshape(-1)).to(dev)
        X0 = torch.from_numpy(xb.astype(np.int16)).to(dev)
        R = replicas(W0.numel() + 2 * X0.numel() + 4 * ms * p.n)
        W = [W0.clone() for _ in range(R)]
        X = [X0.clone() for _ in range(R)]
        Y = [torch.empty((ms, p.n), dtype=torch.float32, device=dev) for _ in range(R)]
        WS = [torch.empty(qmm.qmm_gemm_workspace_bytes(p.n, p.k), dtype=torch.uint8, device=dev)
              for _ in range(2)]
        del W0, X0
        flops_s = 2.0 * ms * p.n * p.k
        entry(f"q4_0_gemm_{ms}x{p.n}x{p.k}", flops_s,
              timed([lambda r=r: qmm.qmm_gemm_q4_0(W[r], X[r], Y[r], ms, p.n, p.k, s) for r in range(R)]),
              path="fused, one pass over K per tile", replicas=R)
        entry(f"q4_0_gemm_ws_{ms}x{p.n}x{p.k}", flops_s,
              timed([lambda r=r: qmm.qmm_gemm_q4_0_ws(W[r], X[r], Y[r], ms, p.n, p.k, WS[r % 2],
                                                      WS[r % 2].numel(), s) for r in range(R)]),
              path="fused with K split into parts through the workspace, then the parts added",
              replicas=R)
        del W, X, Y, WS
        # practical ceiling of the same contraction: cuBLAS bf16 with the
        # weights already dense bf16 (no dequantization), same rotation
        Wd = [torch.randn((p.n, p.k), device=dev).to(torch.bfloat16) for _ in range(2)]
        Xd = [torch.randn((m, p.k), device=dev).to(torch.bfloat16) for _ in range(2)]
        Rd = replicas(2 * (p.n * p.k + m * p.k + m * p.n))
        entry(f"cublas_bf16_dense_{m}x{p.n}x{p.k}", flops,
              timed([lambda r=r: torch.matmul(Xd[r % 2], Wd[r % 2].t()) for r in range(Rd)]),
              what="torch.matmul bf16 x bf16 -> bf16 of dense weights: a practical ceiling, "
                   "not this library (two operand sets; outputs allocated per call)")
        del Wd, Xd
        torch.cuda.empty_cache()
    # Q8_0 weights (the 8192 x 2048 shape)
    p = synth.PREFILL_SHAPES[0]
    W0 = torch.from_numpy(synth.q8_0_weights(p.n, p.k, seed=0, stream=75).reshape(-1)).to(dev)
    X0 = torch.from_numpy(synth.activations_bf16(m, p.k, seed=0, stream=76).astype(np.int16)).to(dev)
    R = replicas(W0.numel() + 2 * X0.numel() + 4 * m * p.n)
    W = [W0.clone() for _ in range(R)]
    X = [X0.clone() for _ in range(R)]
    Y = [torch.empty((m, p.n), dtype=torch.float32, device=dev) for _ in range(R)]
    WS = torch.empty(qmm.qmm_gemm_workspace_bytes(p.n, p.k), dtype=torch.uint8, device=dev)
    del W0, X0
    flops = 2.0 * m * p.n * p.k
    entry(f"q8_0_gemm_{m}x{p.n}x{p.k}", flops,
          timed([lambda r=r: qmm.qmm_gemm_q8_0(W[r], X[r], Y[r], m, p.n, p.k, s) for r in range(R)]),
          path="fused", replicas=R)
    entry(f"q8_0_gemm_two_phase_{m}x{p.n}x{p.k}", flops,
          timed([lambda r=r: qmm.qmm_gemm_q8_0_ws(W[r], X[r], Y[r], m, p.n, p.k, WS, WS.numel(), s)
                 for r in range(R)]),
          path="dequant to bf16 workspace + shared-memory-operand GEMM", replicas=R)
    del W, X, Y, WS
    torch.cuda.empty_cache()
    # prefill GeGLU: the 8192 x 2048 gate/up pair over the same prompt, h bf16
    gate = next(p for p in synth.DECODE_LAYER if p.name == "gate")
    n, k = gate.n, gate.k
    wg, xb = synth.gemm_case(m, n, k, seed=0, stream=80)
    wu = synth.q4_0_weights(n, k, seed=0, stream=81)
    WG0, WU0 = torch.from_numpy(wg.reshape(-1)).to(dev), torch.from_numpy(wu.reshape(-1)).to(dev)
    X0 = torch.from_numpy(xb.astype(np.int16)).to(dev)
    R = replicas(2 * WG0.numel() + 2 * X0.numel() + 2 * m * n)
    WG = [WG0.clone() for _ in range(R)]
    WU = [WU0.clone() for _ in range(R)]
    X = [X0.clone() for _ in range(R)]
    H = [torch.empty((m, n), dtype=torch.int16, device=dev) for _ in range(R)]
    WS = torch.empty(qmm.qmm_gemm_workspace_bytes(n, k, geglu=True), dtype=torch.uint8, device=dev)
    del WG0, WU0, X0
    flops = 2.0 * m * (2 * n) * k
    what = ("h = bf16(gelu_tanh(X.Wg^T) * (X.Wu^T)), gate and up %dx%d Q4_0; flops count both "
            "products" % (n, k))
    entry(f"q4_0_gemm_geglu_{m}x{n}x{k}", flops,
          timed([lambda r=r: qmm.qmm_gemm_q4_0_geglu(WG[r], WU[r], X[r], H[r], m, n, k, s)
                 for r in range(R)]), what=what, path="fused", replicas=R)
    entry(f"q4_0_gemm_geglu_two_phase_{m}x{n}x{k}", flops,
          timed([lambda r=r: qmm.qmm_gemm_q4_0_geglu_ws(WG[r], WU[r], X[r], H[r], m, n, k, WS,
                                                         WS.numel(), s) for r in range(R)]),
          what=what, path="dequant to bf16 workspace + shared-memory-operand GEMM", replicas=R)
    del WG, WU, X, H, WS
    torch.cuda.empty_cache()
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

def time_dominant_kernel(torch, qmm, l2, stream, timer):
    """The decode step's dominant launch, the grouped gate+up call (two
    8192 x 2048 Q4_0 matrices sharing x, one gemv_stream_kernel launch), on
    its own: R rotating replicas (> 4x L2), back-to-back launches timed with
    CUDA events on the launching stream.  Returns (s per launch, bytes per
    launch, launches timed)."""
    ffn = tuple(p for p in synth.DECODE_LAYER if p.name in ("gate", "up"))
    layer = DecodeLayer(torch, qmm, l2, stream, m=1, projections=ffn, stream_base=14,
                        groups=(("gate", "up"),))
    layer.warm_graphs()
    steps = max(layer.R, (2000 // layer.R) * layer.R)
    layer.prepare_timed(steps)
    el = timer.run(lambda: layer.time_steps(steps))
    nbytes = layer.step_bytes
    del layer
    torch.cuda.empty_cache()
    return el / steps, nbytes, steps


def kernel_summary(secondary):
    """Compact figures of the other single-GPU workloads (a copy of what
    `secondary` holds, kept short so that it survives truncated logs)."""
    out = {}
    pick = {
        "gemv_q8_0_lm_head_262144x2048_m1": ("q8_0_lm_head_262144x2048_m1", "gbs", "frac_hbm"),
        "gemv_q8_0_lm_head_262144x2048_m8": ("q8_0_lm_head_262144x2048_m8", "gbs", "frac_of_min_ceiling"),
        "gemv_q4_0_262144x2048_m1": ("q4_0_gemv_262144x2048_m1", "gbs", "frac_hbm"),
        "gemv_q4_0_8192x2048_m16": ("q4_0_gemv_8192x2048_m16", "gbs", "frac_of_min_ceiling"),
        "gemm_q4_0_2048x8192x2048": ("q4_0_gemm_2048x8192x2048", "tflops", "frac_bf16_peak"),
        "gemm_q4_0_2048x2048x8192": ("q4_0_gemm_2048x2048x8192", "tflops", "frac_bf16_peak"),
        "gemm_q4_0_two_phase_2048x8192x2048": ("q4_0_gemm_two_phase_2048x8192x2048", "tflops",
                                               "frac_bf16_peak"),
        "gemm_q4_0_two_phase_2048x2048x8192": ("q4_0_gemm_two_phase_2048x2048x8192", "tflops",
                                               "frac_bf16_peak"),
    }
    for key, (src, val, frac) in pick.items():
        e = secondary.get(src)
        if isinstance(e, dict) and val in e:
            out[key] = {val: e[val], frac: e.get(frac)}
    for key, e in secondary.items():
        if key.startswith("q4_0_gemv_tc_") and isinstance(e, dict) and "gbs" in e:
            out["gemv_tc_" + key[len("q4_0_gemv_tc_"):]] = {"gbs": e["gbs"],
                                                           "frac_of_min_ceiling": e.get("frac_of_min_ceiling")}
    return out


def run_ours(args, dist):
    import torch
    from block_quantized_matmul_gguf_gb300 import qmm

    torch.cuda.set_device(dist.local_rank)
    qmm.load()
    props = torch.cuda.get_device_properties(dist.local_rank)
    l2 = int(getattr(props, "L2_cache_size", 126 * 1024 * 1024))
    sms = int(props.multi_processor_count)
    peaks, peak_src = load_peaks()
    stream = torch.cuda.Stream()
    timer = Timer(torch, stream)

    layer = DecodeLayer(torch, qmm, l2, stream, groups=DECODE_GROUPS)
    warm = max(3, args.warmup)
    layer.warm_graphs()
    layer.run_steps(warm)              # the W warm-up steps
    layer.prepare_timed(args.steps)    # the timed graphs, captured and uploaded
    torch.cuda.synchronize()

    clocks = ClockSampler(dist.local_rank)
    clocks.start()
    el = timer.run(lambda: layer.time_steps(args.steps), dist)
    clk = clocks.stop()
    el_max = dist.max(el)
    err = qmm.qmm_get_device_error(stream)
    if err != 0:
        raise RuntimeError(f"device error word after the timed region: {err}")

    value = aggregate(layer.step_bytes * args.steps, el_max, dist.world) / 1e9
    step_achieved = layer.step_bytes / (el_max / args.steps) / 1e9

    e2e_steps = max(200, args.steps // 20)
    e2e_el, h2d, d2h, _ = measure_e2e(torch, qmm, layer, e2e_steps, dist, graphs=True)
    e2e_value = aggregate(layer.step_bytes * e2e_steps, dist.max(e2e_el), dist.world) / 1e9
    e2e_el_d, _, _, _ = measure_e2e(torch, qmm, layer, e2e_steps, dist, graphs=False)
    e2e_direct = aggregate(layer.step_bytes * e2e_steps, dist.max(e2e_el_d), dist.world) / 1e9
    e2e_el_ce, _, _, _ = measure_e2e(torch, qmm, layer, e2e_steps, dist, graphs=True, copy_engine=True)
    e2e_ce = aggregate(layer.step_bytes * e2e_steps, dist.max(e2e_el_ce), dist.world) / 1e9
    e2e_el_rot, _, _, rot_steps = measure_e2e(torch, qmm, layer, e2e_steps, dist, graphs=True,
                                              rotation_graph=True)
    e2e_rot = aggregate(layer.step_bytes * rot_steps, dist.max(e2e_el_rot), dist.world) / 1e9
    step_bytes, launches_per_step, R = layer.step_bytes, layer.launches_per_step, layer.R
    del layer
    torch.cuda.empty_cache()

    t_dom, dom_bytes, dom_launches = time_dominant_kernel(torch, qmm, l2, stream, timer)
    achieved = dom_bytes / t_dom / 1e9
    traffic = read_profile_traffic("gemv_q4_0_gate_up_8192x2048_m1.md")

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
            "weight_bytes_per_step": step_bytes,
            "launches_per_step": launches_per_step,
            "replicas": R,
            "l2": f"inputs larger than L2: {R} rotating weight replicas "
                  f"({R * step_bytes / 1e6:.0f} MB) vs {l2 / 1e6:.0f} MB L2; each step's weights "
                  f"were last read {R} steps earlier",
            "timing": "the K timed steps are CUDA graphs of consecutive steps from replica 0 "
                      "(launches chained by programmatic dependent launch), each captured and "
                      "replayed once before the timed region; CUDA events on the launching "
                      "stream behind a queued 2 ms spin, so no host launch gap is timed",
            "parallelism": f"replicas x{dist.world}",
        },
        "roofline": {
            "bound": "hbm",
            "achieved": round(achieved, 1),
            "peak": peaks["hbm_gbs"],
            "unit": "GB/s",
            "frac": round(achieved / peaks["hbm_gbs"], 4),
            "traffic": traffic,
            "kernel": "gemv_stream_kernel<Q4_0, M=1, L=1, R=2>: the grouped gate+up launch "
                      "(2 x 8192x2048 Q4_0, x shared), the step's largest",
            "bytes_per_launch": dom_bytes,
            "timing": f"{dom_launches} back-to-back launches over rotating replicas, CUDA events",
            "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs, burst copy)"
            if peak_src == "measured" else "fallback 6.8 TB/s",
            "step_achieved": round(step_achieved, 1),
            "step_frac": round(step_achieved / peaks["hbm_gbs"], 4),
        },
        "clocks": clk,
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s",
                "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                "steps": e2e_steps,
                "path": "per step: pinned host x (the step's activations, one buffer) -> device "
                        "in one qmm_copy launch, the step's 4 C-ABI calls, the 7 outputs -> "
                        "pinned host in one qmm_copy launch; each step replays a CUDA graph "
                        "captured from those calls (one per weight replica); host wall clock",
                "direct_calls": {"value": round(e2e_direct, 2), "unit": "GB/s",
                                 "path": "the same copies and calls issued from Python every "
                                         "step (no graph): host-bound"},
                "copy_engine": {"value": round(e2e_ce, 2), "unit": "GB/s",
                                "path": "as `path`, with the two copies made by cudaMemcpyAsync "
                                        "(torch non-blocking copy_) instead of qmm_copy"},
                "rotation_graph": {"value": round(e2e_rot, 2), "unit": "GB/s", "steps": rot_steps,
                                   "path": f"as `path`, with one CUDA graph holding {R} consecutive "
                                           "steps (one weight rotation), each step still copying "
                                           "its activations in and its outputs out"}},
        "gpu_launches": args.steps * launches_per_step,
    }
    if not args.no_secondary and dist.rank == 0:
        secondary = run_secondary(torch, qmm, l2, stream, timer, peaks, sms, args.only)
        result["kernels"] = kernel_summary(secondary)
        result["secondary"] = secondary
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
