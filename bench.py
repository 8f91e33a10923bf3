"""Benchmark: achieved HBM GB/s of the fused QK-Norm + RoPE + FP8 prologue on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--no-extras]

A step is one launch of the whole hot path (load -> sum of squares -> normalise -> NeoX RoPE ->
amax/scale -> e4m3 codes -> store) over one batch of the prologue workload: 4096 tokens x (32 q + 8
kv heads) x head_dim 128, bf16 in, fp32 cos/sin tables, e4m3 + fp32 scale out. The throughput is
the ideal byte ledger per step (every input read once, every output written once, tables and
weights once) divided by the step time.

Timing: 8 rotating input/output sets (8 x 65.7 MB > the 129 MB L2), launches captured in CUDA
graphs and replayed, CUDA events on the launching stream, a barrier + synchronize on both sides,
max over ranks. N > 1 (torchrun, one process per GPU): every rank runs its own batch (weak
scaling, no data-path collective; the process group only carries the barrier and the max).

Beside the number (rank 0): `roofline.size_matched_copy`, the same byte counts streamed by a copy
kernel with the same work distribution and no arithmetic (`fq.stream_floor`), and the prologue's
fraction of it; `cold_launch`, one launch after 256 MB of writes have evicted L2; `e2e`, the same
metric through the public API with host buffers; `cpu_baseline` (one core) and
`cpu_baseline_all_cores` (one token slice per core), the oracle on bounded samples.

--impl reference times the oracle (plain single-threaded C++) on this machine's host cores over
bounded samples of the same workload.
"""
from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import math
import os
import re
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (and % of ~8 TB/s) for fused QK-norm+RoPE+FP8, 1 GB300"
UNIT = "GB/s"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
T_TOK, HQ, HK, D = 4096, 32, 8, 128
WORKLOAD = "qk_norm_rope_quant T=4096 Hq=32 Hk=8 D=128 rope_dim=128 bf16->e4m3 fp32-tables"
KERNEL_SOURCES = ["fp8_quant_memory_gb300/csrc/fq_prologue.cu", "fp8_quant_memory_gb300/csrc/fq_device.cuh",
                  "fp8_quant_memory_gb300/csrc/fq_sync.cuh"]
PROFILE_SUMMARY = os.path.join(ROOT, "profiles", "qk_norm_rope_quant_4k.md")


def dist_env():
    return int(os.environ.get("RANK", "0")), int(os.environ.get("LOCAL_RANK", "0")), int(os.environ.get("WORLD_SIZE", "1"))


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            j = json.load(f)
        return float(j["hbm_gbs"]), "measured"
    except Exception:
        return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash() -> str:
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES:
        with open(os.path.join(ROOT, rel), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def profiled_traffic():
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the current kernel."""
    try:
        with open(PROFILE_SUMMARY) as f:
            text = f.read()
    except OSError:
        return None
    m = re.search(r"kernel_source_sha256:\s*([0-9a-f]+)", text)
    t = re.search(r"traffic_bytes_per_launch:\s*([0-9]+)", text)
    if not (m and t) or m.group(1) != kernel_source_hash():
        return None
    return int(t.group(1))


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None
        self.t0 = self.t1 = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
        time.sleep(0.3)

    def mark(self, begin: bool):
        if begin:
            self.t0 = time.time()
        else:
            self.t1 = time.time()

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        time.sleep(0.25)
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        rows = [r for r in csv.reader(io.StringIO(out)) if len(r) >= 9]
        sm = [float(r[1]) for r in rows if r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        loaded = [s for s in sm if mx and s > 0.5 * max(mx)] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(rows)}


# ------------------------------------------------------------------------------------------------ cases
class Case:
    """One workload: rotating device buffer sets, a launch per set, and the ideal bytes per launch."""

    name = ""
    kernels_per_step = 1

    def bytes_per_step(self) -> int:
        raise NotImplementedError

    def launch(self, i: int):
        raise NotImplementedError


def _make_sets(host: dict, n_sets: int, dev):
    import torch

    sets = []
    for _ in range(n_sets):
        sets.append({k: (v.to(dev).clone() if isinstance(v, torch.Tensor) else v) for k, v in host.items()})
    return sets


class PrologueCase(Case):
    def __init__(self, dev, T=T_TOK, Hq=HQ, Hk=HK, D_=D, std=2.0, theta=1e4, positions="arange",
                 outlier_frac=0.0, n_sets=8, seed=20261202 + 2):
        import torch

        import fp8_quant_memory_gb300 as fq
        from fp8_quant_memory_gb300 import ledger
        from fp8_quant_memory_gb300 import workloads as wl

        self.fq = fq
        self.T, self.Hq, self.Hk, self.D = T, Hq, Hk, D_
        self.name = f"qk_norm_rope_quant T={T} Hq={Hq} Hk={Hk} D={D_}"
        self.host = wl.qk_inputs(T, Hq, Hk, D_, "bf16", "fp32", seed=seed, std=std, theta=theta,
                                 positions=positions, outlier_frac=outlier_frac)
        self.sets = _make_sets({k: self.host[k] for k in ("qk", "wq", "wk", "cos", "sin")}, n_sets, dev)
        for s in self.sets:
            s["q"] = torch.empty((T, Hq + Hk, D_), dtype=torch.uint8, device=dev)
            s["scale"] = torch.empty((T, Hq + Hk), dtype=torch.float32, device=dev)
        self._bytes = ledger.qk_prologue_bytes(T, Hq, Hk, D_)

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.qk_norm_rope_quant(s["qk"], s["wq"], s["wk"], s["cos"], s["sin"], self.Hq, self.Hk,
                                   q_out=s["q"], scale=s["scale"])


class PrologueDesignCase(PrologueCase):
    """The 4k prologue computed as one of the Ch.28 page's designs: one CTA per block of `rpb` rows."""

    def __init__(self, dev, rpb, label):
        super().__init__(dev)
        self.rpb = rpb
        self.name = f"qk_norm_rope_quant T={self.T} Hq={self.Hq} Hk={self.Hk} D={self.D} as design {label} " \
                    f"({rpb} rows per block)"

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.qk_norm_rope_quant_blocks(s["qk"], s["wq"], s["wk"], s["cos"], s["sin"], self.Hq, self.Hk, self.rpb,
                                          q_out=s["q"], scale=s["scale"])


class StreamFloorCase(Case):
    """The size-matched streaming floor (`fq.stream_floor`): the prologue's x bytes read and codes
    bytes written, no arithmetic, the same chunked work distribution and launch attributes."""

    def __init__(self, dev, rows=T_TOK * (HQ + HK), n_sets=8):
        import torch

        import fp8_quant_memory_gb300 as fq

        self.fq = fq
        n16 = rows * D * 2 // 16
        self.name = f"size-matched streaming floor: {n16 * 16 / 1e6:.2f} MB read, {n16 * 8 / 1e6:.2f} MB written"
        self.sets = []
        for i in range(n_sets):
            inp = torch.randint(0, 256, (n16 * 16,), dtype=torch.uint8, device=dev)
            self.sets.append({"in": inp, "out": torch.empty(n16 * 8, dtype=torch.uint8, device=dev)})
        self._bytes = n16 * 24

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.stream_floor(s["in"], out=s["out"])


def cold_launch_us(case: Case, stream, runs: int = 5) -> dict:
    """One launch right after 256 MB of writes have evicted the 129 MB L2, timed alone with events."""
    import torch

    flush = torch.empty(256 << 20, dtype=torch.uint8, device=stream.device)
    times = []
    with torch.cuda.stream(stream):
        for i in range(runs):
            flush.zero_()
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            a.record(stream)
            case.launch(i)
            b.record(stream)
            torch.cuda.synchronize()
            times.append(a.elapsed_time(b) * 1e3)
    times.sort()
    return {"us_median": round(times[len(times) // 2], 3), "runs": runs,
            "flush": "256 MB written before each launch (L2 is 129 MB)"}


class RmsnormFwdCase(Case):
    def __init__(self, dev, M=8192, N=4096, n_sets=3):
        import torch

        import fp8_quant_memory_gb300 as fq
        from fp8_quant_memory_gb300 import ledger
        from fp8_quant_memory_gb300 import workloads as wl

        self.fq = fq
        self.name = f"rmsnorm_fwd M={M} N={N} bf16"
        h = wl.rmsnorm_inputs(M, N, "bf16", seed=20261202 + 1)
        self.sets = _make_sets({"x": h["x"], "w": h["w"]}, n_sets, dev)
        for s in self.sets:
            s["y"] = torch.empty_like(s["x"])
        self._bytes = ledger.rmsnorm_fwd_bytes(M, N)

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.rmsnorm_fwd(s["x"], s["w"], out=s["y"])


class RmsnormBwdCase(Case):
    kernels_per_step = 2

    def __init__(self, dev, M=8192, N=4096, n_sets=2):
        import torch

        import fp8_quant_memory_gb300 as fq
        from fp8_quant_memory_gb300 import ledger
        from fp8_quant_memory_gb300 import workloads as wl

        self.fq = fq
        self.name = f"rmsnorm_bwd M={M} N={N} bf16 (dx + deterministic dw)"
        h = wl.rmsnorm_inputs(M, N, "bf16", seed=20261202 + 1)
        self.sets = _make_sets({"x": h["x"], "w": h["w"], "g": h["g"]}, n_sets, dev)
        nbytes = fq.rmsnorm_bwd_workspace_bytes(M, N)
        for s in self.sets:
            s["ws"] = torch.empty((nbytes,), dtype=torch.uint8, device=dev)
        self._bytes = ledger.rmsnorm_bwd_bytes(M, N)
        self.workspace_bytes = nbytes

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.rmsnorm_bwd(s["x"], s["w"], s["g"], workspace=s["ws"], want_dw_f32=False)


class RmsnormBwdRstdCase(RmsnormBwdCase):
    """The backward with the forward's saved rstd: reads 4 more bytes per row, skips the sum of squares."""

    def __init__(self, dev, M=8192, N=4096, n_sets=2):
        import torch

        super().__init__(dev, M, N, n_sets)
        self.name = f"rmsnorm_bwd_rstd M={M} N={N} bf16 (saved rstd, dx + deterministic dw)"
        for s in self.sets:
            s["rstd"] = self.fq.rmsnorm_fwd_rstd(s["x"], s["w"])[1]
        torch.cuda.synchronize()
        self._bytes += M * 4

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.rmsnorm_bwd_rstd(s["x"], s["w"], s["g"], s["rstd"], workspace=s["ws"], want_dw_f32=False)


class LayerNormCase(Case):
    """LayerNorm forward with bias at the Ch.13 ledger's shape (4096 x 4096)."""

    def __init__(self, dev, M=4096, N=4096, n_sets=8):
        import torch

        import fp8_quant_memory_gb300 as fq
        from fp8_quant_memory_gb300 import workloads as wl

        self.fq = fq
        self.name = f"layernorm_fwd M={M} N={N} bf16 (with bias)"
        h = wl.rmsnorm_inputs(M, N, "bf16", seed=20261202 + 5)
        h = {"x": h["x"], "g": h["w"], "b": (h["w"].float() - 1.0).to(torch.bfloat16)}
        self.sets = _make_sets(h, n_sets, dev)
        for s in self.sets:
            s["y"] = torch.empty_like(s["x"])
        self._bytes = 2 * M * N * 2 + 2 * N * 2

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.layernorm_fwd(s["x"], s["g"], s["b"], out=s["y"])


class RopeCase(Case):
    def __init__(self, dev, M=65536, N=192, R=64, n_sets=8):
        import torch

        import fp8_quant_memory_gb300 as fq
        from fp8_quant_memory_gb300 import ledger
        from fp8_quant_memory_gb300 import workloads as wl

        self.fq = fq
        self.name = f"rmsnorm_rope M={M} N={N} R={R} fp16"
        h = wl.rows_inputs(M, N, R, "fp16", "fp16", seed=20261202 + 3, heads_per_token=32)
        self.sets = _make_sets(h, n_sets, dev)
        for s in self.sets:
            s["y"] = torch.empty_like(s["x"])
        self._bytes = ledger.rope_bytes(M, N, R, "fp16", "fp16")

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        self.fq.rmsnorm_rope(s["x"], s["w"], s["cos"], s["sin"], out=s["y"])


class RopeQuantCase(Case):
    """rmsnorm_rope_quant (one scale per row) or rmsnorm_rope_quant_groups (one per group_size columns)."""

    def __init__(self, dev, M=256, N=512, R=64, group_size=None, write_y=True, n_sets=8, note="",
                 seed=20261202):
        import fp8_quant_memory_gb300 as fq
        from fp8_quant_memory_gb300 import ledger
        from fp8_quant_memory_gb300 import workloads as wl

        import torch

        self.fq = fq
        self.gs = group_size
        self.write_y = write_y
        kind = "rmsnorm_rope_quant" if group_size is None else f"rmsnorm_rope_quant_groups gs={group_size}"
        self.name = f"{kind} M={M} N={N} R={R} bf16{'' if write_y else ' (no y)'}{note}"
        h = wl.rows_inputs(M, N, R, "bf16", "bf16", seed=seed)
        self.sets = _make_sets(h, n_sets, dev)
        n_scales = M if group_size is None else M * (N // group_size)
        for s in self.sets:
            s["y"] = torch.empty_like(s["x"]) if write_y else None
            s["q"] = torch.empty((M, N), dtype=torch.uint8, device=dev)
            s["scale"] = torch.empty((n_scales,), dtype=torch.float32, device=dev)
        self._bytes = ledger.rope_quant_bytes(M, N, R, "bf16", "bf16", write_y=write_y, group_size=group_size)

    def bytes_per_step(self):
        return self._bytes

    def launch(self, i):
        s = self.sets[i % len(self.sets)]
        if self.gs is None:
            self.fq.rmsnorm_rope_quant(s["x"], s["w"], s["cos"], s["sin"], want_y=self.write_y, y=s["y"],
                                       q=s["q"], scale=s["scale"])
        else:
            self.fq.rmsnorm_rope_quant_groups(s["x"], s["w"], s["cos"], s["sin"], self.gs, want_y=self.write_y,
                                              y=s["y"], q=s["q"], scale=s["scale"])


class TorchEagerPrologueCase(Case):
    """Unfused per-op PyTorch sequence for the same prologue (RMSNorm -> RoPE -> amax -> divide ->
    cast), the comparison the Ch.13 ledger's unfused plan models. Bench-only comparator."""

    def __init__(self, prologue: PrologueCase):
        import torch

        self.torch = torch
        self.p = prologue
        self.name = "torch eager unfused prologue (same workload)"
        self.kernels_per_step = None

    def bytes_per_step(self):
        return self.p.bytes_per_step()

    def launch(self, i):
        torch = self.torch
        p = self.p
        s = p.sets[i % len(p.sets)]
        x = s["qk"].float()
        rstd = torch.rsqrt(x.pow(2).mean(-1, keepdim=True) + 1e-6)
        w = torch.cat([s["wq"].float().expand(p.Hq, p.D), s["wk"].float().expand(p.Hk, p.D)])
        n = x * rstd * w
        half = p.D // 2
        c = s["cos"][:, None, :]
        sn = s["sin"][:, None, :]
        lo, hi = n[..., :half], n[..., half:]
        y = torch.cat([lo * c - hi * sn, hi * c + lo * sn], dim=-1)
        amax = y.abs().amax(-1, keepdim=True).clamp(min=1e-4)
        scale = amax / 448.0
        s["q"].copy_((y / scale).clamp(-448, 448).to(torch.float8_e4m3fn).view(torch.uint8))
        s["scale"].copy_(scale.squeeze(-1))


# ------------------------------------------------------------------------------------------------ timing
def _external_timing_events():
    """Two timing events that become event-record nodes when recorded during graph capture, or None
    where this torch has no such events."""
    import torch

    try:
        return (torch.cuda.Event(enable_timing=True, external=True),
                torch.cuda.Event(enable_timing=True, external=True))
    except TypeError:
        return None


TIMING_MODE = {"mode": None}  # how the last time_case call timed its launches


def time_case(case: Case, steps: int, warmup: int, stream, use_graph=True, graph_len=256, single_graph_max=4096):
    """Run at least `warmup` untimed steps, then exactly `steps` timed steps; returns (ms_total,
    warm-up launches actually run).

    Up to `single_graph_max` launches in all, one CUDA graph holds the `warmup` launches, the start
    event, the `steps` timed launches and the end event (event-record nodes): the timed region runs
    from the completion of the last warm-up launch to the completion of the last timed one, `steps`
    launch periods of a back-to-back stream. The graph is replayed twice (the first replay uploads
    it) and timed on the second. Longer runs replay a
    graph of `graph_len` launches: the warm-up is whole replays, and the last warm-up replay is
    queued right before the start event, so that the event fires on a busy stream and the timed
    launches are already submitted (the host-side submission of a replay does not land inside the
    device timing; the device-side gap between two replays, a few microseconds, does, once per
    `graph_len` launches). Every timed launch does its full work."""
    import torch

    torch.cuda.synchronize()
    events = _external_timing_events() if use_graph and warmup + steps <= single_graph_max else None
    if events is not None:
        TIMING_MODE["mode"] = "one CUDA graph of the warm-up and timed launches, events as graph nodes"
        start, end = events
        case.launch(0)  # eager first call: caches occupancy queries outside capture
        torch.cuda.synchronize()
        side = torch.cuda.Stream(stream.device)
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(warmup):
                case.launch(i)
            # The start event hangs off the last warm-up launch on a side branch: it fires when that
            # launch completes, and the first timed launch keeps its programmatic-launch edge to it
            # (an event node in the main chain would make the first timed launch wait for a full
            # completion that no other launch waits for).
            side.wait_stream(stream)
            with torch.cuda.stream(side):
                start.record(side)
            for i in range(steps):
                case.launch(warmup + i)
            stream.wait_stream(side)
            end.record(stream)
        with torch.cuda.stream(stream):
            graph.replay()  # uploads the graph; its launches are more warm-up
        torch.cuda.synchronize()
        barrier()
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            graph.replay()
        torch.cuda.synchronize()
        barrier()
        return start.elapsed_time(end), 2 * warmup + steps + 1

    graph = None
    TIMING_MODE["mode"] = f"CUDA graphs of up to {graph_len} launches, replayed" if use_graph else "eager launches"
    if use_graph:
        case.launch(0)  # eager first call: caches occupancy queries outside capture
        torch.cuda.synchronize()
        n = max(1, min(graph_len, steps))
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for i in range(n):
                case.launch(i)
        rem = steps % n
        graph_rem = None
        if rem:
            graph_rem = torch.cuda.CUDAGraph()
            with torch.cuda.graph(graph_rem, stream=stream):
                for i in range(rem):
                    case.launch(i)
        # one replay of each graph uploads it
        done = 0
        with torch.cuda.stream(stream):
            graph.replay()
            done += n
            if graph_rem is not None:
                graph_rem.replay()
                done += rem
    else:
        done = 0
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    barrier()
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        if use_graph:
            # the rest of the warm-up, ending with one replay queued just ahead of the start event
            while True:
                graph.replay()
                done += n
                if done >= warmup:
                    break
        else:
            for i in range(warmup):
                case.launch(i)
            done = warmup
        start.record(stream)
        if use_graph:
            for _ in range(steps // n):
                graph.replay()
            if graph_rem is not None:
                graph_rem.replay()
        else:
            for i in range(steps):
                case.launch(i)
        end.record(stream)
    torch.cuda.synchronize()
    barrier()
    return start.elapsed_time(end), done


_PG = None
_PG_DEVICE = "cpu"


def barrier():
    if _PG is not None:
        import torch.distributed as dist

        dist.barrier()


def max_over_ranks(v: float) -> float:
    """Largest value of `v` over all ranks (the job's time is its slowest rank's)."""
    if _PG is None:
        return v
    import torch
    import torch.distributed as dist

    t = torch.tensor([v], dtype=torch.float64, device=_PG_DEVICE)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput_gbs(bytes_per_step: int, steps: int, max_ms: float, world: int) -> float:
    """Whole-job GB/s: every rank processed `steps` batches of `bytes_per_step` (weak scaling) in
    the slowest rank's time."""
    return world * bytes_per_step * steps / (max_ms * 1e-3) / 1e9


def e2e_prologue(case: PrologueCase, steps: int, stream):
    """Same metric through the public API with host buffers: every step copies its inputs from pinned
    host memory to the device, runs the call, and copies q and scale back to pinned host memory.
    Two device buffer sets and three streams pipeline the steps: step i+1's upload (one copy engine)
    overlaps step i's kernel and download (the other direction); events keep each buffer set's
    copies, kernel and read-back in order."""
    import torch

    fq = case.fq
    keys = ("qk", "wq", "wk", "cos", "sin")
    sets = case.sets[:2]
    host_in = {k: case.host[k].pin_memory() for k in keys}
    host_q = [torch.empty(sets[0]["q"].shape, dtype=torch.uint8).pin_memory() for _ in sets]
    host_s = [torch.empty(sets[0]["scale"].shape, dtype=torch.float32).pin_memory() for _ in sets]
    h2d = sum(t.numel() * t.element_size() for t in host_in.values())
    d2h = host_q[0].numel() + host_s[0].numel() * 4
    dev = sets[0]["qk"].device
    up, down = torch.cuda.Stream(dev), torch.cuda.Stream(dev)
    ev_up = [torch.cuda.Event() for _ in sets]      # inputs of set b are on the device
    ev_run = [torch.cuda.Event() for _ in sets]     # the kernel on set b is done
    ev_down = [torch.cuda.Event() for _ in sets]    # the results of set b are on the host
    started = [False, False]

    def run(n):
        for i in range(n):
            b = i % 2
            s = sets[b]
            with torch.cuda.stream(up):
                if started[b]:
                    up.wait_event(ev_run[b])         # the previous kernel on this set has read its inputs
                for k in keys:
                    s[k].copy_(host_in[k], non_blocking=True)
                ev_up[b].record(up)
            with torch.cuda.stream(stream):
                stream.wait_event(ev_up[b])
                if started[b]:
                    stream.wait_event(ev_down[b])    # the previous results of this set have been read back
                fq.qk_norm_rope_quant(s["qk"], s["wq"], s["wk"], s["cos"], s["sin"], case.Hq, case.Hk,
                                      q_out=s["q"], scale=s["scale"])
                ev_run[b].record(stream)
            with torch.cuda.stream(down):
                down.wait_event(ev_run[b])
                host_q[b].copy_(s["q"], non_blocking=True)
                host_s[b].copy_(s["scale"], non_blocking=True)
                ev_down[b].record(down)
            started[b] = True

    run(4)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(up)
    run(steps)
    for b in range(len(sets)):
        up.wait_event(ev_down[b])
    end.record(up)
    torch.cuda.synchronize()
    ms = start.elapsed_time(end)
    return {"value": round(case.bytes_per_step() * steps / (ms * 1e-3) / 1e9, 2), "unit": UNIT,
            "steps": steps, "ms_per_step": round(ms / steps, 4), "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h, "pipelining": "2 buffer sets; upload, kernel, download on 3 streams"}


def cpu_oracle_sample(budget_s: float = 12.0):
    """The oracle on bounded samples of the prologue workload (whole batches, repeated until the time
    budget is spent): GB/s of the same ledger, single thread."""
    import oracle
    from fp8_quant_memory_gb300 import ledger
    from fp8_quant_memory_gb300 import workloads as wl

    d = wl.qk_inputs(T_TOK, HQ, HK, D, "bf16", "fp32", seed=20261202 + 2, std=2.0)
    oracle.lib()
    bytes_per = ledger.qk_prologue_bytes(T_TOK, HQ, HK, D)
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle.qk_norm_rope_quant(d["qk"], d["wq"], d["wk"], d["cos"], d["sin"], HQ, HK)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s:
            break
    return {"value": round(bytes_per * reps / el / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"{reps} full batches of {T_TOK} tokens x {HQ + HK} heads x {D} in {el:.1f} s"}


def cpu_oracle_all_cores(budget_s: float = 10.0):
    """The same oracle, unchanged, on every host core: the 4096 tokens split into one slice per core,
    the slices run on a thread pool (the oracle is a C library called through ctypes, which releases
    the interpreter lock, and it keeps no global state). Whole batches repeated until the budget is
    spent; GB/s of the same ledger."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle
    from fp8_quant_memory_gb300 import ledger
    from fp8_quant_memory_gb300 import workloads as wl

    d = wl.qk_inputs(T_TOK, HQ, HK, D, "bf16", "fp32", seed=20261202 + 2, std=2.0)
    oracle.lib()
    cores = max(1, os.cpu_count() or 1)
    bounds = [(T_TOK * i // cores, T_TOK * (i + 1) // cores) for i in range(cores)]
    slices = [{k: d[k][a:b].contiguous() for k in ("qk", "cos", "sin")} for a, b in bounds if b > a]

    def run(sl):
        oracle.qk_norm_rope_quant(sl["qk"], d["wq"], d["wk"], sl["cos"], sl["sin"], HQ, HK)

    bytes_per = ledger.qk_prologue_bytes(T_TOK, HQ, HK, D)
    reps = 0
    with ThreadPoolExecutor(len(slices)) as ex:
        t0 = time.perf_counter()
        while True:
            list(ex.map(run, slices))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
    return {"value": round(bytes_per * reps / el / 1e9, 4), "unit": UNIT, "cores": len(slices), "kind": "oracle",
            "sample": f"{reps} full batches of {T_TOK} tokens x {HQ + HK} heads x {D}, one token slice per core, "
                      f"in {el:.1f} s"}


def run_reference(args):
    rank, _, world = dist_env()
    if rank != 0:
        return 0
    import oracle
    from fp8_quant_memory_gb300 import ledger
    from fp8_quant_memory_gb300 import workloads as wl

    d = wl.qk_inputs(T_TOK, HQ, HK, D, "bf16", "fp32", seed=20261202 + 2, std=2.0)
    oracle.lib()
    # size each step so the whole run stays within about a minute
    t0 = time.perf_counter()
    oracle.qk_norm_rope_quant(d["qk"][:64].contiguous(), d["wq"], d["wk"], d["cos"][:64].contiguous(),
                              d["sin"][:64].contiguous(), HQ, HK)
    per_token = (time.perf_counter() - t0) / 64
    total = max(args.steps + args.warmup, 1)
    tok = int(max(1, min(T_TOK, 60.0 / (total * per_token))))
    sl = {k: d[k][:tok].contiguous() for k in ("qk", "cos", "sin")}
    bytes_per = ledger.qk_prologue_bytes(tok, HQ, HK, D)
    for _ in range(args.warmup):
        oracle.qk_norm_rope_quant(sl["qk"], d["wq"], d["wk"], sl["cos"], sl["sin"], HQ, HK)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.qk_norm_rope_quant(sl["qk"], d["wq"], d["wk"], sl["cos"], sl["sin"], HQ, HK)
    el = time.perf_counter() - t0
    val = bytes_per * args.steps / el / 1e9
    sample = f"each step: the first {tok} of {T_TOK} tokens x {HQ + HK} heads x {D}"
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(val, 4), "unit": UNIT, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(el * 1e3 / max(args.steps, 1), 4),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens_per_step": tok},
        "cpu_baseline": {"value": round(val, 4), "unit": UNIT, "cores": 1, "kind": "oracle", "sample": sample},
        "e2e": {"value": round(val, 4), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))
    return 0


SECONDARY = {
    "rmsnorm_fwd_8k_4k": lambda dev: RmsnormFwdCase(dev),
    "rmsnorm_bwd_8k_4k": lambda dev: RmsnormBwdCase(dev),
    "rmsnorm_bwd_rstd_8k_4k": lambda dev: RmsnormBwdRstdCase(dev),
    "rope_fp16_64k": lambda dev: RopeCase(dev),
    "layernorm_4k_4k": lambda dev: LayerNormCase(dev),
    "rope_quant_tiny": lambda dev: RopeQuantCase(dev, note=" (launch-bound)"),
    "rope_quant_groups_tiny": lambda dev: RopeQuantCase(dev, group_size=128, note=" (launch-bound)"),
    "rope_quant_ledger_4k": lambda dev: RopeQuantCase(dev, M=4096, N=4096, R=128, write_y=False, n_sets=8,
                                                      note=" (Ch.13 ledger fused workload)"),
    "rope_quant_groups_ledger_4k": lambda dev: RopeQuantCase(dev, M=4096, N=4096, R=128, group_size=128,
                                                             write_y=False, n_sets=8),
    "rope_quant_16k": lambda dev: RopeQuantCase(dev, M=16384, N=4096, R=128, write_y=False, n_sets=4,
                                                note=" (the ledger workload at four times the rows)"),
    "prologue_4k_design_a": lambda dev: PrologueDesignCase(dev, 1, "A"),
    "prologue_4k_design_b": lambda dev: PrologueDesignCase(dev, 8, "B"),
    "prologue_4k_design_c": lambda dev: PrologueDesignCase(dev, HQ + HK, "C"),
    "qk_prologue_32k": lambda dev: PrologueCase(dev, T=32768, Hq=64, Hk=8, std=1.0, theta=1e6, positions="uniform",
                                                outlier_frac=0.01, n_sets=2, seed=20261202 + 4),
}


def time_secondary(c: Case, steps: int, warmup: int, stream, peak: float) -> dict:
    ms, _ = time_case(c, steps, warmup, stream)
    us = ms * 1e3 / steps
    gbs = c.bytes_per_step() / (us * 1e-6) / 1e9
    return {"workload": c.name, "us_per_step": round(us, 3), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4),
            "bytes_per_step": c.bytes_per_step(), "kernels_per_step": c.kernels_per_step}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100000)
    ap.add_argument("--warmup", type=int, default=1024)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-extras", action="store_true", help="skip the secondary workloads")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--workload", choices=["qk_prologue_4k", "torch_eager_prologue", *SECONDARY], default="qk_prologue_4k",
                    help="time one secondary workload alone (for profiling) instead of the benchmark step")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)

    import torch

    global _PG, _PG_DEVICE
    rank, local_rank, world = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
        _PG = dist.group.WORLD
        _PG_DEVICE = f"cuda:{local_rank}"
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    import fp8_quant_memory_gb300 as fq
    from fp8_quant_memory_gb300 import _capi

    _capi.load()
    stream = torch.cuda.Stream(dev)
    if args.workload == "torch_eager_prologue":
        # The unfused per-op torch sequence alone (no graphs), then one more step inside an NVTX range
        # ("eager_step") so that a profiler can sum the DRAM bytes of exactly one step's kernels.
        eager = TorchEagerPrologueCase(PrologueCase(dev))
        ms, _ = time_case(eager, args.steps, args.warmup, stream, use_graph=False)
        with torch.cuda.stream(stream):
            torch.cuda.nvtx.range_push("eager_step")
            eager.launch(0)
            torch.cuda.nvtx.range_pop()
        torch.cuda.synchronize()
        if rank == 0:
            us = ms * 1e3 / args.steps
            print(json.dumps({"workload": eager.name, "us_per_step": round(us, 3),
                              "GB/s_of_fused_ledger": round(eager.bytes_per_step() / (us * 1e-6) / 1e9, 1)}),
                  flush=True)
        return 0
    if args.workload != "qk_prologue_4k":
        res = time_secondary(SECONDARY[args.workload](dev), args.steps, args.warmup, stream, peaks()[0])
        if rank == 0:
            print(json.dumps(res), flush=True)
        return 0

    case = PrologueCase(dev)
    sampler = ClockSampler(int(os.environ.get("CUDA_VISIBLE_DEVICES", str(local_rank)).split(",")[0])
                           if os.environ.get("CUDA_VISIBLE_DEVICES", "").split(",")[0].isdigit() else local_rank)
    sampler.start()
    ms, warm_done = time_case(case, args.steps, args.warmup, stream)
    launch_mode = TIMING_MODE["mode"]
    clocks = sampler.stop()
    ms = max_over_ranks(ms)
    status = fq.device_status(clear=True)

    per_launch_us = ms * 1e3 / args.steps
    bytes_step = case.bytes_per_step()
    from fp8_quant_memory_gb300 import ledger as _ledger

    ledger_flops = _ledger.qk_prologue_flops(T_TOK, HQ, HK, D)
    value = job_throughput_gbs(bytes_step, args.steps, ms, world)
    achieved = bytes_step / (per_launch_us * 1e-6) / 1e9
    peak, peak_kind = peaks()

    line = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "warmup_launches_run": warm_done, "ms_per_step": round(ms / args.steps, 6),
        "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": WORKLOAD, "tokens": T_TOK, "q_heads": HQ, "kv_heads": HK, "head_dim": D,
                   "rope_dim": D, "bytes_per_step": bytes_step, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2: 8 rotating input/output sets, 525 MB per rotation",
                   "launch": launch_mode},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "peak_kind": peak_kind,
                     "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
                     "traffic": profiled_traffic(), "kernel": "prologue_tma_kernel<bf16,float,32>",
                     "us_per_launch": round(per_launch_us, 3)},
        "rows_per_s": round(T_TOK * (HQ + HK) * args.steps * world / (ms * 1e-3), 1),
        "flops_per_step": ledger_flops, "arithmetic_intensity_flop_per_byte": round(ledger_flops / bytes_step, 3),
        "gpu_launches": args.steps * case.kernels_per_step,
        "clocks": clocks,
        "device_status": status,
    }
    if rank == 0:
        # Context for the fraction: the size-matched streaming floor and one cold launch.
        fl = StreamFloorCase(dev)
        floor = time_secondary(fl, 2048, 64, stream, peak)
        del fl
        torch.cuda.empty_cache()
        line["roofline"]["size_matched_copy"] = {"us_per_launch": floor["us_per_step"], "GB/s": floor["GB/s"],
                                                 "bytes": floor["bytes_per_step"],
                                                 "kernel": "stream_floor_kernel (fq_stream_floor)"}
        line["roofline"]["frac_of_size_matched_copy"] = round(achieved / floor["GB/s"], 4)
        line["cold_launch"] = cold_launch_us(case, stream)
        line["e2e"] = e2e_prologue(case, min(args.steps, 200), stream)
        if not args.no_extras:
            extras = []
            for name, mk in SECONDARY.items():
                c = mk(dev)
                k = 2000 if c.bytes_per_step() < 3e8 else 400
                extras.append(time_secondary(c, k, 16, stream, peak))
                del c
                torch.cuda.empty_cache()
            eager = TorchEagerPrologueCase(case)
            m3, _ = time_case(eager, 50, 5, stream, use_graph=False)
            us = m3 * 1e3 / 50
            extras.append({"workload": eager.name, "us_per_step": round(us, 3),
                           "GB/s_of_fused_ledger": round(bytes_step / (us * 1e-6) / 1e9, 1)})
            line["also"] = extras
        if world == 1 and not args.no_cpu:
            line["cpu_baseline"] = cpu_oracle_sample()
            line["cpu_baseline_all_cores"] = cpu_oracle_all_cores()
        print(json.dumps(line), flush=True)
    if _PG is not None:
        import torch.distributed as dist

        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
