"""Benchmark: batch-one N:M bitmask SpMV on one decode step of a 70B-shaped model.

One *step* is one token through an 80-layer Llama-3.3-70B-shaped decoder: per
layer four SpMVs (W_qkv 10240x8192, W_o 8192x8192, W_gate+up 57344x8192,
W_down 8192x28672), 320 nm_spmv calls in all.  The packed weights sit in a
rotating set of physical layer slots (far larger than the 129 MB L2) that the
80 logical layers cycle through, so every call streams its weights from HBM.

Reported (one JSON line on stdout, rank 0):
  value        achieved HBM GB/s of the whole step: algorithmic bytes
               (values + masks + x + y) / device time, inputs resident;
  us_per_call  per matrix, from CUDA events around each launch;
  speedup_vs_dense   dense_gemv step time / nm_spmv step time, same shapes;
  patterns     the same step for 2:4, 4:8, 8:16, 16:32;
  e2e          the same metric through the Python/C-ABI calls with x copied
               in from pinned host memory and y copied back every step;
  roofline     the SpMV kernel's achieved GB/s over the measured HBM peak;
  workloads    the other decode-layer workloads (8B, 32B, pattern sweep, 4096^2);
  small_batch  the same step at 2, 4, 6 and 8 tokens through nm_spmm, against
               cuBLAS (torch.mm) at the same batch;
  swiglu_fused the same step with gate+up through nm_spmv_swiglu (the SwiGLU
               activation fused into the SpMV's epilogue);
  prefill      one layer's projections at 64 and 256 tokens through the
               tensor-core nm_spmm_prefill, against cuBLAS fp16 GEMM;
  cpu_baseline the plain C oracle on a bounded sample of the same workload.
Timing: CUDA graph replays timed with CUDA events on the launching stream,
W untimed warm-up steps, then exactly K timed steps between barriers and
device synchronisation; L2 is defeated by the rotating set (stated in config).

``--prefill T`` times the prefill regime instead: the same layer's four
projections for T tokens at once through nm_spmm_prefill (tensor cores),
against cuBLAS fp16 GEMM on the dense weights (dense-equivalent TFLOP/s).

``--impl reference`` times the CPU oracle instead (the slow reference arm).
Multi-GPU (torchrun, N ranks): every rank runs an independent replica (the
path has no exchange step); value = all ranks' bytes / the slowest rank's time.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "N:M SpMV µs/call & achieved HBM GB/s (% peak) at batch 1; speedup vs dense GEMV"
PREFILL_METRIC = ("N:M prefill SpMM dense-equivalent TFLOP/s (2*rows*cols*tokens per call) on the "
                  "tensor cores; speedup vs cuBLAS fp16 GEMM")
FALLBACK_HBM_GBS = 6800.0
FALLBACK_BF16_TFLOPS = 1900.0
NOMINAL_HBM_GBS = 7900.0

WORKLOADS = {
    "llama33_70b_layer": [("qkv", 10240, 8192), ("o", 8192, 8192), ("gate_up", 57344, 8192),
                          ("down", 8192, 28672)],
    "qwen3_32b_layer": [("qkv", 10240, 5120), ("o", 5120, 8192), ("gate_up", 51200, 5120),
                        ("down", 5120, 25600)],
    "llama31_8b_layer": [("qkv", 6144, 4096), ("o", 4096, 4096), ("gate_up", 28672, 4096),
                         ("down", 4096, 14336)],
    "pattern_sweep": [("up", 14336, 4096), ("down", 4096, 14336)],
    "single_4096": [("W", 4096, 4096)],
}
PATTERNS = [(2, 4), (4, 8), (8, 16), (16, 32)]
# decoder layers of each model (one step = one token through all of them)
LAYERS = {"llama33_70b_layer": 80, "qwen3_32b_layer": 64, "llama31_8b_layer": 32,
          "pattern_sweep": 32, "single_4096": 64}


# ---------------------------------------------------------------------------
# byte accounting (the algorithmic traffic of one call)
# ---------------------------------------------------------------------------
def sparse_bytes(rows: int, cols: int) -> int:
    return rows * cols + rows * cols // 8 + 2 * cols + 2 * rows


def dense_bytes(rows: int, cols: int) -> int:
    return 2 * rows * cols + 2 * cols + 2 * rows


# ---------------------------------------------------------------------------
# multi-rank plumbing (host logic; tested with gloo on CPU)
# ---------------------------------------------------------------------------
def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def aggregate(local_units: float, local_seconds: float, group=None):
    """Whole-job totals across ranks: (sum of units, max of seconds)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()):
        return local_units, local_seconds
    dev = "cuda" if dist.get_backend(group) == "nccl" else "cpu"
    u = torch.tensor([float(local_units)], dtype=torch.float64, device=dev)
    s = torch.tensor([float(local_seconds)], dtype=torch.float64, device=dev)
    dist.all_reduce(u, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(s, op=dist.ReduceOp.MAX, group=group)
    return float(u.item()), float(s.item())


def barrier():
    import torch.distributed as dist
    if dist.is_available() and dist.is_initialized():
        dist.barrier()


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("timestamp,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.dev = self.smi_id(device_index)
        self.proc = None
        self.path = None
        self.windows = []  # [start, stop] of every timed region

    def start(self):
        import datetime
        self.windows.append([datetime.datetime.now(), None])

    def stop(self):
        import datetime
        if self.windows and self.windows[-1][1] is None:
            self.windows[-1][1] = datetime.datetime.now()

    @staticmethod
    def smi_id(local: int) -> str:
        """nvidia-smi id of the CUDA device (PCI bus id when torch exposes it)."""
        try:
            import torch
            p = torch.cuda.get_device_properties(local)
            return f"{p.pci_domain_id:08X}:{p.pci_bus_id:02X}:{p.pci_device_id:02X}.0"
        except (AttributeError, RuntimeError):
            vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
            ids = [t for t in vis.split(",") if t.strip()]
            return ids[local].strip() if local < len(ids) else str(local)

    def __enter__(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        """Clock samples taken inside the start()/stop() windows (all if unmarked)."""
        import datetime
        if self.proc is None or not self.path or not os.path.exists(self.path):
            return None
        rows = []
        for line in open(self.path):
            f = [t.strip() for t in line.split(",")]
            if len(f) < 9:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f")
                rows.append((float(f[1]), float(f[2]), float(f[3]), f[5:9], ts))
            except ValueError:
                continue
        os.unlink(self.path)
        wins = [(a, b) for a, b in self.windows if a is not None and b is not None]
        first = [r for r in rows if wins and wins[0][0] <= r[4] <= wins[0][1]]
        if wins:
            inside = [r for r in rows if any(a <= r[4] <= b for a, b in wins)]
            rows = inside or rows
        if not rows:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

        def reasons_of(rs):
            return sorted({names[i] for r in rs for i, v in enumerate(r[3]) if v.lower() == "active"})

        out = {"sm_mhz": statistics.median(r[0] for r in rows),
               "sm_max_mhz": max(r[1] for r in rows),
               "power_w_max": max(r[2] for r in rows),
               "samples": len(rows), "reasons": reasons_of(rows)}
        if first and len(wins) > 1:
            # the first timed region is the headline's: its own record, apart
            # from the later sections (dense GEMMs can reach the power cap)
            out["headline_window"] = {"sm_mhz": statistics.median(r[0] for r in first),
                                      "power_w_max": max(r[2] for r in first),
                                      "samples": len(first), "reasons": reasons_of(first)}
        return out


# ---------------------------------------------------------------------------
# peaks, profiles
# ---------------------------------------------------------------------------
def hbm_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def tensor_peak(seconds_timed: float):
    """Measured dense bf16 tensor peak (fp16 runs at the same nominal rate):
    the sustained figure for a timed region of a second or more, else burst."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        if seconds_timed >= 1.0 and "bf16_tflops_sustained" in d:
            return float(d["bf16_tflops_sustained"]), "measured sustained (bf16_tflops_sustained)"
        return float(d["bf16_tflops"]), "measured burst (bf16_tflops)"
    except (OSError, KeyError, ValueError):
        return FALLBACK_BF16_TFLOPS, "fallback 1900 TFLOP/s"


def kernel_source_hash(names=("spmv.cu", "device.cuh", "split.cuh")) -> str:
    """Hash of the files that define a kernel's code (by default the SpMV
    kernels'); a committed ncu traffic record is used only while it matches."""
    h = hashlib.sha256()
    for name in names:
        with open(os.path.join(ROOT, "sparse_spmv_memory_gb300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


PREFILL_SOURCES = ("prefill.cu", "tc.cuh", "device.cuh")
SPMM_SOURCES = ("spmm.cu", "spmm_kernels.cuh", "spmm_variants.h", "spmm_b2.cu", "spmm_b4.cu",
                "spmm_b6.cu", "spmm_b8.cu", "device.cuh", "split.cuh")


def ncu_traffic(shape_key: str, record="nm_spmv_traffic.json", sources=None):
    """DRAM bytes per launch from a committed ncu summary, if it was taken on
    the kernel source as it is now (else None)."""
    p = os.path.join(ROOT, "profiles", record)
    try:
        with open(p) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    want = kernel_source_hash(sources) if sources else kernel_source_hash()
    if d.get("kernel_source_hash") != want:
        return None
    e = d.get("per_launch", {}).get(shape_key)
    return None if e is None else float(e["dram_bytes"])


# ---------------------------------------------------------------------------
# CPU oracle timing (cpu_baseline leg and the reference arm)
# ---------------------------------------------------------------------------
def batch_metric(batch: int) -> str:
    """The line's metric: the headline's at one token, the SpMM's at 2..8."""
    if batch == 1:
        return METRIC
    return f"N:M SpMM at {batch} tokens: achieved HBM GB/s (% peak); speedup vs cuBLAS"


def oracle_pack_sample(mats, pattern, rows_per, tokens=1):
    """Oracle-packed first ``rows_per`` rows of every matrix and ``tokens``
    activation vectors per matrix (not timed)."""
    import oracle
    import synth
    orc = oracle.Oracle()
    N, M = pattern
    packed = []
    for mi, (name, rows, cols) in enumerate(mats):
        n = min(rows_per, rows)
        W = synth.normal_f16((n, cols), 0, synth.stream_id(2, mi, 0), synth.WEIGHT_SIGMA)
        xs = [synth.activations(cols, 0, synth.stream_id(2, mi, 1) if t == 0
                                else synth.stream_id(2, mi, 1, t)) for t in range(tokens)]
        v, m = orc.prune_pack(W, N, M)
        packed.append((v, m, cols, xs, n))
    return orc, packed


def oracle_run(orc, packed):
    """The timed oracle work: unpack to dense + double matvec per token;
    returns the weight bytes (counted once per step, whatever the tokens)."""
    nbytes = 0
    for v, m, cols, xs, n in packed:
        for x in xs:
            orc.spmv_f64(v, m, cols, x)
        nbytes += sparse_bytes(n, cols)
    return nbytes


def oracle_sample(mats, pattern, seconds: float):
    """Grow a sample of rows until the oracle takes about ``seconds`` on it.
    Returns (rows_per_matrix, bytes, elapsed_s, description)."""
    rows_per = 8
    while True:
        orc, packed = oracle_pack_sample(mats, pattern, rows_per)
        t0 = time.perf_counter()
        nbytes = oracle_run(orc, packed)
        dt = time.perf_counter() - t0
        full = all(rows_per >= r for _, r, _ in mats)
        if dt >= seconds * 0.5 or full:
            desc = (f"first {rows_per} rows of each of the {len(mats)} matrices, "
                    f"{pattern[0]}:{pattern[1]}, oracle unpack + double matvec, 1 thread")
            return rows_per, nbytes, dt, desc
        rows_per = int(rows_per * max(2.0, min(16.0, seconds / max(dt, 1e-4))))


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------
def make_xs(mats, device, batch=1):
    """The step's activations: [batch][cols] fp16 per matrix (token 0 is the
    batch-one x)."""
    import torch
    import synth
    xs = []
    for mi, (name, rows, cols) in enumerate(mats):
        xh = np.stack([synth.activations(cols, 0, synth.stream_id(2, mi, 1) if j == 0
                                         else synth.stream_id(2, mi, 1, j))
                       for j in range(batch)])
        xs.append(torch.from_numpy(xh.view(np.int16)).to(device).view(torch.float16))
    return xs


def make_dense(mats, device, batch=1):
    import torch
    import synth
    dense = []
    for mi, (name, rows, cols) in enumerate(mats):
        host = torch.empty((rows, cols), dtype=torch.int16, pin_memory=True)
        synth.normal_f16_into(host.data_ptr(), rows * cols, 0, synth.stream_id(2, mi, 0),
                              synth.WEIGHT_SIGMA)
        dense.append(host.to(device, non_blocking=True).view(torch.float16))
    xs = make_xs(mats, device, batch)
    torch.cuda.synchronize()
    return dense, xs


def pack_slots(nm, dense, pattern, slots):
    """Pack every matrix once, then copy it into ``slots`` physical layer slots."""
    import torch
    N, M = pattern
    out = []
    base = [nm.nm_pack(W, N, M) for W in dense]
    for s in range(slots):
        if s == 0:
            out.append(base)
        else:
            out.append([(v.clone(), m.clone()) for v, m in base])
    torch.cuda.synchronize()
    return out


def dense_slots(dense, slots):
    import torch
    out = [dense] + [[W.clone() for W in dense] for _ in range(slots - 1)]
    torch.cuda.synchronize()
    return out


class Step:
    """The calls of one decode step over `layers` logical layers, for a batch
    of `batch` tokens (1: nm_spmv / dense_gemv; 2..8: nm_spmm, and cuBLAS as
    the dense reference since dense_gemv is batch-one)."""

    def __init__(self, nm, mats, layers, device, flags=None, batch=1, swiglu=False, tc24=False):
        import torch
        self.nm, self.mats, self.layers, self.flags, self.batch = nm, mats, layers, flags, batch
        # 2:4 weights through nm_spmm24 (tensor cores, 1..8 tokens) instead of nm_spmm
        self.tc24 = tc24
        # fuse the SwiGLU activation into the gate+up call (batch one only)
        self.swiglu = [swiglu and batch == 1 and name == "gate_up" for name, _, _ in mats]
        self.x_off, self.y_off = [], []
        xo = yo = 0
        for _, rows, cols in mats:
            self.x_off.append(xo)
            self.y_off.append(yo)
            xo += cols
            yo += rows
        self.x_per_layer, self.y_per_layer = xo, yo
        # per-layer inputs and outputs, contiguous so one copy moves a whole step
        self.x_all = torch.empty((layers, batch, xo), dtype=torch.float16, device=device)
        self.y_all = torch.empty((layers, batch, yo), dtype=torch.float16, device=device)
        self.ws = None
        if tc24:  # zero-filled once; every call leaves it zero-filled
            need = max(nm.nm_spmm24_workspace_bytes(r, c, batch) for _, r, c in mats)
            self.ws = torch.zeros(need, dtype=torch.uint8, device=device)
        if batch > 1:
            need = 0 if tc24 else max(nm.nm_spmm_workspace_bytes(r, c, batch) for _, r, c in mats)
            if need:
                self.ws = torch.empty(need, dtype=torch.uint8, device=device)
            self.dense_out = [torch.empty((batch, r), dtype=torch.float16, device=device)
                              for _, r, _ in mats]

    def fill_x(self, xs):
        """xs[i]: [batch][cols] (or [cols]) activations of matrix i, reused by every layer."""
        for i, x in enumerate(xs):
            self.x_all[:, :, self.x_off[i]:self.x_off[i] + x.shape[-1]] = x

    def x(self, layer, i):
        _, rows, cols = self.mats[i]
        v = self.x_all[layer, :, self.x_off[i]:self.x_off[i] + cols]
        return v[0] if self.batch == 1 else v

    def y(self, layer, i):
        _, rows, cols = self.mats[i]
        v = self.y_all[layer, :, self.y_off[i]:self.y_off[i] + rows]
        return v[0] if self.batch == 1 else v

    def call_sparse(self, v, m, l, i):
        if self.tc24:
            X = self.x(l, i)
            Y = self.y(l, i)
            self.nm.nm_spmm24(v, m, X.view(self.batch, -1), Y=Y.view(self.batch, -1),
                              workspace=self.ws, flags=self.flags)
        elif self.swiglu[i]:
            y = self.y(l, i)
            self.nm.nm_spmv_swiglu(v, m, self.x(l, i), h=y[: y.numel() // 2], flags=self.flags)
        elif self.batch == 1:
            self.nm.nm_spmv(v, m, self.x(l, i), y=self.y(l, i), flags=self.flags)
        else:
            self.nm.nm_spmm(v, m, self.x(l, i), Y=self.y(l, i), workspace=self.ws,
                            flags=self.flags)

    def run_sparse(self, slots):
        for l in range(self.layers):
            slot = slots[l % len(slots)]
            for i, (v, m) in enumerate(slot):
                self.call_sparse(v, m, l, i)

    def run_dense(self, slots):
        import torch
        nm = self.nm
        for l in range(self.layers):
            slot = slots[l % len(slots)]
            for i, W in enumerate(slot):
                if self.batch == 1:
                    nm.dense_gemv(W, self.x(l, i), y=self.y(l, i), flags=self.flags)
                else:
                    torch.mm(self.x(l, i), W.t(), out=self.dense_out[i])

    def run_cublas(self, slots):
        """The batch-one sanity line: cuBLAS (torch.mm, a GEMV at one token)
        on the same dense slots, x as a one-row matrix."""
        import torch
        for l in range(self.layers):
            slot = slots[l % len(slots)]
            for i, W in enumerate(slot):
                torch.mm(self.x(l, i).view(1, -1), W.t(), out=self.y(l, i).view(1, -1))

    def bytes_sparse(self):
        B = self.batch
        # a fused SwiGLU call writes rows/2 outputs instead of rows
        return self.layers * sum(sparse_bytes(r, c) + (B - 1) * 2 * (r + c) - (r if f else 0)
                                 for (_, r, c), f in zip(self.mats, self.swiglu))

    def bytes_dense(self):
        B = self.batch
        return self.layers * sum(dense_bytes(r, c) + (B - 1) * 2 * (r + c) for _, r, c in self.mats)

    def calls(self):
        return self.layers * len(self.mats)

    def launches(self):
        """Kernels per step: one per call, plus the slice-combining kernel of
        every nm_spmm call whose rows are cut into column slices."""
        if self.tc24:
            return self.calls()
        if self.batch == 1:
            return self.calls()
        extra = sum(1 for _, r, c in self.mats
                    if self.nm.nm_spmm_workspace_bytes(r, c, self.batch) > 0)
        return self.layers * (len(self.mats) + extra)


def time_graph(fn, steps, warmup, stream, clock=None, seconds=None):
    """Capture fn() in a CUDA graph, replay `warmup` times, then time `steps`
    replays with CUDA events on `stream` (steps None: as many as fill about
    `seconds`, from a 3-replay estimate).  Returns per-step ms and total s."""
    import torch
    with torch.cuda.stream(stream):
        fn()  # eager once: plan caches and function attributes before capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        fn()
    with torch.cuda.stream(stream):
        for _ in range(warmup):
            g.replay()
    torch.cuda.synchronize()
    if steps is None:
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(3):
                g.replay()
            e1.record(stream)
        torch.cuda.synchronize()
        est = e0.elapsed_time(e1) / 3e3
        steps = int(min(2000, max(5, (seconds or 0.5) / max(est, 1e-6))))
    barrier()
    torch.cuda.synchronize()
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    if clock:
        clock.start()
    with torch.cuda.stream(stream):
        ev[0].record(stream)
        for k in range(steps):
            g.replay()
            ev[k + 1].record(stream)
    torch.cuda.synchronize()
    if clock:
        clock.stop()
    barrier()
    per = [ev[k].elapsed_time(ev[k + 1]) for k in range(steps)]
    total = ev[0].elapsed_time(ev[steps]) / 1e3
    del g
    return per, total


def time_per_matrix(step, slots, stream, reps):
    """µs per call of each matrix: a CUDA graph of `step.layers` calls of that
    matrix alone (cycling the slots, so every call streams from HBM), timed
    with CUDA events over `reps` replays after warm-up."""
    out = {}
    for i in range(len(step.mats)):
        def fn(i=i):
            for l in range(step.layers):
                v, m = slots[l % len(slots)][i]
                step.call_sparse(v, m, l, i)
        per, total = time_graph(fn, reps, 3, stream)
        out[i] = [t * 1e3 / step.layers for t in per]  # us per call, per replay
    return out


# The other decode-layer workloads the headline line also reports (the
# pattern sweep under all four patterns, the 32B layer under 2:4 and 16:32).
SIDE_PATTERNS = {"single_4096": [(2, 4)], "llama31_8b_layer": [(2, 4)],
                 "pattern_sweep": PATTERNS, "qwen3_32b_layer": [(2, 4), (16, 32)],
                 "llama33_70b_layer": PATTERNS}


def spmv_kernel_label(nm, rows, cols, batch=1):
    """Which kernel and plan the library runs for one nm_spmv (batch one) or
    nm_spmm (2..8 tokens) call."""
    if batch > 1:
        ws = nm.nm_spmm_workspace_bytes(rows, cols, batch)
        slices = ws // (batch * rows * 4) if ws else 1
        kern = "spmm_full_kernel" if cols % 1024 == 0 else "spmm_kernel"
        return (f"nm_spmm: {kern} (default plan, {slices} column slice"
                f"{'s + spmm_combine_kernel' if slices > 1 else ''})")
    v, g, w = nm.nm_spmv_plan(rows, cols)
    kern = "spmv_full_kernel" if cols % 1024 == 0 else "spmv_kernel"
    return f"nm_spmv: {kern} (nm_spmv plan: variant {v}, {w} warps x {g} blocks)"


def time_dense_lines(step, dslots, stream, args, clock):
    """dense_gemv and cuBLAS on the same dense slots: (ms per step) each."""
    dper, dtotal = time_graph(lambda: step.run_dense(dslots), None, args.warmup, stream,
                              clock=clock, seconds=args.side_seconds)
    cper, ctotal = time_graph(lambda: step.run_cublas(dslots), None, args.warmup, stream,
                              clock=clock, seconds=args.side_seconds)
    return dtotal / len(dper) * 1e3, ctotal / len(cper) * 1e3


def measure_side(nm, wname, device, stream, args, peak, clock):
    """One more decode-layer workload, batch one: the whole step through
    nm_spmv for each of its patterns, dense_gemv and cuBLAS on the same shapes,
    and the µs per call of every matrix (graphs of one matrix, CUDA events)."""
    import torch
    mats, layers = WORKLOADS[wname], LAYERS[wname]
    dense, xs = make_dense(mats, device, 1)
    step = Step(nm, mats, layers, device)
    step.fill_x(xs)
    step_bytes = step.bytes_sparse()
    out = {"shapes": ", ".join(f"{n} {r}x{c}" for n, r, c in mats), "layers": layers,
           "physical_slots": args.slots, "patterns": {}}
    per_call = None
    for pat in SIDE_PATTERNS[wname]:
        slots = pack_slots(nm, dense, pat, args.slots)
        per, total = time_graph(lambda: step.run_sparse(slots), None, args.warmup, stream,
                                clock=clock, seconds=args.side_seconds)
        ms = total / len(per) * 1e3
        out["patterns"][f"{pat[0]}:{pat[1]}"] = {"ms_per_step": round(ms, 4),
                                                 "GB_s": round(step_bytes / ms / 1e6, 1)}
        if per_call is None:
            per_call = time_per_matrix(step, slots, stream, 10)
        del slots
        torch.cuda.empty_cache()
    dslots = dense_slots(dense, args.dense_slots)
    d_ms, c_ms = time_dense_lines(step, dslots, stream, args, clock)
    del dslots, dense
    torch.cuda.empty_cache()
    head = out["patterns"]["2:4"]
    best_dense = min(d_ms, c_ms)
    out.update({
        "GB_s": head["GB_s"], "frac_of_measured_peak": round(head["GB_s"] / peak, 4),
        "ms_per_step": head["ms_per_step"],
        "dense_gemv": {"ms_per_step": round(d_ms, 4),
                       "GB_s": round(step.bytes_dense() / d_ms / 1e6, 1)},
        "cublas": {"ms_per_step": round(c_ms, 4),
                   "GB_s": round(step.bytes_dense() / c_ms / 1e6, 1),
                   "kernel": "torch.mm (cuBLAS) on the dense weights, one token"},
        "speedup_vs_dense": round(best_dense / head["ms_per_step"], 4),
        "speedup_vs_dense_basis": "the faster of dense_gemv and cuBLAS",
        "speedup_ideal": round(step.bytes_dense() / step_bytes, 4),
    })
    for k, v in out["patterns"].items():
        v["speedup_vs_dense"] = round(best_dense / v["ms_per_step"], 4)
    if len(out["patterns"]) > 1:
        g = [v["GB_s"] for v in out["patterns"].values()]
        out["pattern_spread"] = round((max(g) - min(g)) / statistics.median(g), 4)
    out["us_per_call"] = {}
    for i, (name, rows, cols) in enumerate(mats):
        mu = statistics.median(per_call[i])
        out["us_per_call"][name] = {"shape": f"{rows}x{cols}", "us_per_call": round(mu, 2),
                                    "GB_s": round(sparse_bytes(rows, cols) / mu / 1e3, 1),
                                    "frac_of_measured_peak":
                                        round(sparse_bytes(rows, cols) / mu / 1e3 / peak, 4)}
    return out


SMALL_BATCHES = (2, 4, 6, 8)


def measure_small_batches(nm, mats, layers, slots, dslots, device, stream, args, peak, clock,
                          tc24=False):
    """The headline workload's whole step at 2..8 tokens: nm_spmm on the packed
    slots against cuBLAS (torch.mm) at the same batch on the dense slots,
    graphs of the step, CUDA events (about args.side_seconds each); with
    tc24 (2:4 slots) also nm_spmm24 on the same slots."""
    out = {}
    for B in SMALL_BATCHES:
        step = Step(nm, mats, layers, device, batch=B)
        step.fill_x(make_xs(mats, device, B))
        per, total = time_graph(lambda: step.run_sparse(slots), None, args.warmup, stream,
                                clock=clock, seconds=args.side_seconds)
        ms = total / len(per) * 1e3
        dper, dtotal = time_graph(lambda: step.run_dense(dslots), None, args.warmup, stream,
                                  clock=clock, seconds=args.side_seconds)
        d_ms = dtotal / len(dper) * 1e3
        gbs = step.bytes_sparse() / ms / 1e6
        dom = max(mats, key=lambda m: m[1] * m[2])
        out[str(B)] = {"ms_per_step": round(ms, 4), "GB_s": round(gbs, 1),
                       "frac_of_measured_peak": round(gbs / peak, 4),
                       "cublas_ms_per_step": round(d_ms, 4),
                       "speedup_vs_cublas": round(d_ms / ms, 4),
                       "gpu_launches": step.launches() * len(per),
                       "kernel": spmv_kernel_label(nm, dom[1], dom[2], B)}
        del step
        if tc24:
            # the same 2:4 step through nm_spmm24 (mma.sync on register-built tiles)
            step = Step(nm, mats, layers, device, batch=B, tc24=True)
            step.fill_x(make_xs(mats, device, B))
            per, total = time_graph(lambda: step.run_sparse(slots), None, args.warmup, stream,
                                    clock=clock, seconds=args.side_seconds)
            ms = total / len(per) * 1e3
            gbs = step.bytes_sparse() / ms / 1e6
            out[str(B)]["nm_spmm24"] = {
                "ms_per_step": round(ms, 4), "GB_s": round(gbs, 1),
                "frac_of_measured_peak": round(gbs / peak, 4),
                "speedup_vs_cublas": round(d_ms / ms, 4),
                "gpu_launches": step.launches() * len(per),
                "kernel": "spmm24_kernel"}
            del step
    return out


PREFILL_SUMMARY_TOKENS = (64, 256)


def measure_prefill_summary(nm, mats, slots, dslots, device, stream, args, clock):
    """One decoder layer's four projections at 64 and 256 tokens through
    nm_spmm_prefill_ws (the library's plan: token tile, K slices) against
    cuBLAS fp16 GEMM (torch.mm) on the dense weights: dense-equivalent TFLOP/s
    (2 rows cols T per call), two layers per replay over two slots each,
    about args.side_seconds of replays per measurement."""
    import torch
    import synth
    out = {}
    for T in PREFILL_SUMMARY_TOKENS:
        X, Y, ws = [], [], []
        for mi, (_, rows, cols) in enumerate(mats):
            h = torch.empty((T, cols), dtype=torch.int16, pin_memory=True)
            synth.normal_f16_into(h.data_ptr(), T * cols, 0, synth.stream_id(4, mi, T),
                                  synth.X_SIGMA)
            X.append(h.to(device).view(torch.float16))
            Y.append(torch.empty((T, rows), dtype=torch.float16, device=device))
            b = nm.nm_spmm_prefill_workspace_bytes(rows, cols, T)
            ws.append(torch.empty(b, dtype=torch.uint8, device=device) if b else None)

        def sparse():
            for l in range(2):
                for i, (v, m) in enumerate(slots[l % len(slots)]):
                    nm.nm_spmm_prefill(v, m, X[i], Y=Y[i], workspace=ws[i])

        def dense():
            for l in range(2):
                for i, W in enumerate(dslots[l % len(dslots)]):
                    torch.mm(X[i], W.t(), out=Y[i])

        flops = 2 * sum(2.0 * r * c * T for _, r, c in mats)  # two layers per replay
        per, total = time_graph(sparse, None, args.warmup, stream, clock=clock,
                                seconds=args.side_seconds)
        s_ms = total / len(per) * 1e3
        dper, dtotal = time_graph(dense, None, args.warmup, stream, clock=clock,
                                  seconds=args.side_seconds)
        d_ms = dtotal / len(dper) * 1e3
        plans = {n: list(nm.nm_spmm_prefill_plan(r, c, T)[1:]) for n, r, c in mats}
        out[str(T)] = {"TFLOP_s": round(flops / s_ms / 1e9, 1),
                       "cublas_TFLOP_s": round(flops / d_ms / 1e9, 1),
                       "vs_cublas": round(d_ms / s_ms, 4),
                       "ms_per_layer": round(s_ms / 2, 4),
                       "plan_k_slices_tile_tokens": plans}
        del X, Y, ws
    return out


def run_gpu(args):
    import torch
    import sparse_spmv_memory_gb300 as nm

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    nm.lib()
    mats = WORKLOADS[args.workload]
    layers = args.layers
    stream = torch.cuda.Stream(device)
    peak, peak_kind = hbm_peak()

    t_setup = time.time()
    dense, xs = make_dense(mats, device, args.batch)
    step = Step(nm, mats, layers, device, flags=None if args.flags < 0 else args.flags,
                batch=args.batch, swiglu=args.swiglu)
    step.fill_x(xs)
    setup_s = time.time() - t_setup

    head = tuple(int(t) for t in args.pattern.split(":"))
    patterns = [head] + ([p for p in PATTERNS if p != head] if args.patterns else [])
    results = {}
    per_launch = None
    cs = ClockSampler(local).__enter__()
    try:
        for pat in patterns:
            slots = pack_slots(nm, dense, pat, args.slots)
            fn = lambda: step.run_sparse(slots)
            if pat == head:
                per, total = time_graph(fn, args.steps, args.warmup, stream, clock=cs)
                per_launch = time_per_matrix(step, slots, stream, 10)
            else:
                per, total = time_graph(fn, max(3, args.steps // 4), max(3, args.warmup), stream,
                                        clock=cs)
            results[pat] = (per, total, len(per))
            del slots, fn
            torch.cuda.empty_cache()

        # end to end through the public calls: pinned host x in, y out, every step
        slots = pack_slots(nm, dense, head, args.slots)
        x_host = torch.empty(step.x_all.shape, dtype=torch.float16, pin_memory=True)
        x_host.copy_(step.x_all)
        y_host = torch.empty(step.y_all.shape, dtype=torch.float16, pin_memory=True)
        with torch.cuda.stream(stream):
            for _ in range(args.warmup):
                step.x_all.copy_(x_host, non_blocking=True)
                step.run_sparse(slots)
                y_host.copy_(step.y_all, non_blocking=True)
        torch.cuda.synchronize()
        barrier()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        t0 = time.perf_counter()
        with torch.cuda.stream(stream):
            e0.record(stream)
            for _ in range(args.steps):
                step.x_all.copy_(x_host, non_blocking=True)
                step.run_sparse(slots)
                y_host.copy_(step.y_all, non_blocking=True)
            e1.record(stream)
        torch.cuda.synchronize()
        e2e_wall = time.perf_counter() - t0
        e2e_s = e0.elapsed_time(e1) / 1e3
        barrier()

        # dense baselines on the same shapes and rotation scheme: the library's own
        # dense_gemv, and cuBLAS as the sanity line (batch one)
        dense_res = cublas_ms = None
        small, prefill = {}, {}
        if args.dense:
            dslots = dense_slots(dense, args.dense_slots)
            dper, dtotal = time_graph(lambda: step.run_dense(dslots), max(3, args.steps // 2),
                                      args.warmup, stream, clock=cs)
            dense_res = (dper, dtotal, len(dper))
            if args.batch == 1:
                cper, ctotal = time_graph(lambda: step.run_cublas(dslots), max(3, args.steps // 2),
                                          args.warmup, stream, clock=cs)
                cublas_ms = ctotal / len(cper) * 1e3
            # the same step at 2..8 tokens (nm_spmm against cuBLAS at that batch)
            if args.small_batch and args.batch == 1 and not args.swiglu:
                small = measure_small_batches(nm, mats, layers, slots, dslots, device, stream,
                                              args, peak, cs, tc24=tuple(head) == (2, 4))
            # the same layer's prefill on the tensor cores (nm_spmm_prefill_ws)
            if args.prefill_summary and args.batch == 1 and not args.swiglu:
                prefill = measure_prefill_summary(nm, mats, slots, dslots, device, stream,
                                                  args, cs)
            del dslots
            torch.cuda.empty_cache()
        # the same step with the SwiGLU activation fused into the gate+up call
        fused = {}
        if args.batch == 1 and not args.swiglu and any(n == "gate_up" for n, _, _ in mats):
            sw = Step(nm, mats, layers, device, swiglu=True)
            sw.fill_x(xs)
            fper, ftotal = time_graph(lambda: sw.run_sparse(slots), None, args.warmup, stream,
                                      clock=cs, seconds=args.side_seconds)
            f_ms = ftotal / len(fper) * 1e3
            u_ms = results[head][1] / results[head][2] * 1e3
            fused = {"ms_per_step": round(f_ms, 4),
                     "GB_s": round(sw.bytes_sparse() / f_ms / 1e6, 1),
                     "unfused_ms_per_step": round(u_ms, 4),
                     "time_vs_unfused": round(f_ms / u_ms, 4),
                     "gate_up": "nm_spmv_swiglu: h = silu(gate) * up written once, rows/2 outputs"}
            del sw
        del slots, dense
        torch.cuda.empty_cache()

        # the other decode-layer workloads, batch one, on the same line
        side = {}
        if args.side and args.batch == 1 and not args.swiglu:
            for wname in WORKLOADS:
                if wname != args.workload:
                    side[wname] = measure_side(nm, wname, device, stream, args, peak, cs)
    finally:
        cs.__exit__(None, None, None)
    clocks = cs.summary()

    # ---- assemble ------------------------------------------------------------
    per, total, k = results[head]
    step_bytes = step.bytes_sparse()
    units, secs = aggregate(step_bytes * k, total)
    gbs = units / secs / 1e9
    med_ms = statistics.median(per)
    out = {
        "metric": batch_metric(args.batch),
        "value": round(gbs, 1),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": k,
        "warmup": args.warmup,
        "ms_per_step": round(secs / k * 1e3, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "fp16 in/out, fp32 accumulate",
        "data": "synthetic (seeded N(0,0.02) fp16 weights, top-N |w| per M-group; N(0,1) fp16 x)",
        "config": {
            "workload": (f"{args.workload} x{layers} layers, batch {args.batch}, "
                         + ", ".join(f"{n} {r}x{c}" for n, r, c in mats)),
            "pattern": f"{head[0]}:{head[1]}",
            "calls_per_step": step.calls(),
            "physical_slots": args.slots,
            "l2_defeat": (f"rotating set of {args.slots} packed layer slots = "
                          f"{args.slots * step_bytes / layers / 1e9:.1f} GB > L2 (129 MB)"),
            "parallelism": f"replicas x{world}",
            "launch_flags": "library default (programmatic dependent launch)" if args.flags < 0 else args.flags,
            "gate_up": ("nm_spmv_swiglu (SwiGLU fused)" if args.swiglu and args.batch == 1
                        else ("nm_spmv" if args.batch == 1 else "nm_spmm")),
        },
        "step_ms": {"median": round(med_ms, 4), "p10": round(float(np.percentile(per, 10)), 4),
                    "p90": round(float(np.percentile(per, 90)), 4)},
        "pct_peak": {"of_measured" if peak_kind == "measured" else "of_fallback":
                     round(gbs / world / peak, 4), "of_nominal_7900": round(gbs / world / NOMINAL_HBM_GBS, 4)},
        "gpu_launches": step.launches() * k,
    }
    # per-matrix µs per call (graphs of one matrix, CUDA events)
    calls = {}
    for i, (name, rows, cols) in enumerate(mats):
        us = per_launch.get(i, [])
        if not us:
            continue
        mu = statistics.median(us)
        calls[name] = {"shape": f"{rows}x{cols}", "us_per_call": round(mu, 2),
                       "GB_s": round(sparse_bytes(rows, cols) / mu / 1e3, 1),
                       "frac_of_measured_peak": round(sparse_bytes(rows, cols) / mu / 1e3 / peak, 4),
                       "bytes": sparse_bytes(rows, cols)}
    out["us_per_call"] = calls
    # The dominant kernel is the launch that moves the most bytes (gate+up on
    # the decode layers): its algorithmic bytes per launch over its average
    # launch duration, from CUDA events around a graph of back-to-back
    # launches of that matrix alone on the launching stream.
    di, dom = max(enumerate(mats), key=lambda im: sparse_bytes(im[1][1], im[1][2]))
    dom_bytes = sparse_bytes(dom[1], dom[2])
    dom_us = statistics.median(per_launch[di])
    achieved = dom_bytes / dom_us / 1e3
    traffic = (ncu_traffic(f"{dom[1]}x{dom[2]}") if args.batch == 1 else
               ncu_traffic(f"{dom[1]}x{dom[2]}x{args.batch}", "nm_spmm_traffic.json", SPMM_SOURCES))
    out["roofline"] = {
        "bound": "hbm", "kernel": spmv_kernel_label(nm, dom[1], dom[2], args.batch),
        "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
        "frac": round(achieved / peak, 4),
        "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)" if peak_kind == "measured" else "fallback 6.8 TB/s",
        "traffic": traffic,
        "traffic_shape": f"{dom[1]}x{dom[2]}",
        "traffic_algorithmic": dom_bytes,
        "achieved_basis": (f"algorithmic bytes of one {dom[1]}x{dom[2]} launch ({dom_bytes} B: "
                           "values + masks + x + y) / its average launch duration "
                           f"({dom_us:.2f} us, CUDA events around a graph of {layers} "
                           "back-to-back launches over the rotating slots)"),
        "step_frac": round(gbs / world / peak, 4),
        "step_frac_basis": ("the whole step's algorithmic bytes / the step's CUDA-event time, "
                            "launch gaps and the smaller matrices included"),
    }
    out["patterns"] = {
        f"{p[0]}:{p[1]}": {"ms_per_step": round(results[p][1] / results[p][2] * 1e3, 4),
                           "GB_s": round(step_bytes * results[p][2] / results[p][1] / 1e9, 1),
                           "us_per_call_avg": round(results[p][1] / results[p][2] / step.calls() * 1e6, 2),
                           "masks_bytes_per_step": layers * sum(r * c // 8 for _, r, c in mats)}
        for p in patterns}
    if dense_res:
        dper, dtotal, dk = dense_res
        d_ms = dtotal / dk * 1e3
        out["dense"] = {"ms_per_step": round(d_ms, 4),
                        "GB_s": round(step.bytes_dense() * dk / dtotal / 1e9, 1),
                        "physical_slots": args.dense_slots,
                        "kernel": "dense_gemv" if args.batch == 1 else "cuBLAS via torch.mm"}
        best = d_ms
        if cublas_ms is not None:
            out["cublas"] = {"ms_per_step": round(cublas_ms, 4),
                             "GB_s": round(step.bytes_dense() / cublas_ms / 1e6, 1),
                             "kernel": "torch.mm (cuBLAS) on the dense weights, one token"}
            best = min(d_ms, cublas_ms)
            out["speedup_vs_cublas"] = round(cublas_ms / (total / k * 1e3), 4)
        out["speedup_vs_dense"] = round(best / (total / k * 1e3), 4)
        out["speedup_vs_dense_basis"] = ("the faster of dense_gemv and cuBLAS"
                                         if cublas_ms is not None else
                                         ("dense_gemv" if args.batch == 1 else "cuBLAS (torch.mm)"))
        out["speedup_ideal"] = round(step.bytes_dense() / step_bytes, 4)
        for p in patterns:
            out["patterns"][f"{p[0]}:{p[1]}"]["speedup_vs_dense"] = round(
                best / (results[p][1] / results[p][2] * 1e3), 4)
    if side:
        out["workloads"] = side
    if small:
        out["small_batch"] = small
    if fused:
        out["swiglu_fused"] = fused
    if prefill:
        out["prefill"] = prefill
        out["prefill_wait_timeouts"] = nm.nm_wait_timeouts()
    xb = step.x_all.numel() * 2
    yb = step.y_all.numel() * 2
    e_units, e_secs = aggregate(step_bytes * args.steps, e2e_s)
    out["e2e"] = {"value": round(e_units / e_secs / 1e9, 1), "unit": "GB/s",
                  "h2d_bytes_per_step": xb, "d2h_bytes_per_step": yb,
                  "ms_per_step": round(e_secs / args.steps * 1e3, 4),
                  "host_wall_ms_per_step": round(e2e_wall / args.steps * 1e3, 4),
                  "path": (f"Python binding -> C ABI {'nm_spmv' if args.batch == 1 else 'nm_spmm'} "
                           "per call, eager, pinned host x/y")}
    out["clocks"] = clocks
    out["setup_s"] = round(setup_s, 1)

    if rank == 0 and world == 1 and args.cpu and args.batch == 1:
        _, nb, dt, desc = oracle_sample(mats, head, args.cpu_seconds)
        out["cpu_baseline"] = {**host_cpu(), "value": round(nb / dt / 1e9, 4), "unit": "GB/s", "cores": 1,
                               "kind": "oracle", "sample": desc, "seconds": round(dt, 2)}
    return out


def host_cpu():
    """The host the oracle runs on: logical CPUs and a model string (the
    model name on x86; architecture, implementer and part codes on Arm)."""
    fields = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                if ":" in line:
                    k, v = line.split(":", 1)
                    fields.setdefault(k.strip().lower(), v.strip())
    except OSError:
        pass
    model = fields.get("model name")
    if not model and "cpu part" in fields:
        model = (f"{os.uname().machine} (implementer {fields.get('cpu implementer', '?')}, "
                 f"part {fields['cpu part']})")
    return {"host_logical_cpus": os.cpu_count(), "host_cpu": model or os.uname().machine}


def prefill_flops(mats, T):
    """Dense-equivalent flops of one pass of the matrices over T tokens."""
    return sum(2.0 * r * c * T for _, r, c in mats)


def oracle_prefill_rate(mats, pattern, seconds: float):
    """The oracle on a bounded sample: the sampled rows of every matrix for a
    handful of tokens; returns (dense-equivalent TFLOP/s, description, s)."""
    rows_per, _, _, _ = oracle_sample(mats, pattern, seconds / 4)
    orc, packed = oracle_pack_sample(mats, pattern, rows_per)
    import synth
    tokens = 4
    xs = [[synth.activations(cols, 0, synth.stream_id(3, mi, t)) for t in range(tokens)]
          for mi, (_, _, cols, _, _) in enumerate(packed)]
    t0 = time.perf_counter()
    fl = 0.0
    for mi, (v, m, cols, _, n) in enumerate(packed):
        for t in range(tokens):
            orc.spmv_f64(v, m, cols, xs[mi][t])
            fl += 2.0 * n * cols
    dt = time.perf_counter() - t0
    desc = (f"first {rows_per} rows of each of the {len(mats)} matrices x {tokens} tokens, "
            f"{pattern[0]}:{pattern[1]}, oracle unpack + double matvec per token, 1 thread")
    return fl / dt / 1e12, desc, dt


def run_prefill(args):
    """Prefill regime: Y = W X for T tokens per call, every matrix of the
    workload, ``args.prefill_layers`` logical layers per step cycling two
    packed slots (the call is compute-bound, so L2 residency is immaterial)."""
    import torch
    import synth
    import sparse_spmv_memory_gb300 as nm

    world, rank, local = dist_env()
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    nm.lib()
    nm.nm_wait_timeouts(reset=True)
    mats = WORKLOADS[args.workload]
    T, layers = args.prefill, args.prefill_layers
    stream = torch.cuda.Stream(device)
    head = tuple(int(t) for t in args.pattern.split(":"))
    dense, _ = make_dense(mats, device, 1)
    X = []
    for mi, (_, rows, cols) in enumerate(mats):
        h = torch.empty((T, cols), dtype=torch.int16, pin_memory=True)
        synth.normal_f16_into(h.data_ptr(), T * cols, 0, synth.stream_id(4, mi, T), synth.X_SIGMA)
        X.append(h.to(device).view(torch.float16))
    Y = [torch.empty((T, r), dtype=torch.float16, device=device) for _, r, _ in mats]
    slots = pack_slots(nm, dense, head, 2)
    # the library's plan per matrix: a K split (fp32 partials in a workspace,
    # then a combine launch) where few row tiles would leave SMs idle
    ws_bytes = [nm.nm_spmm_prefill_workspace_bytes(r, c, T) for _, r, c in mats]
    ws = [torch.empty(b, dtype=torch.uint8, device=device) if b else None for b in ws_bytes]
    k_slices = {n: (b // (4 * T * r) if b else 1) for (n, r, _), b in zip(mats, ws_bytes)}
    tile_tokens = {n: nm.nm_spmm_prefill_plan(r, c, T)[2] for n, r, c in mats}

    def run_sparse():
        for l in range(layers):
            for i, (v, m) in enumerate(slots[l % 2]):
                nm.nm_spmm_prefill(v, m, X[i], Y=Y[i], workspace=ws[i])

    with ClockSampler(local) as cs:
        per, total = time_graph(run_sparse, args.steps, args.warmup, stream, clock=cs)
    clocks = cs.summary()
    k = len(per)
    per_matrix = {}
    # At least 8 calls per replay: one short launch per replay would time the
    # host's replay loop rather than the kernel.
    calls = max(layers, 8)
    for i, (name, rows, cols) in enumerate(mats):
        def one(i=i):
            for l in range(calls):
                v, m = slots[l % 2][i]
                nm.nm_spmm_prefill(v, m, X[i], Y=Y[i], workspace=ws[i])
        p1, t1 = time_graph(one, 5, 3, stream)
        us = statistics.median(p1) * 1e3 / calls
        per_matrix[name] = {"shape": f"{rows}x{cols}", "tokens": T, "us_per_call": round(us, 1),
                            "TFLOP_s": round(2.0 * rows * cols * T / us / 1e6, 1)}

    # end to end: pinned host X in and Y out every step, eager public calls
    x_host = [x.cpu().pin_memory() for x in X]
    y_host = [torch.empty(y.shape, dtype=torch.float16, pin_memory=True) for y in Y]
    with torch.cuda.stream(stream):
        for _ in range(args.warmup):
            for i in range(len(mats)):
                X[i].copy_(x_host[i], non_blocking=True)
            run_sparse()
            for i in range(len(mats)):
                y_host[i].copy_(Y[i], non_blocking=True)
    torch.cuda.synchronize()
    barrier()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        e0.record(stream)
        for _ in range(args.steps):
            for i in range(len(mats)):
                X[i].copy_(x_host[i], non_blocking=True)
            run_sparse()
            for i in range(len(mats)):
                y_host[i].copy_(Y[i], non_blocking=True)
        e1.record(stream)
    torch.cuda.synchronize()
    e2e_s = e0.elapsed_time(e1) / 1e3
    timeouts = nm.nm_wait_timeouts()
    del slots
    torch.cuda.empty_cache()

    # cuBLAS on the dense weights, same tokens and layer count
    Yd = [torch.empty_like(y) for y in Y]

    def run_dense():
        for l in range(layers):
            for i, W in enumerate(dense):
                torch.mm(X[i], W.t(), out=Yd[i])

    dper, dtotal = time_graph(run_dense, max(3, args.steps // 2), args.warmup, stream)

    step_flops = layers * prefill_flops(mats, T)
    units, secs = aggregate(step_flops * k, total)
    tf = units / secs / 1e12
    peak, peak_kind = tensor_peak(total)
    d_tf = step_flops * len(dper) / dtotal / 1e12
    dom = max(mats, key=lambda m: m[1] * m[2])
    out = {
        "metric": PREFILL_METRIC, "value": round(tf, 1), "unit": "TFLOP/s", "n_gpus": world,
        "steps": k, "warmup": args.warmup, "ms_per_step": round(secs / k * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp16 in/out, fp32 accumulate (tensor cores, kind::f16)",
        "data": "synthetic (seeded N(0,0.02) fp16 weights, top-N |w| per M-group; N(0,1) fp16 X)",
        "config": {
            "workload": (f"{args.workload} x{layers} layers, prefill {T} tokens, "
                         + ", ".join(f"{n} {r}x{c}" for n, r, c in mats)),
            "pattern": f"{head[0]}:{head[1]}", "calls_per_step": layers * len(mats),
            "physical_slots": 2,
            "l2_defeat": (f"inputs larger than L2: 2 packed layer slots of "
                          f"{sum(sparse_bytes(r, c) for _, r, c in mats) / 1e9:.2f} GB each "
                          "(129 MB L2) cycled over the layers"),
            "parallelism": f"replicas x{world}", "kernel_variant": "library default for T",
            "k_slices": k_slices, "tile_tokens": tile_tokens,
        },
        "gpu_launches": layers * k * sum(1 if z == 1 else 2 for z in k_slices.values()),
        "us_per_call": per_matrix,
        "cublas": {"TFLOP_s": round(d_tf, 1), "ms_per_step": round(dtotal / len(dper) * 1e3, 3),
                   "kernel": "torch.mm (cuBLAS) fp16 on the dense weights"},
        "speedup_vs_dense": round(tf / d_tf, 4),
        "roofline": {"bound": "tensor", "kernel": "nm_spmm_prefill (spmm_tc_kernel)",
                     "achieved": round(tf, 1), "peak": peak, "unit": "TFLOP/s",
                     "frac": round(tf / peak, 4), "peak_kind": peak_kind,
                     "traffic": ncu_traffic(f"{dom[1]}x{dom[2]}x{T}", "nm_spmm_prefill_traffic.json",
                                            PREFILL_SOURCES),
                     "traffic_shape": f"{dom[1]}x{dom[2]}, {T} tokens",
                     "achieved_basis": ("dense-equivalent MMA flops of the timed region's launches "
                                        "/ the region's CUDA-event device time (a lower bound); "
                                        "fp16 and bf16 share the nominal dense rate"),
                     "dominant_shape": f"{dom[1]}x{dom[2]}"},
        "e2e": {"value": round(step_flops * args.steps / e2e_s / 1e12, 1), "unit": "TFLOP/s",
                "h2d_bytes_per_step": sum(x.numel() * 2 for x in X),
                "d2h_bytes_per_step": sum(y.numel() * 2 for y in Y),
                "ms_per_step": round(e2e_s / args.steps * 1e3, 3),
                "path": "Python binding -> C ABI nm_spmm_prefill_ws per call, eager, pinned host X/Y"},
        "clocks": clocks, "wait_timeouts": timeouts,
    }
    if rank == 0 and world == 1 and args.cpu:
        rate, desc, dt = oracle_prefill_rate(mats, head, args.cpu_seconds)
        out["cpu_baseline"] = {**host_cpu(), "value": round(rate, 6), "unit": "TFLOP/s", "cores": 1,
                               "kind": "oracle", "sample": desc, "seconds": round(dt, 2)}
    return out


def run_reference(args):
    """The reference arm: the plain CPU oracle, timed as it stands."""
    world, rank, _ = dist_env()
    if rank != 0:
        return None
    mats = WORKLOADS[args.workload]
    head = tuple(int(t) for t in args.pattern.split(":"))
    if args.prefill:
        secs = max(1.0, args.ref_seconds / 4)
        rate, desc, dt = oracle_prefill_rate(mats, head, secs)
        return {
            "impl": "reference", "metric": PREFILL_METRIC, "value": round(rate, 6),
            "unit": "TFLOP/s", "n_gpus": world, "steps": 1, "warmup": 0,
            "ms_per_step": round(dt * 1e3, 1), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
            "config": {"workload": f"{args.workload}, prefill {args.prefill} tokens, oracle sample",
                       "pattern": args.pattern},
            "cpu_baseline": {**host_cpu(), "kind": "oracle", "cores": 1, "sample": desc,
                             "value": round(rate, 6),
                             "unit": "TFLOP/s"},
            "e2e": {"value": round(rate, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                    "d2h_bytes_per_step": 0},
        }
    per_step = max(0.5, args.ref_seconds / max(1, args.steps + args.warmup))
    # the row sample is sized for one token; B tokens take B SpMVs of it
    rows_per, _, _, desc = oracle_sample(mats, head, per_step / args.batch)
    orc, packed = oracle_pack_sample(mats, head, rows_per, args.batch)
    if args.batch > 1:
        desc += f", {args.batch} tokens (one oracle SpMV per token)"
    step_bytes = sum(sparse_bytes(n, cols) for _, _, cols, _, n in packed)
    for _ in range(args.warmup):
        oracle_run(orc, packed)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_run(orc, packed)
    secs = time.perf_counter() - t0
    val = step_bytes * args.steps / secs / 1e9
    return {
        "impl": "reference", "metric": batch_metric(args.batch), "value": round(val, 4), "unit": "GB/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(secs / args.steps * 1e3, 3), "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)", "data": "synthetic",
        "config": {"workload": f"{args.workload}, batch {args.batch}, oracle sample",
                   "pattern": args.pattern},
        "cpu_baseline": {**host_cpu(), "kind": "oracle", "cores": 1, "sample": desc,
                         "value": round(val, 4),
                         "unit": "GB/s"},
        "e2e": {"value": round(val, 4), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def parse(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(WORKLOADS), default="llama33_70b_layer")
    ap.add_argument("--pattern", default="2:4")
    ap.add_argument("--swiglu", action="store_true",
                    help="run the gate+up projection as nm_spmv_swiglu (SwiGLU fused; "
                         "rows interleaved gate/up)")
    ap.add_argument("--batch", type=int, default=1,
                    help="tokens per step: 1 = nm_spmv (the headline); 2..8 = nm_spmm, with "
                         "cuBLAS (torch.mm) as the dense reference")
    ap.add_argument("--prefill", type=int, default=0,
                    help="tokens per call for the prefill regime (nm_spmm_prefill on the tensor "
                         "cores, cuBLAS fp16 GEMM as the dense reference); 0 = decode (default)")
    ap.add_argument("--prefill-layers", type=int, default=4,
                    help="logical layers per prefill step")
    ap.add_argument("--layers", type=int, default=None,
                    help="logical layers per step (default: the model's layer count)")
    ap.add_argument("--slots", type=int, default=16, help="physical sparse layer slots")
    ap.add_argument("--dense-slots", type=int, default=8)
    ap.add_argument("--no-dense", dest="dense", action="store_false")
    ap.add_argument("--no-patterns", dest="patterns", action="store_false")
    ap.add_argument("--no-cpu", dest="cpu", action="store_false")
    ap.add_argument("--no-prefill-summary", dest="prefill_summary", action="store_false",
                    help="skip the layer's prefill at 64 and 256 tokens (nm_spmm_prefill vs cuBLAS)")
    ap.add_argument("--no-small-batch", dest="small_batch", action="store_false",
                    help="skip the headline step at 2, 4, 6 and 8 tokens (nm_spmm vs cuBLAS)")
    ap.add_argument("--no-side", dest="side", action="store_false",
                    help="skip the other decode-layer workloads (reported under 'workloads')")
    ap.add_argument("--side-seconds", type=float, default=0.4,
                    help="timed seconds per measurement of each other workload")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--flags", type=int, default=-1,
                    help="launch flags for every call (default: the library's own, i.e. "
                         "programmatic dependent launch): 0 = plain launches, 1 = programmatic "
                         "dependent launch, 3 = also issue the first weight loads before the "
                         "dependency wait")
    ap.add_argument("--ref-seconds", type=float, default=60.0)
    a = ap.parse_args(argv)
    if not 1 <= a.batch <= 8:
        ap.error("--batch must be in 1..8")
    if a.prefill < 0 or (a.prefill and a.batch != 1):
        ap.error("--prefill takes a positive token count and no --batch")
    if a.layers is None:
        a.layers = LAYERS[a.workload]
    if a.warmup < 3:
        ap.error("--warmup must be >= 3")
    return a


def main(argv=None):
    args = parse(argv)
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if args.impl == "ours" else "gloo"
        if args.impl == "ours":
            import torch
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    if args.impl == "reference":
        out = run_reference(args)
    else:
        out = run_prefill(args) if args.prefill else run_gpu(args)
    if rank == 0 and out is not None:
        print(json.dumps(out), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
