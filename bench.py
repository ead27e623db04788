"""Benchmark of the block-sparse attention forward (one JSON line on stdout).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload I] [--impl reference]

A step is one ``bsa_forward`` over one batch of the workload (one kernel launch).
The default workload is 5 (B=1, H=32, L=65536, block 128, d 128, Sparse-Transformer
layout, causal diagonal): the largest of the five and one of the three the 55%-of-peak
target names.  ``value`` is active-block TFLOPS (4 * block^2 * d per active block per
batch entry) over the whole job, timed with CUDA events on the launching stream.
Under torchrun every rank runs its own replica of the workload (weak scaling) and the
slowest rank's time counts.

After the headline the forward is timed alone, by the same method, on the other
workloads of the 55% target (3 and 4 by default), reported under ``per_workload``, and
the backward (dQ, dK, dV) on workloads 3, 4 and 5 under ``backward``, and the top-k
token-gather attention workload under ``topk``.

``--impl reference`` times the fp64 CPU oracle instead, on bounded samples of the same
workload (query blocks drawn across the work list), one process per host core.
"""

from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "block-sparse attn fwd active-block TFLOPS and % of GB300 bf16 tensor peak"
L2_BYTES = 129 * 1024 * 1024
KERNEL_SOURCES = ["bsa_fwd_kernel.cuh", "bsa_ptx.cuh", "bsa_host.cpp", "bsa_internal.h"]


def kernel_sources_sha() -> str:
    """Hash of the kernel sources with comments and blank space removed, so that a
    comment edit keeps the recorded ncu counters attached to the code they measured."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "block_sparse_head_gb300", "csrc", name)) as f:
            text = f.read()
        text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
        text = re.sub(r"//[^\n]*", " ", text)
        h.update(" ".join(text.split()).encode())
    return h.hexdigest()[:16]


def measured_peaks() -> dict:
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"bf16_burst": d["bf16_tflops"], "bf16_sustained": d["bf16_tflops_sustained"],
                "hbm_gbs": d["hbm_gbs"], "source": "measured"}
    return {"bf16_burst": 1900.0, "bf16_sustained": 1700.0, "hbm_gbs": 6800.0,
            "source": "fallback"}


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on the
    current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"bsa_fwd_{workload_name}.md")
    if not os.path.exists(path):
        return None
    text = open(path).read()
    m_t = re.search(r"traffic_per_launch_bytes\s*=\s*([0-9.eE+]+)", text)
    m_h = re.search(r"kernel_sources_sha256\s*=\s*([0-9a-f]+)", text)
    if not m_t or not m_h or m_h.group(1) != kernel_sources_sha():
        return None
    return float(m_t.group(1))


# ----------------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi clock/throttle sampling during the timed region."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.proc = None
        self.gpu = gpu_index
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={gpu_index}", f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self) -> dict:
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                smax.append(float(f[2]))
            except ValueError:
                continue
            for n, val in zip(names, f[5:9]):
                if val.lower().startswith("active"):
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax),
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ CPU oracle

_OP = {}  # oracle worker state
_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _op_init(tmp, shape, lay, scale, block, causal):
    import numpy as np

    for name in ("q", "k", "v"):
        _OP[name] = np.memmap(os.path.join(tmp, name), np.float32, "r", shape=shape)
    _OP["lay"], _OP["par"] = lay, (scale, block, causal)


def _op_task(items) -> int:
    """Oracle over a list of work items (b, h, i, nnz); returns their FLOPs."""
    import oracle

    scale, block, causal = _OP["par"]
    flops = 0
    for b, h, i, nnz in items:
        # mapped fp32 views; the oracle gathers the rows it needs and computes in fp64
        q, k, v = (_OP[n][b, h] for n in ("q", "k", "v"))
        oracle.query_block(q, k, v, _OP["lay"][h], scale, block, causal, i)
        flops += 4 * block * block * q.shape[1] * nnz
    return flops


class OraclePool:
    """The fp64 oracle, as it stands, over a pool of processes (one per host core).

    The inputs are written once to memory-mapped files that the workers map read only;
    work items are sampled across the whole work list (a seeded permutation), so the
    sample mixes long and short rows as the workload does."""

    def __init__(self, wl, q, k, v, lay, procs: int):
        import multiprocessing as mp
        import tempfile

        import numpy as np
        import torch

        import oracle

        self.tmp = tempfile.TemporaryDirectory(prefix="bsa_oracle_")
        for name, t in (("q", q), ("k", k), ("v", v)):  # bf16 -> fp32 is exact
            for b in range(t.shape[0]):
                with open(os.path.join(self.tmp.name, name), "ab") as f:
                    t[b].float().numpy().tofile(f)
        lay = np.ascontiguousarray(np.asarray(lay, dtype=np.int64))
        _, _, items = oracle.oracle_lut(lay, wl.B)
        perm = np.random.default_rng(0).permutation(len(items))
        self.items = [tuple(int(x) for x in items[t]) for t in perm]
        self.pos = 0
        self.procs = procs
        # One BLAS thread per worker: the variables must be set before a worker first
        # imports numpy (unpickling its arguments does), so they go in through the
        # environment the workers inherit.
        saved = {var: os.environ.get(var) for var in _BLAS_VARS}
        os.environ.update({var: "1" for var in _BLAS_VARS})
        try:
            self.pool = mp.get_context("spawn").Pool(
                procs, initializer=_op_init,
                initargs=(self.tmp.name, tuple(q.shape), lay, wl.scale, wl.block, wl.causal_diag))
        finally:
            for var, val in saved.items():
                if val is None:
                    os.environ.pop(var, None)
                else:
                    os.environ[var] = val
        self.pool.map(_op_task, [[]] * procs)  # start every worker before timing

    def take(self, n: int) -> list:
        out = [self.items[(self.pos + j) % len(self.items)] for j in range(n)]
        self.pos += n
        return out

    def run(self, n_items: int, per_task: int = 2):
        """Runs the next n_items sampled items; returns (FLOPs, seconds)."""
        items = self.take(n_items)
        tasks = [items[j:j + per_task] for j in range(0, len(items), per_task)]
        t0 = time.perf_counter()
        flops = sum(self.pool.map(_op_task, tasks, chunksize=1))
        return flops, time.perf_counter() - t0

    def close(self):
        self.pool.close()
        self.pool.join()
        self.tmp.cleanup()


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def cpu_baseline(wl, q, k, v, lay, budget_s: float) -> dict:
    """Oracle throughput on the host cores: rounds of 2 items per process until
    `budget_s` seconds of timed work."""
    procs = host_cores()
    op = OraclePool(wl, q, k, v, lay, procs)
    try:
        flops = secs = 0.0
        n = 0
        while secs < budget_s:
            f, t = op.run(2 * procs)
            flops, secs, n = flops + f, secs + t, n + 2 * procs
    finally:
        op.close()
    return {"tflops": flops / secs / 1e12, "items": n, "seconds": secs, "cores": procs}


# ------------------------------------------------------------------- GPU arm


def dist_setup():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(values, pg, device="cuda") -> list:
    """The slowest rank's value of each timing (ranks run weak-scaling replicas); the
    values themselves on one rank.  `pg` is torch.distributed or None."""
    if pg is None:
        return [float(x) for x in values]
    import torch

    t = torch.tensor([float(x) for x in values], device=device, dtype=torch.float64)
    pg.all_reduce(t, op=pg.ReduceOp.MAX)
    return [float(x) for x in t]


def job_tflops(world: int, flops_per_step: int, steps: int, ms: float) -> float:
    """Whole-job throughput: every rank does `steps` steps of `flops_per_step` in `ms`."""
    return world * flops_per_step * steps / (ms * 1e-3) / 1e12


def l2_note_for(wl) -> str:
    """How the timed region keeps the L2 from serving the inputs of the previous launch."""
    if 3 * wl.B * wl.H * wl.L * wl.d * 2 < 2 * L2_BYTES:
        return "L2 flushed between steps (256 MiB write, outside the events)"
    return "inputs larger than L2"


def workload_config(wl, l2_note: str, world: int) -> dict:
    return {"workload": f"{wl.name} (workload {wl.index})", "batch": wl.B, "heads": wl.H,
            "seq_len": wl.L, "block": wl.block, "head_dim": wl.d,
            "causal_diag": bool(wl.causal_diag), "layout": wl.name, "l2": l2_note,
            "parallelism": "replicas" if world > 1 else "single-gpu"}


def time_kernel(index: int, order: str, warmup: int, min_steps: int, min_seconds: float,
                max_steps: int, gpu: int, backward: bool = False) -> dict:
    """Device time of the forward alone on workload `index` (no e2e leg), or of the
    backward (three kernels: delta, dQ, dK/dV): CUDA events around each step on the
    launching stream, the L2 flushed between steps when the inputs would fit in it,
    clocks sampled during the timed region, which lasts at least `min_seconds` (and at
    least `min_steps` steps).  The backward counts 10 * block^2 * d FLOPs per active
    block per batch entry (2.5 times the forward: dS, dQ, dK, dV and the recomputed S)."""
    import torch

    import block_sparse_head_gb300 as bsa
    from block_sparse_head_gb300 import workloads as wls

    wl = wls.WORKLOADS[index]
    lay = wls.layout_for(wl)
    flops_step = (10 if backward else 4) * wl.block * wl.block * wl.d * int(lay.sum()) * wl.B
    q, k, v = wls.qkv(wl)
    lut = bsa.build_lut(lay, wl.B, order)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    del q, k, v
    out = torch.empty_like(qd)
    lse = torch.empty(wl.B, wl.H, wl.L, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    flush = None
    l2_note = "inputs larger than L2"
    if (5 if backward else 3) * qd.numel() * 2 < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
        l2_note = "L2 flushed between steps (256 MiB write, outside the events)"

    if backward:
        bsa.forward(qd, kd, vd, lut, wl.scale, wl.block, wl.causal_diag, out=out, lse=lse,
                    stream=stream)
        dout = wls.randn_qkv(wl.B, wl.H, wl.L, wl.d, seed=5000 + index)[0].cuda()
        grads = tuple(torch.empty_like(qd) for _ in range(3))
        delta = torch.empty_like(lse)

        def step():
            bsa.backward(qd, kd, vd, out, lse, dout, lut, wl.scale, wl.block, wl.causal_diag,
                         *grads, delta=delta, stream=stream)
    else:
        def step():
            bsa.forward(qd, kd, vd, lut, wl.scale, wl.block, wl.causal_diag, out=out, lse=lse,
                        stream=stream)

    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(5):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    est_ms = e0.elapsed_time(e1) / 5
    st, word = lut.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({word:#x}) during warm-up of {wl.name}")
    n = int(min(max_steps, max(min_steps, math.ceil(min_seconds * 1e3 / max(est_ms, 1e-3)))))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    torch.cuda.synchronize()
    clocks = ClockSampler(gpu)
    time.sleep(0.3)
    for s in range(n):
        if flush is not None:
            flush.fill_(s)
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    st, word = lut.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({word:#x}) in the timed region of {wl.name}")
    per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(per_ms)
    peaks = measured_peaks()
    peak_kind = "bf16_burst" if total_ms < 3000 else "bf16_sustained"
    achieved = flops_step / (statistics.mean(per_ms) * 1e-3) / 1e12
    return {"config": workload_config(wl, l2_note, 1), "steps": n,
            "ms_per_step": round(total_ms / n, 5), "value": round(achieved, 2), "unit": "TFLOPS",
            "pct_of_peak": round(100 * achieved / peaks[peak_kind], 2),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks[peak_kind], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks[peak_kind], 4),
                         "peak_source": f"{peaks['source']} {peak_kind} (MEASURED_PEAKS.json)",
                         "traffic": recorded_traffic(wl.name), "flops_per_launch": flops_step},
            "gpu_launches": n * (3 if backward else 1), "clocks": clk}


def time_topk(warmup: int, min_steps: int, min_seconds: float, max_steps: int, gpu: int) -> dict:
    """Device time of bsa_topk_forward on the top-k workload (64 heads of 512, 4096
    positions listing 2048 rows each of a 65536-row context), by the forward's method;
    4 * H * D FLOPs per valid listed row."""
    import torch

    import block_sparse_head_gb300 as bsa
    from block_sparse_head_gb300 import workloads as wls

    wl = wls.TOPK
    q, kv, sink, idx = (t.cuda() for t in wls.topk_inputs(wl.B, wl.M, wl.N, wl.H, wl.D, wl.K,
                                                           seed=2024))
    flops_step = 4 * wl.H * wl.D * int(((idx >= 0) & (idx < wl.N)).sum())
    out = torch.empty_like(q)
    lse = torch.empty(wl.B, wl.M, wl.H, device="cuda", dtype=torch.float32)
    status = torch.zeros(4, device="cuda", dtype=torch.int32)
    stream = torch.cuda.current_stream()

    def step():
        bsa.topk_forward(q, kv, sink, idx, wl.scale, out=out, lse=lse, status=status,
                         stream=stream)

    for _ in range(warmup):
        step()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(3):
        step()
    e1.record(stream)
    torch.cuda.synchronize()
    est_ms = e0.elapsed_time(e1) / 3
    if int(status[0]) != 0:
        raise RuntimeError(f"top-k status {int(status[0]):#x} during warm-up")
    n = int(min(max_steps, max(min_steps, math.ceil(min_seconds * 1e3 / max(est_ms, 1e-3)))))
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    clocks = ClockSampler(gpu)
    time.sleep(0.3)
    for i in range(n):
        starts[i].record(stream)
        step()
        ends[i].record(stream)
    torch.cuda.synchronize()
    clk = clocks.stop()
    if int(status[0]) != 0:
        raise RuntimeError(f"top-k status {int(status[0]):#x} in the timed region")
    per_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    total_ms = sum(per_ms)
    peaks = measured_peaks()
    peak_kind = "bf16_burst" if total_ms < 3000 else "bf16_sustained"
    achieved = flops_step / (statistics.mean(per_ms) * 1e-3) / 1e12
    return {"config": {"workload": f"{wl.name} (top-k token gather with sink)", "batch": wl.B,
                       "positions": wl.M, "kv_rows": wl.N, "heads": wl.H, "head_dim": wl.D,
                       "topk": wl.K, "l2": "inputs larger than L2"},
            "steps": n, "ms_per_step": round(total_ms / n, 5), "value": round(achieved, 2),
            "unit": "TFLOPS", "pct_of_peak": round(100 * achieved / peaks[peak_kind], 2),
            "roofline": {"bound": "tensor", "achieved": round(achieved, 2),
                         "peak": peaks[peak_kind], "unit": "TFLOP/s",
                         "frac": round(achieved / peaks[peak_kind], 4),
                         "peak_source": f"{peaks['source']} {peak_kind} (MEASURED_PEAKS.json)",
                         "traffic": None, "flops_per_launch": flops_step},
            "gpu_launches": n, "clocks": clk}


def gpu_arm(args) -> None:
    import numpy as np  # noqa: F401
    import torch

    import block_sparse_head_gb300 as bsa
    from block_sparse_head_gb300 import binding
    from block_sparse_head_gb300 import workloads as wls

    world, rank, local = dist_setup()
    torch.cuda.set_device(local)
    pg = None
    if world > 1:
        import torch.distributed as dist

        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
        pg = dist

    wl = wls.WORKLOADS[args.workload]
    lay = wls.layout_for(wl)
    flops_step = 4 * wl.block * wl.block * wl.d * int(lay.sum()) * wl.B
    q, k, v = wls.qkv(wl)
    in_bytes = 3 * q.numel() * 2
    lut = bsa.build_lut(lay, wl.B, args.order)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    out = torch.empty_like(qd)
    lse = torch.empty(wl.B, wl.H, wl.L, device="cuda", dtype=torch.float32)
    stream = torch.cuda.current_stream()
    flush = None
    l2_note = "inputs larger than L2"
    if in_bytes < 2 * L2_BYTES:
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.int32, device="cuda")
        l2_note = "L2 flushed between steps (256 MiB write, outside the events)"

    def step():
        bsa.forward(qd, kd, vd, lut, wl.scale, wl.block, wl.causal_diag, out=out, lse=lse,
                    stream=stream)

    for _ in range(args.warmup):
        step()
    st, word = lut.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({word:#x}) during warm-up")

    starts = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(args.steps)]
    if pg:
        pg.barrier()
    torch.cuda.synchronize()
    clocks = ClockSampler(local) if rank == 0 else None
    time.sleep(0.3 if clocks else 0)  # let the sampler start
    t_wall0 = time.perf_counter()
    for s in range(args.steps):
        if flush is not None:
            flush.fill_(s)
        starts[s].record(stream)
        step()
        ends[s].record(stream)
    torch.cuda.synchronize()
    t_wall = time.perf_counter() - t_wall0
    if pg:
        pg.barrier()
    clk = clocks.stop() if clocks else None
    per_step_ms = [a.elapsed_time(b) for a, b in zip(starts, ends)]
    local_ms = sum(per_step_ms)
    st, word = lut.device_status()
    if st != 0:
        raise RuntimeError(f"device status {st} ({word:#x}) in the timed region")

    # e2e: host (pinned) buffers through the same C-ABI call, copies inside the region.
    # Each step copies its q, k, v in, runs the forward and copies out, lse back.  Steps
    # alternate between two streams, each with its own device buffers and LUT, so one
    # step's copies overlap the neighbouring steps' forward and copies (as a serving loop
    # would run); the serial figure (one stream, one step at a time) is reported beside it.
    e2e_steps = max(3, min(args.steps, args.e2e_steps))
    qh, kh, vh = (t.pin_memory() for t in (q, k, v))
    slots = []
    for i in range(2):
        lut_i = lut if i == 0 else bsa.build_lut(lay, wl.B, args.order)
        bufs_i = (qd, kd, vd, out, lse) if i == 0 else tuple(torch.empty_like(t) for t in (qd, kd, vd, out, lse))
        outs_i = (torch.empty(q.shape, dtype=q.dtype, pin_memory=True),
                  torch.empty(q.shape[:3], dtype=torch.float32, pin_memory=True))
        slots.append((lut_i, bufs_i, outs_i, stream if i == 0 else torch.cuda.Stream()))

    def e2e_step(i, serial):
        lut_i, bufs_i, (oh, lh), st_i = slots[0 if serial else i % 2]
        binding.forward_host(qh, kh, vh, lut_i, wl.scale, wl.block, wl.causal_diag, out=oh, lse=lh,
                             dev_bufs=bufs_i, stream=st_i)

    def e2e_time(serial):
        for i in range(2):
            e2e_step(i, serial)
        torch.cuda.synchronize()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        if pg:
            pg.barrier()
        torch.cuda.synchronize()
        e0.record(slots[0][3])
        slots[1][3].wait_event(e0)
        for i in range(e2e_steps):
            e2e_step(i, serial)
        done = torch.cuda.Event()
        done.record(slots[1][3])
        slots[0][3].wait_event(done)
        e1.record(slots[0][3])
        torch.cuda.synchronize()
        return e0.elapsed_time(e1)

    e2e_serial_ms = e2e_time(True)
    e2e_ms_local = e2e_time(False)
    for lut_i, *_ in slots:
        st, word = lut_i.device_status()
        if st != 0:
            raise RuntimeError(f"device status {st} ({word:#x}) in the e2e region")

    local_ms, e2e_ms, e2e_serial_ms = max_over_ranks([local_ms, e2e_ms_local, e2e_serial_ms], pg)
    if rank != 0:
        if pg:
            pg.destroy_process_group()
        return

    ms_per_step = local_ms / args.steps
    value = job_tflops(world, flops_step, args.steps, local_ms)
    peaks = measured_peaks()
    peak_kind = "bf16_burst" if local_ms < 3000 else "bf16_sustained"
    peak = peaks[peak_kind]
    achieved = flops_step / (statistics.mean(per_step_ms) * 1e-3) / 1e12
    traffic = recorded_traffic(wl.name)
    e2e_value = job_tflops(world, flops_step, e2e_steps, e2e_ms)
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 4),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0,1) Q/K/V rounded to bf16; layouts generated from seeds)",
        "config": workload_config(wl, l2_note, world),
        "pct_of_peak": round(100 * value / world / peak, 2),
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peak,
                     "unit": "TFLOP/s", "frac": round(achieved / peak, 4),
                     "peak_source": f"{peaks['source']} {peak_kind} (MEASURED_PEAKS.json)",
                     "traffic": traffic, "flops_per_launch": flops_step},
        "e2e": {"value": round(e2e_value, 2), "unit": "TFLOPS",
                "h2d_bytes_per_step": in_bytes,
                "d2h_bytes_per_step": out.numel() * 2 + lse.numel() * 4,
                "steps": e2e_steps, "ms_per_step": round(e2e_ms / e2e_steps, 3),
                "pipeline": "steps alternate over two streams (own buffers and LUT each)",
                "serial_value": round(job_tflops(world, flops_step, e2e_steps, e2e_serial_ms), 2),
                "serial_ms_per_step": round(e2e_serial_ms / e2e_steps, 3)},
        "gpu_launches": args.steps,
        "clocks": clk,
        "wall_s_timed_region": round(t_wall, 3),
        "order": args.order,
    }
    extra = [int(x) for x in args.extra_workloads.split(",") if x.strip()] if world == 1 else []
    if extra:
        # The forward timed alone on the other target workloads, after the headline, in
        # the same process and by the same method.
        del qd, kd, vd, out, lse, slots
        torch.cuda.empty_cache()
        line["per_workload"] = {}
        for index in extra:
            if index == wl.index:
                continue
            r = time_kernel(index, args.order, max(3, args.warmup), args.steps, args.min_seconds,
                            20000, local)
            line["per_workload"][wls.WORKLOADS[index].name] = r
            torch.cuda.empty_cache()
    bwd = [int(x) for x in args.backward_workloads.split(",") if x.strip()] if world == 1 else []
    if bwd:
        # The backward (bsa_backward: delta, dQ, dK/dV kernels) on the same workloads.
        line["backward"] = {}
        for index in bwd:
            r = time_kernel(index, args.order, max(3, args.warmup), 10, args.min_seconds, 5000,
                            local, backward=True)
            line["backward"][wls.WORKLOADS[index].name] = r
            torch.cuda.empty_cache()
    if args.topk and world == 1:
        # The second workload: top-k token-gather attention with a sink.
        line["topk"] = time_topk(max(3, args.warmup), 10, args.min_seconds, 5000, local)
        torch.cuda.empty_cache()
    if not args.no_cpu_baseline and world == 1:
        cb = cpu_baseline(wl, q, k, v, lay, args.cpu_budget)
        line["cpu_baseline"] = {
            "value": round(cb["tflops"], 6), "unit": "TFLOPS", "cores": cb["cores"],
            "kind": "oracle",
            "sample": (f"{cb['items']} query blocks drawn across the whole work list (seeded "
                       f"permutation), {cb['seconds']:.1f} s of the fp64 numpy oracle, one "
                       f"process per host core ({cb['cores']} processes)")}
    print(json.dumps(line), flush=True)
    if pg:
        pg.destroy_process_group()


def reference_arm(args) -> None:
    world, rank, _ = dist_setup()
    if rank != 0:
        return
    from block_sparse_head_gb300 import workloads as wls

    wl = wls.WORKLOADS[args.workload]
    lay = wls.layout_for(wl)
    q, k, v = wls.qkv(wl)
    procs = host_cores()
    op = OraclePool(wl, q, k, v, lay, procs)
    per_step = args.ref_items * procs
    try:
        for _ in range(args.warmup):
            op.run(per_step)
        flops = secs = 0.0
        for _ in range(args.steps):
            f, t = op.run(per_step)
            flops, secs = flops + f, secs + t
    finally:
        op.close()
    value = flops / secs / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 6),
        "unit": "TFLOPS",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * secs / args.steps, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0,1) Q/K/V rounded to bf16; layouts generated from seeds)",
        "config": workload_config(wl, l2_note_for(wl), 1),
        "impl": "reference",
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOPS", "cores": procs,
                         "kind": "oracle",
                         "sample": (f"each step = {per_step} query blocks drawn across the "
                                    "whole work list (seeded permutation), fp64 numpy oracle, "
                                    f"one process per host core ({procs} processes)")},
        "e2e": {"value": round(value, 6), "unit": "TFLOPS", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--workload", type=int, default=5, choices=[1, 2, 3, 4, 5])
    ap.add_argument("--order", default="global", choices=["global", "grouped"])
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle timing")
    ap.add_argument("--ref-items", type=int, default=2,
                    help="query blocks per host core in each reference step")
    ap.add_argument("--extra-workloads", default="3,4",
                    help="other workloads timed (kernel only) after the headline, comma list")
    ap.add_argument("--backward-workloads", default="3,4,5",
                    help="workloads whose backward is timed after the forward, comma list")
    ap.add_argument("--no-topk", dest="topk", action="store_false",
                    help="skip the top-k token-gather workload")
    ap.add_argument("--min-seconds", type=float, default=0.5,
                    help="shortest timed region of each extra workload")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    args = ap.parse_args()
    if args.warmup < 3 and args.impl == "gb300":
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        reference_arm(args)
    else:
        gpu_arm(args)


if __name__ == "__main__":
    main()
