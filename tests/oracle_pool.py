"""Full-size comparison of GPU results with the fp64 oracle over a process pool.

Test helper.  The inputs (bf16 bit patterns) and the GPU's O (bf16) and lse (fp32)
are written once to memory-mapped files in a temporary directory; each worker maps
them read only, runs ``oracle.query_block`` for chunks of query blocks of one
(batch, head), and returns error statistics only.  Every query block of every
(batch, head) is compared, so a fault confined to rare rows cannot hide.

The pool uses the ``spawn`` start method: a process forked after CUDA initialised
in the parent can hang.
"""

from __future__ import annotations

import multiprocessing as mp
import os
import tempfile

import numpy as np

_W = {}  # per-worker state (maps, layout, parameters)


def _bf16_to_f32(a: np.ndarray) -> np.ndarray:
    """bf16 bit patterns (uint16) to fp32 (exact)."""
    return (a.astype(np.uint32) << 16).view(np.float32)


_BLAS_VARS = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS")


def _init(tmp, shape, lay, scale, block, causal):
    B, H, L, d = shape
    _W["q"] = np.memmap(os.path.join(tmp, "q"), np.uint16, "r", shape=shape)
    _W["k"] = np.memmap(os.path.join(tmp, "k"), np.uint16, "r", shape=shape)
    _W["v"] = np.memmap(os.path.join(tmp, "v"), np.uint16, "r", shape=shape)
    _W["o"] = np.memmap(os.path.join(tmp, "o"), np.uint16, "r", shape=shape)
    _W["lse"] = np.memmap(os.path.join(tmp, "lse"), np.float32, "r", shape=(B, H, L))
    _W["lay"] = lay
    _W["par"] = (scale, block, causal)
    _W["bh"] = None


def _task(args):
    import oracle

    b, h, i0, i1 = args
    scale, block, causal = _W["par"]
    if _W["bh"] != (b, h):
        _W["cur"] = tuple(_bf16_to_f32(np.asarray(_W[n][b, h])) for n in ("q", "k", "v", "o"))
        _W["bh"] = (b, h)
    q, k, v, o = _W["cur"]
    lse = np.asarray(_W["lse"][b, h])
    st = {"max": 0.0, "sum": 0.0, "n": 0, "lse_max": 0.0, "inf_mismatch": 0, "nonfinite": 0}
    for i in range(i0, i1):
        ro, rl = oracle.query_block(q, k, v, _W["lay"][h], scale, block, causal, i)
        sl = slice(i * block, (i + 1) * block)
        og = o[sl].astype(np.float64)
        lg = lse[sl].astype(np.float64)
        st["nonfinite"] += int((~np.isfinite(og)).sum())
        d = np.abs(og - ro)
        st["max"] = max(st["max"], float(np.nanmax(d)) if d.size else 0.0)
        st["sum"] += float(np.nansum(d))
        st["n"] += d.size
        fin = np.isfinite(rl)
        st["inf_mismatch"] += int(((fin != np.isfinite(lg)) | (~fin & (lg != -np.inf))).sum())
        if fin.any():
            st["lse_max"] = max(st["lse_max"], float(np.abs(lg[fin] - rl[fin]).max()))
    return st


def compare_full(q, k, v, lay, scale: float, block: int, causal: bool, o_gpu, lse_gpu,
                 workers: int | None = None, chunk: int = 64) -> dict:
    """Compare every output row of a forward with the oracle.

    q, k, v, o_gpu: torch bf16 CPU tensors [B, H, L, d]; lse_gpu: torch fp32 CPU tensor
    [B, H, L]; lay: int [H, nb, nb].  Returns max and mean |O_gpu - O_oracle| over all
    elements, the max |lse_gpu - lse_oracle| over rows with a finite oracle lse, the
    number of rows whose -inf pattern differs, and the number of non-finite outputs."""
    import torch

    shape = tuple(q.shape)
    B, H, L, d = shape
    nb = L // block
    lay = np.ascontiguousarray(np.asarray(lay, dtype=np.int64))
    if workers is None:
        workers = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    with tempfile.TemporaryDirectory(prefix="bsa_parity_") as tmp:
        for name, t in (("q", q), ("k", k), ("v", v), ("o", o_gpu)):
            assert t.dtype == torch.bfloat16 and tuple(t.shape) == shape
            t.contiguous().view(torch.int16).numpy().view(np.uint16).tofile(os.path.join(tmp, name))
        lse_gpu.contiguous().numpy().astype(np.float32).tofile(os.path.join(tmp, "lse"))
        tasks = [(b, h, i0, min(nb, i0 + chunk)) for b in range(B) for h in range(H)
                 for i0 in range(0, nb, chunk)]
        ctx = mp.get_context("spawn")
        # One BLAS thread per worker, set in the environment the workers inherit (a
        # worker imports numpy while unpickling its arguments, before any initializer).
        saved = {var: os.environ.get(var) for var in _BLAS_VARS}
        os.environ.update({var: "1" for var in _BLAS_VARS})
        try:
            pool = ctx.Pool(max(1, min(workers, len(tasks))), initializer=_init,
                            initargs=(tmp, shape, lay, scale, block, causal))
        finally:
            for var, val in saved.items():
                if val is None:
                    os.environ.pop(var, None)
                else:
                    os.environ[var] = val
        with pool:
            parts = pool.map(_task, tasks, chunksize=1)
    n = sum(p["n"] for p in parts)
    return {"max_abs": max(p["max"] for p in parts), "mean_abs": sum(p["sum"] for p in parts) / max(n, 1),
            "lse_max": max(p["lse_max"] for p in parts),
            "inf_mismatch": sum(p["inf_mismatch"] for p in parts),
            "nonfinite": sum(p["nonfinite"] for p in parts), "elements": n,
            "rows": B * H * L, "workers": workers}
