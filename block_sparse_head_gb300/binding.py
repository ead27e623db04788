"""ctypes binding of libbsa (include/bsa.h): argument marshalling only.

Every step of the forward runs inside the library's CUDA kernel; torch supplies device
memory and streams.  Calls fail loudly (``BsaError``) when the library is missing or
a call returns an error; there is no fallback path.
"""

from __future__ import annotations

import ctypes
import os
import threading

import numpy as np
import torch

_HERE = os.path.dirname(os.path.abspath(__file__))

BSA_ORDER_GLOBAL = 0
BSA_ORDER_GROUPED = 1
_ORDERS = {"global": BSA_ORDER_GLOBAL, "grouped": BSA_ORDER_GROUPED,
           BSA_ORDER_GLOBAL: BSA_ORDER_GLOBAL, BSA_ORDER_GROUPED: BSA_ORDER_GROUPED}

BSA_ERR_DEVICE_TIMEOUT = -8

# Every symbol declared in include/bsa.h.
EXPORTED = (
    "bsa_build_lut", "bsa_lut_info", "bsa_lut_export", "bsa_lut_schedule", "bsa_lut_upload",
    "bsa_lut_free",
    "bsa_forward", "bsa_device_status", "bsa_set_schedule", "bsa_set_wait_limit",
    "bsa_wait_selftest",
    "bsa_status_string", "bsa_version", "bsa_forward_noalloc", "bsa_debug_expire_wait",
    "bsa_build_lut_rect", "bsa_lut_kv_blocks", "bsa_forward_ext", "bsa_lut_export_csc",
    "bsa_backward", "bsa_topk_forward",
)


class ExtArgs(ctypes.Structure):
    """bsa_ext_args of include/bsa.h."""
    _fields_ = [("window_left", ctypes.c_int), ("window_right", ctypes.c_int),
                ("softcap", ctypes.c_float), ("sinks", ctypes.c_void_p),
                ("q_segment_ids", ctypes.c_void_p), ("kv_segment_ids", ctypes.c_void_p)]

_lib = None
_lock = threading.Lock()


class BsaError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        text = _lib.bsa_status_string(status).decode() if _lib is not None else str(status)
        super().__init__(f"{what}: {text} ({status})")


def library_path() -> str:
    return os.path.join(_HERE, "libbsa.so")


def load_library():
    """Load libbsa.so (built by ``block_sparse_head_gb300.build``) and declare its ABI."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(
                f"{path} is missing: build it with `python -m block_sparse_head_gb300.build` "
                "(the CUDA path has no fallback)")
        lib = ctypes.CDLL(path)
        i32p = ctypes.POINTER(ctypes.c_int32)
        ip = ctypes.POINTER(ctypes.c_int)
        vp = ctypes.c_void_p
        lib.bsa_build_lut.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                      ctypes.POINTER(vp)]
        lib.bsa_build_lut_rect.argtypes = [vp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int, ctypes.POINTER(vp)]
        lib.bsa_lut_kv_blocks.argtypes = [vp, ip]
        lib.bsa_forward_ext.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                        ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.POINTER(ExtArgs), vp]
        lib.bsa_topk_forward.argtypes = [vp, vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                         ctypes.c_float, vp]
        lib.bsa_lut_export_csc.argtypes = [vp, vp, vp, vp]
        lib.bsa_backward.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, vp, ctypes.c_int,
                                     ctypes.c_int, ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                     ctypes.c_int, ctypes.c_int, vp]
        lib.bsa_lut_info.argtypes = [vp, ip, ip, ip, ip, ip]
        lib.bsa_lut_export.argtypes = [vp, vp, vp, vp]
        lib.bsa_lut_schedule.argtypes = [vp, ctypes.c_int, ctypes.c_int, vp, vp]
        lib.bsa_lut_upload.argtypes = [vp, vp]
        lib.bsa_lut_free.argtypes = [vp]
        lib.bsa_lut_free.restype = None
        lib.bsa_forward.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                                    ctypes.c_int, vp]
        lib.bsa_forward_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, ctypes.c_int, ctypes.c_int,
                                            ctypes.c_int, ctypes.c_int, ctypes.c_float,
                                            ctypes.c_int, ctypes.c_int, vp, ctypes.c_int]
        lib.bsa_forward_noalloc.restype = ctypes.c_int
        lib.bsa_device_status.argtypes = [vp, vp, i32p]
        lib.bsa_set_wait_limit.argtypes = [vp, ctypes.c_uint64]
        lib.bsa_set_schedule.argtypes = [vp, ctypes.c_int]
        lib.bsa_debug_expire_wait.argtypes = [vp, ctypes.c_int]
        lib.bsa_wait_selftest.argtypes = [ctypes.c_uint64, vp]
        lib.bsa_status_string.argtypes = [ctypes.c_int]
        lib.bsa_status_string.restype = ctypes.c_char_p
        lib.bsa_version.argtypes = []
        lib.bsa_version.restype = ctypes.c_char_p
        for name in ("bsa_build_lut", "bsa_lut_info", "bsa_lut_export", "bsa_lut_schedule",
                     "bsa_lut_upload",
                     "bsa_forward", "bsa_device_status", "bsa_set_schedule", "bsa_set_wait_limit",
                     "bsa_wait_selftest", "bsa_debug_expire_wait", "bsa_build_lut_rect",
                     "bsa_lut_kv_blocks", "bsa_forward_ext", "bsa_lut_export_csc",
                     "bsa_backward", "bsa_topk_forward"):
            getattr(lib, name).restype = ctypes.c_int
        _lib = lib
        return lib


def _check(status: int, what: str) -> None:
    if status != 0:
        raise BsaError(status, what)


def _stream_handle(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


class Lut:
    """A built look-up table (CSR of active column blocks + work list)."""

    def __init__(self, layout, batch: int, order="global"):
        lib = load_library()
        lay = layout.detach().cpu().numpy() if isinstance(layout, torch.Tensor) else np.asarray(layout)
        if lay.ndim != 3:
            raise ValueError(f"layout must be [H, nb, nbk], got {lay.shape}")
        lay = np.ascontiguousarray(lay.astype(np.int32, copy=False))
        self._lib = lib
        self.handle = ctypes.c_void_p()
        if lay.shape[1] == lay.shape[2]:
            _check(lib.bsa_build_lut(lay.ctypes.data, lay.shape[0], lay.shape[1], int(batch),
                                     _ORDERS[order], ctypes.byref(self.handle)), "bsa_build_lut")
        else:
            _check(lib.bsa_build_lut_rect(lay.ctypes.data, lay.shape[0], lay.shape[1],
                                          lay.shape[2], int(batch), _ORDERS[order],
                                          ctypes.byref(self.handle)), "bsa_build_lut_rect")
        H, nb, b, nnz, n, nbk = (ctypes.c_int() for _ in range(6))
        _check(lib.bsa_lut_info(self.handle, *(ctypes.byref(x) for x in (H, nb, b, nnz, n))),
               "bsa_lut_info")
        _check(lib.bsa_lut_kv_blocks(self.handle, ctypes.byref(nbk)), "bsa_lut_kv_blocks")
        self.H, self.nb, self.batch, self.nbk = H.value, nb.value, b.value, nbk.value
        self.nnz_total, self.n_items = nnz.value, n.value
        self.device = None

    def export(self):
        """(row_ptr [H*nb+1], col_idx [nnz], items [n_items, 4]) as int32 numpy arrays."""
        rp = np.empty(self.H * self.nb + 1, np.int32)
        ci = np.empty(max(self.nnz_total, 1), np.int32)
        it = np.empty((self.n_items, 4), np.int32)
        _check(self._lib.bsa_lut_export(self.handle, rp.ctypes.data, ci.ctypes.data, it.ctypes.data),
               "bsa_lut_export")
        return rp, ci[:self.nnz_total], it

    def export_csc(self):
        """(col_ptr [H*nb+1], row_idx [nnz], items [n_items, 4]) of the column view."""
        cp = np.empty(self.H * self.nb + 1, np.int32)
        ri = np.empty(max(self.nnz_total, 1), np.int32)
        it = np.empty((self.n_items, 4), np.int32)
        _check(self._lib.bsa_lut_export_csc(self.handle, cp.ctypes.data, ri.ctypes.data,
                                            it.ctypes.data), "bsa_lut_export_csc")
        return cp, ri[:self.nnz_total], it

    def schedule(self, grid: int, by_head: bool = False):
        """(items [n_items, 4], cta_start [grid + 1]) of the per-CTA schedule for ``grid``
        CTAs: CTA c runs items[cta_start[c]:cta_start[c + 1]].  ``by_head`` hands the items
        out (batch, head) by (batch, head) instead of in work-list order."""
        it = np.empty((max(self.n_items, 1), 4), np.int32)
        cs = np.empty(int(grid) + 1, np.int32)
        _check(self._lib.bsa_lut_schedule(self.handle, int(grid), int(bool(by_head)),
                                          it.ctypes.data, cs.ctypes.data), "bsa_lut_schedule")
        return it[:self.n_items], cs

    def upload(self, stream=None):
        _check(self._lib.bsa_lut_upload(self.handle, _stream_handle(stream)), "bsa_lut_upload")
        self.device = torch.cuda.current_device()
        return self

    _SCHEDULES = {"auto": 0, "list": 1, "by_head": 2}

    def set_schedule(self, policy: str = "auto"):
        """Device schedule of later forwards: "auto", "list" or "by_head"."""
        _check(self._lib.bsa_set_schedule(self.handle, self._SCHEDULES[policy]), "bsa_set_schedule")

    def set_wait_limit(self, ns: int):
        _check(self._lib.bsa_set_wait_limit(self.handle, int(ns)), "bsa_set_wait_limit")

    def debug_expire_wait(self, site: int):
        """Test knob: later forwards treat every wait at ``site`` as run out (0: off)."""
        _check(self._lib.bsa_debug_expire_wait(self.handle, int(site)), "bsa_debug_expire_wait")

    def device_status(self, stream=None) -> tuple[int, int]:
        """(status, raw word) of the device status word; synchronizes the stream."""
        word = ctypes.c_int32(0)
        st = self._lib.bsa_device_status(self.handle, _stream_handle(stream), ctypes.byref(word))
        return st, word.value

    def __del__(self):
        h = getattr(self, "handle", None)
        if h is not None and h.value:
            self._lib.bsa_lut_free(h)
            self.handle = None


def build_lut(layout, batch: int, order="global", upload: bool | None = None, stream=None) -> Lut:
    """Build the LUT on the host; upload it to the current CUDA device when one exists
    (or when ``upload`` is True)."""
    lut = Lut(layout, batch, order)
    if upload is None:
        upload = torch.cuda.is_available()
    if upload:
        lut.upload(stream)
    return lut


def _check_qkv(t: torch.Tensor, name: str, shape) -> None:
    if not t.is_cuda or t.dtype != torch.bfloat16 or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous bf16 CUDA tensor")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")


def forward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lut: Lut, scale: float,
            block: int, causal_diag: bool, out: torch.Tensor | None = None,
            lse: torch.Tensor | None = None, stream=None):
    """Block-sparse attention forward.  q, k, v: bf16 [B, H, L, d] on the LUT's device.
    Returns (out bf16 [B, H, L, d], lse fp32 [B, H, L])."""
    lib = load_library()
    B, H, L, d = q.shape
    _check_qkv(q, "q", (B, H, L, d))
    _check_qkv(k, "k", (B, H, L, d))
    _check_qkv(v, "v", (B, H, L, d))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, L, device=q.device, dtype=torch.float32)
    _check_qkv(out, "out", (B, H, L, d))
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, L) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, L] tensor")
    _check(lib.bsa_forward(q.data_ptr(), k.data_ptr(), v.data_ptr(), lut.handle, out.data_ptr(),
                           lse.data_ptr(), B, H, L, d, float(scale), int(block), int(bool(causal_diag)),
                           _stream_handle(stream)), "bsa_forward")
    return out, lse


def forward_ext(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lut: Lut, scale: float,
                q_block: int, kv_block: int, causal_diag: bool, window=None, softcap: float = 0.0,
                sinks: torch.Tensor | None = None, q_segment_ids: torch.Tensor | None = None,
                kv_segment_ids: torch.Tensor | None = None, out: torch.Tensor | None = None,
                lse: torch.Tensor | None = None, stream=None):
    """Extended forward (bsa_forward_ext): q [B,H,Lq,d], k/v [B,H,Lk,d] bf16; ``window``
    an int (both sides) or a (left, right) pair (None or negative: no bound); ``sinks``
    fp32 [H]; segment ids int32 [B,Lq] / [B,Lk].  Returns (out [B,H,Lq,d], lse [B,H,Lq])."""
    lib = load_library()
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    _check_qkv(q, "q", (B, H, Lq, d))
    _check_qkv(k, "k", (B, H, Lk, d))
    _check_qkv(v, "v", (B, H, Lk, d))
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(B, H, Lq, device=q.device, dtype=torch.float32)
    _check_qkv(out, "out", (B, H, Lq, d))
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, Lq) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, Lq] tensor")
    if window is None:
        wl = wr = -1
    elif isinstance(window, int):
        wl = wr = window
    else:
        wl, wr = (-1 if w is None else int(w) for w in window)

    def dev_arr(t, dtype, shape, name):
        if t is None:
            return None
        if not t.is_cuda or t.dtype != dtype or not t.is_contiguous() or tuple(t.shape) != shape:
            raise ValueError(f"{name} must be a contiguous {dtype} CUDA tensor of shape {shape}")
        return t.data_ptr()

    x = ExtArgs(wl, wr, float(softcap), dev_arr(sinks, torch.float32, (H,), "sinks"),
                dev_arr(q_segment_ids, torch.int32, (B, Lq), "q_segment_ids"),
                dev_arr(kv_segment_ids, torch.int32, (B, Lk), "kv_segment_ids"))
    _check(lib.bsa_forward_ext(q.data_ptr(), k.data_ptr(), v.data_ptr(), lut.handle,
                               out.data_ptr(), lse.data_ptr(), B, H, Lq, Lk, d, float(scale),
                               int(q_block), int(kv_block), int(bool(causal_diag)),
                               ctypes.byref(x), _stream_handle(stream)), "bsa_forward_ext")
    return out, lse


def backward(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, out: torch.Tensor,
             lse: torch.Tensor, dout: torch.Tensor, lut: Lut, scale: float, block: int,
             causal_diag: bool, dq=None, dk=None, dv=None, delta=None, stream=None):
    """Gradients (dq, dk, dv) of the forward (bsa_backward).  q, k, v, out, dout: bf16
    [B, H, L, d] on the LUT's device; lse fp32 [B, H, L] from the forward.  ``delta`` is
    an fp32 [B, H, L] workspace (allocated when None)."""
    lib = load_library()
    B, H, L, d = q.shape
    for t, name in ((q, "q"), (k, "k"), (v, "v"), (out, "out"), (dout, "dout")):
        _check_qkv(t, name, (B, H, L, d))
    if lse.dtype != torch.float32 or tuple(lse.shape) != (B, H, L) or not lse.is_contiguous():
        raise ValueError("lse must be a contiguous fp32 [B, H, L] tensor")
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(q) if dk is None else dk
    dv = torch.empty_like(q) if dv is None else dv
    for t, name in ((dq, "dq"), (dk, "dk"), (dv, "dv")):
        _check_qkv(t, name, (B, H, L, d))
    if delta is None:
        delta = torch.empty(B, H, L, device=q.device, dtype=torch.float32)
    _check(lib.bsa_backward(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                            lse.data_ptr(), dout.data_ptr(), lut.handle, dq.data_ptr(),
                            dk.data_ptr(), dv.data_ptr(), delta.data_ptr(), B, H, L, d,
                            float(scale), int(block), int(bool(causal_diag)),
                            _stream_handle(stream)), "bsa_backward")
    return dq, dk, dv


def topk_forward(q: torch.Tensor, kv: torch.Tensor, sink: torch.Tensor, idx: torch.Tensor,
                 scale: float, out: torch.Tensor | None = None, lse: torch.Tensor | None = None,
                 status: torch.Tensor | None = None, stream=None):
    """Top-k token-gather attention with a sink (bsa_topk_forward).  q bf16 [B, M, H, D],
    kv bf16 [B, N, D], sink fp32 [H], idx int32 [B, M, K] (-1: unused).  Returns
    (out bf16 [B, M, H, D], lse fp32 [B, M, H], status int32 [1]); a nonzero status
    (read after the stream is synchronized) means a bounded wait gave up."""
    lib = load_library()
    B, M, H, D = q.shape
    N, K = kv.shape[1], idx.shape[2]
    _check_qkv(q, "q", (B, M, H, D))
    _check_qkv(kv, "kv", (B, N, D))
    if not sink.is_cuda or sink.dtype != torch.float32 or tuple(sink.shape) != (H,):
        raise ValueError("sink must be a CUDA fp32 tensor of shape [H]")
    if not idx.is_cuda or idx.dtype != torch.int32 or not idx.is_contiguous() or idx.shape[:2] != (B, M):
        raise ValueError("idx must be a contiguous CUDA int32 tensor [B, M, K]")
    out = torch.empty_like(q) if out is None else out
    lse = torch.empty(B, M, H, device=q.device, dtype=torch.float32) if lse is None else lse
    status = torch.zeros(4, device=q.device, dtype=torch.int32) if status is None else status
    _check_qkv(out, "out", (B, M, H, D))
    _check(lib.bsa_topk_forward(q.data_ptr(), kv.data_ptr(), sink.contiguous().data_ptr(),
                                idx.data_ptr(), out.data_ptr(), lse.data_ptr(), status.data_ptr(),
                                B, M, N, H, D, K, float(scale), _stream_handle(stream)),
           "bsa_topk_forward")
    return out, lse, status


def forward_host(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, lut: Lut, scale: float,
                 block: int, causal_diag: bool, out: torch.Tensor | None = None,
                 lse: torch.Tensor | None = None, dev_bufs=None, stream=None):
    """Forward from host (ideally pinned) tensors: copies q, k, v to the device, runs
    ``forward`` and copies out / lse back into host tensors, all on one stream.

    ``dev_bufs`` may hold preallocated device tensors (q, k, v, out, lse) to reuse."""
    dev = torch.device("cuda", torch.cuda.current_device())
    if dev_bufs is None:
        dev_bufs = (torch.empty_like(q, device=dev), torch.empty_like(k, device=dev),
                    torch.empty_like(v, device=dev), torch.empty_like(q, device=dev),
                    torch.empty(q.shape[:3], device=dev, dtype=torch.float32))
    dq, dk, dv, do, dl = dev_bufs
    s = stream if stream is not None else torch.cuda.current_stream()
    with torch.cuda.stream(s):
        dq.copy_(q, non_blocking=True)
        dk.copy_(k, non_blocking=True)
        dv.copy_(v, non_blocking=True)
        forward(dq, dk, dv, lut, scale, block, causal_diag, out=do, lse=dl, stream=s)
        if out is None:
            out = torch.empty(q.shape, dtype=q.dtype, pin_memory=True)
        if lse is None:
            lse = torch.empty(q.shape[:3], dtype=torch.float32, pin_memory=True)
        out.copy_(do, non_blocking=True)
        lse.copy_(dl, non_blocking=True)
    return out, lse


def wait_selftest(limit_ns: int = 1_000_000, stream=None) -> int:
    """Run the bounded-wait self-test kernel; returns its status (expected
    BSA_ERR_DEVICE_TIMEOUT = -8)."""
    lib = load_library()
    return lib.bsa_wait_selftest(int(limit_ns), _stream_handle(stream))


def version() -> str:
    return load_library().bsa_version().decode()
