"""bsa_forward_noalloc: the forward for callers that cannot allocate device memory.

Some callers may not call cudaMalloc (host callbacks or plugin hooks where it could
deadlock, a memory manager that owns the device heap, a process whose footprint must
not grow after start-up).  This entry point keeps the LUT's device copy and its status
word in a fixed array inside the library instead of allocating them.  The test calls
it through the C ABI twice in a row, with a LUT that was never uploaded, and checks
each result against the regular bsa_forward and against the fp64 oracle, within the
parity tolerances used by the other GPU tests.  It lives in its own file, named to be
collected last.
"""

import ctypes
import math

import numpy as np
import pytest
import torch

import oracle
import block_sparse_head_gb300 as bsa
from block_sparse_head_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 2e-2, 2e-3, 1e-3
BSA_ERR_TOO_LARGE = -11


def _noalloc(lib, q, k, v, lut, out, lse, scale, block, causal, stream):
    B, H, L, d = q.shape
    return lib.bsa_forward_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), lut.handle,
                                   out.data_ptr(), lse.data_ptr(), B, H, L, d,
                                   ctypes.c_float(scale), block, int(causal),
                                   ctypes.c_void_p(stream.cuda_stream), 1)


def _close(o, lse, ro, rl):
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    if isinstance(ro, torch.Tensor):
        ro, rl = ro.float().cpu().numpy(), rl.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    d = np.abs(o - ro)
    assert d.max() <= TOL_MAX and d.mean() <= TOL_MEAN
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= TOL_LSE


CASES = [
    # (layout, B, block, d, causal, seed): a workload layout and a random one with empty rows
    ("band4", None, 64, 64, False, 0),
    ("random", 2, 128, 128, True, 1),
    ("random", 1, 64, 128, True, 2),
]


def _case(name, B, block, d, causal, seed):
    if name == "band4":
        wl = wls.WORKLOADS[2]
        return wls.layout_for(wl), wl.B, wls.qkv(wl)
    H, nb = 3, 7
    lay = wls.random_layout(H, nb, 0.4, 50 + seed, empty_rows=1)
    return lay, B, wls.randn_qkv(B, H, nb * block, d, seed=60 + seed)


@pytest.mark.parametrize("name,B,block,d,causal,seed", CASES)
def test_noalloc_matches_forward_two_calls(cuda_lib, name, B, block, d, causal, seed):
    lib = cuda_lib
    lay, B, (q, k, v) = _case(name, B, block, d, causal, seed)
    scale = 1.0 / math.sqrt(d)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    ref_lut = bsa.build_lut(lay, B)  # uploaded: the regular entry point
    ro, rl = bsa.forward(qd, kd, vd, ref_lut, scale, block, causal)
    assert ref_lut.device_status()[0] == 0
    oo, ol = oracle.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                            np.asarray(lay), scale, block, causal)
    lut = bsa.build_lut(lay, B, upload=False)  # host-only LUT
    stream = torch.cuda.current_stream()
    for _ in range(2):
        out = torch.full_like(qd, float("nan"))
        lse = torch.full(q.shape[:3], float("nan"), device="cuda")
        assert _noalloc(lib, qd, kd, vd, lut, out, lse, scale, block, causal, stream) == 0
        torch.cuda.synchronize()
        _close(out, lse, ro, rl)
        _close(out, lse, oo, ol)


def test_noalloc_rejects_oversized_lut(cuda_lib):
    lib = cuda_lib
    # 1 x 1 x 1024 blocks of 64 -> 1024 items (4096 words) + 1024*1024 col_idx words
    nb = 1024
    lay = torch.ones(1, nb, nb, dtype=torch.int32)
    lut = bsa.build_lut(lay, 1, upload=False)
    L = nb * 64
    q = torch.zeros(1, 1, L, 64, dtype=torch.bfloat16, device="cuda")
    lse = torch.empty(1, 1, L, device="cuda")
    st = _noalloc(lib, q, q, q, lut, q, lse, 0.1, 64, False, torch.cuda.current_stream())
    assert st == BSA_ERR_TOO_LARGE
    assert "4 MiB" in lib.bsa_status_string(st).decode()
