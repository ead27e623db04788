"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Bars: max |O_gpu - O_oracle| <= 2e-2, mean <= 2e-3, |lse_gpu - lse_oracle| <= 1e-3
(bf16 inputs, fp32 accumulation), and -inf lse exactly on the rows the oracle has
none.  The oracle always runs on the same bf16-rounded inputs the GPU receives.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import block_sparse_head_gb300 as bsa
from block_sparse_head_gb300 import binding
from block_sparse_head_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def run_gpu(q, k, v, lay, scale, block, causal, order="global", stream=None):
    lut = bsa.build_lut(lay, q.shape[0], order)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = bsa.forward(qd, kd, vd, lut, scale, block, causal, stream=stream)
    st, word = lut.device_status(stream)
    assert st == 0, f"device status {st} word {word:#x}"
    return o.float().cpu().numpy(), lse.cpu().numpy()


def np64(t):
    return t.to(torch.float64).numpy()


def compare(o, lse, ro, rl):
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)), "-inf rows differ"
    assert np.all(lse[~fin] == -np.inf)
    assert np.all(np.isfinite(o))
    d = np.abs(o - ro)
    assert d.max() <= TOL_MAX, d.max()
    assert d.mean() <= TOL_MEAN, d.mean()
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= TOL_LSE, np.abs(lse[fin] - rl[fin]).max()


def check_full(q, k, v, lay, scale, block, causal, order="global"):
    o, lse = run_gpu(q, k, v, lay, scale, block, causal, order)
    ro, rl = oracle.forward(np64(q), np64(k), np64(v), np.asarray(lay), scale, block, causal)
    compare(o, lse, ro, rl)
    return o, lse


def test_wait_selftest():
    assert binding.wait_selftest(1_000_000) == binding.BSA_ERR_DEVICE_TIMEOUT


@pytest.mark.parametrize("index", [1, 2, 3])
def test_workload_full(index):
    wl = wls.WORKLOADS[index]
    q, k, v = wls.qkv(wl)
    check_full(q, k, v, wls.layout_for(wl), wl.scale, wl.block, wl.causal_diag)


@pytest.mark.parametrize("index", [4, 5])
def test_workload_full_size_all_rows(index, parity_report):
    """Full-size launch in the benchmark's configuration; every output row of every
    (batch, head) compared with the fp64 oracle (run over a process pool)."""
    from oracle_pool import compare_full

    wl = wls.WORKLOADS[index]
    q, k, v = wls.qkv(wl)
    lay = wls.layout_for(wl)
    lut = bsa.build_lut(lay, wl.B)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    o, lse = bsa.forward(qd, kd, vd, lut, wl.scale, wl.block, wl.causal_diag)
    st, word = lut.device_status()
    assert st == 0, f"device status {st} word {word:#x}"
    o, lse = o.cpu(), lse.cpu()
    del qd, kd, vd
    r = compare_full(q, k, v, lay.numpy(), wl.scale, wl.block, wl.causal_diag, o, lse)
    parity_report.append(
        f"{wl.name}: all {r['rows']} rows vs oracle: max|dO| {r['max_abs']:.3e} "
        f"mean|dO| {r['mean_abs']:.3e} max|dlse| {r['lse_max']:.3e} "
        f"-inf mismatches {r['inf_mismatch']} non-finite {r['nonfinite']} ({r['workers']} workers)")
    assert r["elements"] == wl.B * wl.H * wl.L * wl.d
    assert r["nonfinite"] == 0 and r["inf_mismatch"] == 0
    assert r["max_abs"] <= TOL_MAX and r["mean_abs"] <= TOL_MEAN and r["lse_max"] <= TOL_LSE, r


VARIANTS = [(128, 128), (128, 64), (64, 128), (64, 64)]


@pytest.mark.parametrize("block,d", VARIANTS)
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("seed", [0, 1])
def test_random_layouts(block, d, causal, seed):
    """Random layouts with empty rows, several items per CTA and a ragged last round
    of the persistent loop (item count not a multiple of the SM count)."""
    B, H, nb = 2, 3, 9
    L = nb * block
    lay = wls.random_layout(H, nb, 0.3 + 0.2 * seed, 100 + seed, empty_rows=2)
    q, k, v = wls.randn_qkv(B, H, L, d, seed=7 + seed)
    check_full(q, k, v, lay, 1.0 / math.sqrt(d), block, causal)


@pytest.mark.parametrize("block,d", VARIANTS)
def test_degenerate_layouts(block, d):
    B, H = 1, 2
    # all-zero layout: every row empty -> O = 0, lse = -inf
    nb = 3
    L = nb * block
    q, k, v = wls.randn_qkv(B, H, L, d, seed=3)
    o, lse = run_gpu(q, k, v, torch.zeros(H, nb, nb, dtype=torch.int32), 0.1, block, True)
    assert np.all(o == 0) and np.all(lse == -np.inf)
    # nb = 1 (a single block, the diagonal), all-ones dense, single-block rows
    q1, k1, v1 = wls.randn_qkv(B, H, block, d, seed=4)
    check_full(q1, k1, v1, torch.ones(H, 1, 1, dtype=torch.int32), 0.2, block, True)
    check_full(q, k, v, torch.ones(H, nb, nb, dtype=torch.int32), 1 / math.sqrt(d), block, False)
    eye = torch.eye(nb, dtype=torch.int32)[None].repeat(H, 1, 1)
    check_full(q, k, v, eye, 1 / math.sqrt(d), block, True)
    col0 = torch.zeros(H, nb, nb, dtype=torch.int32)
    col0[:, :, 0] = 1  # every row attends only to block 0 (above-diagonal-free, no diag mask)
    check_full(q, k, v, col0, 1 / math.sqrt(d), block, True)


@pytest.mark.parametrize("block,d", [(128, 128), (64, 128)])
@pytest.mark.parametrize("scale", [0.0, -0.2, 0.5])
def test_scale_values(block, d, scale):
    """scale 0 (mean of the active rows), a negative scale, and a large one (logits of
    tens: the running max moves and the rescale path runs)."""
    B, H, nb = 1, 2, 6
    L = nb * block
    lay = torch.tril(torch.ones(nb, nb, dtype=torch.int32))[None].repeat(H, 1, 1)
    q, k, v = wls.randn_qkv(B, H, L, d, seed=11)
    check_full(q, k, v, lay, scale, block, True)


def test_growing_max_rescale():
    """Later key blocks carry much larger scores than earlier ones, so the running max
    grows by far more than 2^8 from block to block: the O rescale must be exact."""
    block, d, nb, H = 128, 128, 4, 1
    L = nb * block
    q, k, v = wls.randn_qkv(1, H, L, d, seed=12, dtype=torch.float32)
    for j in range(nb):
        k[:, :, j * block:(j + 1) * block] *= 1.0 + 1.5 * j
    q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
    lay = torch.ones(H, nb, nb, dtype=torch.int32)
    check_full(q, k, v, lay, 0.3, block, False)


def test_orders_agree_bitwise_and_deterministic():
    wl = wls.WORKLOADS[2]
    q, k, v = wls.qkv(wl)
    lay = wls.layout_for(wl)
    o1, l1 = run_gpu(q, k, v, lay, wl.scale, wl.block, wl.causal_diag, "global")
    o2, l2 = run_gpu(q, k, v, lay, wl.scale, wl.block, wl.causal_diag, "grouped")
    o3, l3 = run_gpu(q, k, v, lay, wl.scale, wl.block, wl.causal_diag, "global")
    assert np.array_equal(o1, o2) and np.array_equal(l1, l2)
    assert np.array_equal(o1, o3) and np.array_equal(l1, l3)


@pytest.mark.parametrize("index", [2, 3])
def test_schedules_agree_bitwise(index):
    """The two device schedules (work-list order, (batch, head) by (batch, head)) only
    reorder whole items across CTAs: outputs are bitwise the same, and the same as the
    automatic choice."""
    wl = wls.WORKLOADS[index]
    q, k, v = (t.cuda() for t in wls.qkv(wl))
    lut = bsa.build_lut(wls.layout_for(wl), wl.B)
    res = []
    for policy in ("list", "by_head", "auto"):
        lut.set_schedule(policy)
        o, lse = bsa.forward(q, k, v, lut, wl.scale, wl.block, wl.causal_diag)
        assert lut.device_status()[0] == 0
        res.append((o.clone(), lse.clone()))
    for o, lse in res[1:]:
        assert torch.equal(o, res[0][0]) and torch.equal(lse, res[0][1])


def test_side_stream_and_guard_regions():
    """Runs on a non-default stream; output and lse guard regions stay untouched."""
    block, d, nb, B, H = 64, 128, 5, 2, 2
    L = nb * block
    lay = wls.random_layout(H, nb, 0.5, 5, empty_rows=1)
    q, k, v = wls.randn_qkv(B, H, L, d, seed=13)
    n_o, n_l = B * H * L * d, B * H * L
    guard = 4096
    obuf = torch.full((n_o + 2 * guard,), 7.0, dtype=torch.bfloat16, device="cuda")
    lbuf = torch.full((n_l + 2 * guard,), 7.0, dtype=torch.float32, device="cuda")
    out = obuf[guard:guard + n_o].view(B, H, L, d)
    lse = lbuf[guard:guard + n_l].view(B, H, L)
    s = torch.cuda.Stream()
    lut = bsa.build_lut(lay, B)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        bsa.forward(qd, kd, vd, lut, 0.1, block, True, out=out, lse=lse, stream=s)
    assert lut.device_status(s)[0] == 0
    s.synchronize()
    assert torch.all(obuf[:guard] == 7.0) and torch.all(obuf[guard + n_o:] == 7.0)
    assert torch.all(lbuf[:guard] == 7.0) and torch.all(lbuf[guard + n_l:] == 7.0)
    ro, rl = oracle.forward(np64(q), np64(k), np64(v), lay.numpy(), 0.1, block, True)
    compare(out.float().cpu().numpy(), lse.cpu().numpy(), ro, rl)


def test_forward_host_roundtrip():
    wl = wls.WORKLOADS[1]
    q, k, v = (t.pin_memory() for t in wls.qkv(wl))
    lay = wls.layout_for(wl)
    lut = bsa.build_lut(lay, wl.B)
    o, lse = binding.forward_host(q, k, v, lut, wl.scale, wl.block, wl.causal_diag)
    torch.cuda.synchronize()
    ro, rl = oracle.forward(np64(q), np64(k), np64(v), lay.numpy(), wl.scale, wl.block,
                            wl.causal_diag)
    compare(o.float().numpy(), lse.numpy(), ro, rl)


def test_invalid_arguments_raise():
    lut = bsa.build_lut(torch.ones(2, 4, 4, dtype=torch.int32), 1)
    q = torch.zeros(1, 2, 256, 64, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(binding.BsaError):
        bsa.forward(q, q, q, lut, 0.1, 128, False)  # 4 blocks of 128 != 256
    with pytest.raises(ValueError):
        bsa.forward(q.float(), q, q, lut, 0.1, 64, False)
