"""GPU parity of bsa_backward (dq, dk, dv) against the fp64 backward oracle.

Bars.  Every gradient element is a sum of products in which one factor was rounded to
bf16 before the second product (P or dS, relative error <= 2^-9), accumulated in fp32,
and the result is rounded to bf16 (<= 2^-9 relative); delta uses the bf16-rounded O of
the forward.  So an element's error is of order 2^-8 of the largest magnitudes it sums;
the bars leave a factor of about five above that:
    max |g - g_oracle|  <= 2e-2 * max(1, max |g_oracle|)
    mean |g - g_oracle| <= 2e-3 * max(1, mean |g_oracle|)
Rows with no active key get dq = 0 exactly, keys no row attends get dk = dv = 0.
The oracle runs on the same bf16-rounded q, k, v and dout.
"""

import math

import numpy as np
import pytest
import torch

import oracle
import block_sparse_head_gb300 as bsa
from block_sparse_head_gb300 import workloads as wls

pytestmark = pytest.mark.gpu

VARIANTS = [(128, 128), (128, 64), (64, 128), (64, 64)]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _run(q, k, v, do, lay, scale, block, causal):
    lut = bsa.build_lut(lay, q.shape[0])
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.forward(qd, kd, vd, lut, scale, block, causal)
    dq, dk, dv = bsa.backward(qd, kd, vd, o, lse, dod, lut, scale, block, causal)
    st, word = lut.device_status()
    assert st == 0, hex(word)
    return [t.float().cpu().numpy() for t in (dq, dk, dv)]


def _compare(got, ref, report=None, name=""):
    figs = []
    for g, r, what in zip(got, ref, ("dq", "dk", "dv")):
        assert np.all(np.isfinite(g)), what
        err = np.abs(g - r)
        mx, mn = err.max(), err.mean()
        figs.append(f"{what} max {mx:.2e} (|ref| {np.abs(r).max():.2f}) mean {mn:.2e}")
        assert mx <= 2e-2 * max(1.0, np.abs(r).max()), (what, mx)
        assert mn <= 2e-3 * max(1.0, np.abs(r).mean()), (what, mn)
    if report is not None:
        report.append(f"backward {name}: " + "; ".join(figs))


@pytest.mark.parametrize("block,d", VARIANTS)
@pytest.mark.parametrize("causal", [False, True])
def test_random_layouts(block, d, causal):
    """Random layouts with empty rows and never-attended key blocks, more items than
    one per CTA for neither walk (a ragged persistent loop)."""
    B, H, nb = 2, 3, 9
    L = nb * block
    lay = wls.random_layout(H, nb, 0.4, 70 + block + d, empty_rows=2)
    if causal:
        idx = torch.arange(nb)
        lay[:, idx, idx] = torch.where(lay.sum(2) > 0, 1, 0).to(torch.int32)
    lay[:, :, 4] = 0  # key block 4 is never attended: dk = dv = 0 there
    q, k, v, do = wls.randn_qkv(B, H, L, d, seed=71) + (wls.randn_qkv(B, H, L, d, seed=72)[0],)
    scale = 1 / math.sqrt(d)
    got = _run(q, k, v, do, lay, scale, block, causal)
    ref = oracle.backward(*(t.double().numpy() for t in (q, k, v, do)), lay.numpy(), scale, block,
                          causal)
    _compare(got, ref)
    dk, dv = got[1], got[2]
    assert np.all(dk[:, :, 4 * block:5 * block] == 0) and np.all(dv[:, :, 4 * block:5 * block] == 0)
    empty = (lay.sum(2) == 0).numpy()  # [H, nb]
    for h in range(H):
        for i in np.nonzero(empty[h])[0]:
            assert np.all(got[0][:, h, i * block:(i + 1) * block] == 0)


@pytest.mark.parametrize("index", [1, 2, 3])
def test_workloads(index, parity_report):
    """Workloads 1-3 at full size, every row of every gradient against the oracle."""
    wl = wls.WORKLOADS[index]
    q, k, v = wls.qkv(wl)
    do = wls.randn_qkv(wl.B, wl.H, wl.L, wl.d, seed=5000 + index)[0]
    lay = wls.layout_for(wl)
    got = _run(q, k, v, do, lay, wl.scale, wl.block, wl.causal_diag)
    ref = oracle.backward_blocks(*(t.double().numpy() for t in (q, k, v, do)), lay.numpy(),
                                 wl.scale, wl.block, wl.causal_diag)
    _compare(got, ref, parity_report, wl.name)


def test_negative_and_zero_scale():
    block, d, nb, B, H = 128, 128, 5, 1, 2
    L = nb * block
    lay = torch.tril(torch.ones(nb, nb, dtype=torch.int32))[None].repeat(H, 1, 1)
    q, k, v = wls.randn_qkv(B, H, L, d, seed=81)
    do = wls.randn_qkv(B, H, L, d, seed=82)[0]
    for scale in (-0.1, 0.0):
        got = _run(q, k, v, do, lay, scale, block, True)
        ref = oracle.backward(*(t.double().numpy() for t in (q, k, v, do)), lay.numpy(), scale,
                              block, True)
        _compare(got, ref)


@pytest.mark.parametrize("index", [4, 5])
def test_workload_full_size_sampled(index, parity_report):
    """Full-size backward in the benchmark's configuration: every gradient finite, and the
    rows of three (batch, head) pairs compared with the fp64 oracle -- dq of the longest
    and of random query blocks, dk and dv of the most attended, of random and (if any)
    of unattended key blocks."""
    wl = wls.WORKLOADS[index]
    q, k, v = wls.qkv(wl)
    do = wls.randn_qkv(wl.B, wl.H, wl.L, wl.d, seed=5000 + index)[0]
    lay = wls.layout_for(wl)
    lut = bsa.build_lut(lay, wl.B)
    qd, kd, vd, dod = (t.cuda() for t in (q, k, v, do))
    o, lse = bsa.forward(qd, kd, vd, lut, wl.scale, wl.block, wl.causal_diag)
    g = bsa.backward(qd, kd, vd, o, lse, dod, lut, wl.scale, wl.block, wl.causal_diag)
    st, word = lut.device_status()
    assert st == 0, hex(word)
    for t, what in zip(g, ("dq", "dk", "dv")):
        assert bool(torch.isfinite(t).all()), what
    dq, dk, dv = (t.float().cpu().numpy() for t in g)
    del qd, kd, vd, dod, o, lse, g
    lay_np = lay.numpy()
    nb, blk = lay_np.shape[1], wl.block
    rng = np.random.default_rng(77 + index)
    got, ref = [[], [], []], [[], [], []]
    for b, h in [(0, 0), (wl.B // 2, wl.H // 2), (wl.B - 1, wl.H - 1)]:
        lh = lay_np[h]
        rows, cols = lh.sum(axis=1), lh.sum(axis=0)
        qb = sorted(set(np.argsort(-rows, kind="stable")[:3].tolist() +
                        rng.choice(nb, 5, replace=False).tolist()))
        kb = set(np.argsort(-cols, kind="stable")[:1].tolist() + rng.choice(nb, 6, replace=False).tolist())
        if (cols == 0).any():
            kb.add(int(np.flatnonzero(cols == 0)[0]))
        kb = sorted(kb)
        gq, gk, gv = oracle.backward_sampled(*(t[b, h].double().numpy() for t in (q, k, v, do)), lh,
                                             wl.scale, blk, wl.causal_diag, qb, kb)
        for i in qb:
            got[0].append(dq[b, h, i * blk:(i + 1) * blk])
            ref[0].append(gq[i])
        for j in kb:
            got[1].append(dk[b, h, j * blk:(j + 1) * blk])
            ref[1].append(gk[j])
            got[2].append(dv[b, h, j * blk:(j + 1) * blk])
            ref[2].append(gv[j])
    _compare([np.stack(x) for x in got], [np.stack(x) for x in ref], parity_report,
             f"{wl.name} (full size, sampled rows of 3 heads)")
