"""GPU parity of bsa_forward_ext (ragged lengths, unequal query / key blocks, sliding
window, soft-cap, sinks, segment ids) against the extended fp64 oracle.

Bars as for the plain forward: max |dO| <= 2e-2, mean <= 2e-3, |dlse| <= 1e-3, and the
-inf pattern of lse exact.  The oracle runs on the same bf16-rounded inputs.
"""

import math

import numpy as np
import pytest
import torch

import block_sparse_head_gb300 as bsa
from block_sparse_head_gb300 import binding
from block_sparse_head_gb300 import workloads as wls
from oracle import bsa_oracle_ext as ox

pytestmark = pytest.mark.gpu

TOL_MAX, TOL_MEAN, TOL_LSE = 2e-2, 2e-3, 1e-3
BLOCKS = [(64, 64), (128, 128), (64, 128), (128, 64)]


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _layout(H, nbq, nbk, p, seed, qb, kb, causal):
    g = torch.Generator().manual_seed(seed)
    lay = (torch.rand(H, nbq, nbk, generator=g) < p).to(torch.int32)
    if causal:  # keep the blocks that overlap each query block's rows, so rows are not empty
        for i in range(nbq):
            for j in range(nbk):
                if j * kb < (i + 1) * qb and (j + 1) * kb > i * qb:
                    lay[:, i, j] = 1
    lay[0, nbq // 2] = 0  # an empty query block in head 0
    return lay


def _inputs(B, H, Lq, Lk, d, seed):
    g = torch.Generator().manual_seed(seed)
    q = torch.randn(B, H, Lq, d, generator=g).to(torch.bfloat16)
    k = torch.randn(B, H, Lk, d, generator=g).to(torch.bfloat16)
    v = torch.randn(B, H, Lk, d, generator=g).to(torch.bfloat16)
    return q, k, v


def _run_and_compare(q, k, v, lay, scale, qb, kb, causal, window=(-1, -1), softcap=0.0,
                     sinks=None, qseg=None, kvseg=None):
    B = q.shape[0]
    lut = bsa.build_lut(lay, B)
    dev = lambda t: None if t is None else t.cuda()  # noqa: E731
    o, lse = bsa.forward_ext(q.cuda(), k.cuda(), v.cuda(), lut, scale, qb, kb, causal,
                             window=window, softcap=softcap, sinks=dev(sinks),
                             q_segment_ids=dev(qseg), kv_segment_ids=dev(kvseg))
    st, word = lut.device_status()
    assert st == 0, hex(word)
    n = lambda t: None if t is None else t.numpy()  # noqa: E731
    ro, rl = ox.forward_ext(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                            lay.numpy(), scale, qb, kb, causal, window[0], window[1], softcap,
                            n(sinks), n(qseg), n(kvseg))
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse)), "-inf rows differ"
    assert np.all(lse[~fin] == -np.inf) and np.all(np.isfinite(o))
    d = np.abs(o - ro)
    assert d.max() <= TOL_MAX and d.mean() <= TOL_MEAN, (d.max(), d.mean())
    if fin.any():
        assert np.abs(lse[fin] - rl[fin]).max() <= TOL_LSE
    return o, lse


@pytest.mark.parametrize("qb,kb", BLOCKS)
@pytest.mark.parametrize("d", [64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_ragged_and_block_pairs(qb, kb, d, causal):
    """Lq, Lk not multiples of the blocks (self-attention lengths), every block pair."""
    B, H, L = 2, 3, 5 * 128 + 37
    lay = _layout(H, ox.n_blocks(L, qb), ox.n_blocks(L, kb), 0.4, 11, qb, kb, causal)
    q, k, v = _inputs(B, H, L, L, d, 12)
    _run_and_compare(q, k, v, lay, 1 / math.sqrt(d), qb, kb, causal)


@pytest.mark.parametrize("qb,kb", [(128, 64), (64, 128)])
def test_cross_lengths(qb, kb):
    """Lq != Lk (a shorter query sequence over a longer key sequence)."""
    B, H, Lq, Lk, d = 1, 2, 300, 777, 128
    lay = _layout(H, ox.n_blocks(Lq, qb), ox.n_blocks(Lk, kb), 0.5, 13, qb, kb, False)
    q, k, v = _inputs(B, H, Lq, Lk, d, 14)
    _run_and_compare(q, k, v, lay, 0.1, qb, kb, False)


@pytest.mark.parametrize("qb,kb", BLOCKS)
def test_sliding_window(qb, kb):
    B, H, L, d = 1, 2, 1000, 128
    nbq, nbk = ox.n_blocks(L, qb), ox.n_blocks(L, kb)
    lay = torch.ones(H, nbq, nbk, dtype=torch.int32)
    q, k, v = _inputs(B, H, L, L, d, 15)
    _run_and_compare(q, k, v, lay, 1 / math.sqrt(d), qb, kb, True, window=(200, 0))
    _run_and_compare(q, k, v, lay, 1 / math.sqrt(d), qb, kb, False, window=(37, 90))


@pytest.mark.parametrize("qb,kb", [(128, 128), (64, 64)])
def test_softcap(qb, kb):
    B, H, L, d = 1, 2, 700, 128
    lay = _layout(H, ox.n_blocks(L, qb), ox.n_blocks(L, kb), 0.6, 16, qb, kb, True)
    q, k, v = _inputs(B, H, L, L, d, 17)
    # large scores, so that the cap matters: tanh saturates
    _run_and_compare(q, k, v, lay, 0.5, qb, kb, True, softcap=5.0)
    _run_and_compare(q, k, v, lay, 0.09, qb, kb, True, softcap=30.0)


@pytest.mark.parametrize("qb,kb", [(128, 128), (64, 128)])
def test_sinks(qb, kb):
    B, H, L, d = 2, 3, 600, 64
    lay = _layout(H, ox.n_blocks(L, qb), ox.n_blocks(L, kb), 0.5, 18, qb, kb, True)
    q, k, v = _inputs(B, H, L, L, d, 19)
    sinks = torch.tensor([0.5, -2.0, 3.0], dtype=torch.float32)
    o, lse = _run_and_compare(q, k, v, lay, 1 / math.sqrt(d), qb, kb, True, sinks=sinks)
    # the empty query block of head 0 gives O = 0 and lse = the sink
    i = ox.n_blocks(L, qb) // 2
    rows = slice(i * qb, min((i + 1) * qb, L))
    assert np.all(o[:, 0, rows] == 0) and np.allclose(lse[:, 0, rows], 0.5, atol=1e-6)


@pytest.mark.parametrize("qb,kb", [(128, 128), (128, 64)])
def test_segments(qb, kb):
    """Packed documents: keys of another document are masked."""
    B, H, L, d = 2, 2, 900, 128
    lay = torch.ones(H, ox.n_blocks(L, qb), ox.n_blocks(L, kb), dtype=torch.int32)
    q, k, v = _inputs(B, H, L, L, d, 20)
    bounds = [torch.tensor([0, 130, 500, 501, 900]), torch.tensor([0, 450, 900])]
    seg = torch.zeros(B, L, dtype=torch.int32)
    for b in range(B):
        for s_, (a, e) in enumerate(zip(bounds[b][:-1], bounds[b][1:])):
            seg[b, a:e] = s_
    _run_and_compare(q, k, v, lay, 1 / math.sqrt(d), qb, kb, True, qseg=seg, kvseg=seg)


def test_everything_at_once_many_items():
    """All predicates together over more items than SMs (several items per CTA)."""
    qb, kb, d = 128, 64, 128
    B, H, L = 2, 8, 2000
    nbq, nbk = ox.n_blocks(L, qb), ox.n_blocks(L, kb)
    lay = _layout(H, nbq, nbk, 0.35, 21, qb, kb, True)
    q, k, v = _inputs(B, H, L, L, d, 22)
    g = torch.Generator().manual_seed(23)
    seg = torch.cumsum((torch.rand(B, L, generator=g) < 0.004).to(torch.int32), dim=1).to(torch.int32)
    sinks = torch.linspace(-1, 1, H, dtype=torch.float32)
    _run_and_compare(q, k, v, lay, 1 / math.sqrt(d), qb, kb, True, window=(700, 0), softcap=20.0,
                     sinks=sinks, qseg=seg, kvseg=seg)


def test_plain_arguments_take_the_plain_kernel():
    """Without predicates, equal blocks and whole blocks, the result is bitwise that of
    bsa_forward."""
    wl = wls.WORKLOADS[2]
    q, k, v = (t.cuda() for t in wls.qkv(wl))
    lay = wls.layout_for(wl)
    lut = bsa.build_lut(lay, wl.B)
    o1, l1 = bsa.forward(q, k, v, lut, wl.scale, wl.block, wl.causal_diag)
    o2, l2 = bsa.forward_ext(q, k, v, lut, wl.scale, wl.block, wl.block, wl.causal_diag)
    assert lut.device_status()[0] == 0
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_ext_argument_errors():
    lay = torch.ones(2, 3, 5, dtype=torch.int32)
    lut = bsa.build_lut(lay, 1)
    q = torch.zeros(1, 2, 300, 128, dtype=torch.bfloat16, device="cuda")
    seg = torch.zeros(1, 300, dtype=torch.int32, device="cuda")
    with pytest.raises(binding.BsaError):
        bsa.forward_ext(q, q, q, lut, 0.1, 128, 64, True, q_segment_ids=seg)  # one array only
    with pytest.raises(binding.BsaError):
        bsa.forward_ext(q, q, q, lut, 0.1, 64, 64, True)  # layout is 3 x 5, not 5 x 5
