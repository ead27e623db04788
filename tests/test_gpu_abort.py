"""The forward kernel's failure path on the GPU, driven without a fault or a hang.

``bsa_debug_expire_wait`` makes every wait at one wait site behave as a wait that ran
out.  The kernel must then record the timeout with that site's id, every role must
leave its loop, wait for its own copies and MMAs in flight, free TMEM and return;
``bsa_device_status`` reports BSA_ERR_DEVICE_TIMEOUT.  The next forward on the same
LUT with the knob off must give bitwise the same result as before the failure (no
state left behind), and that result matches the oracle.
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

SITES = [1, 2, 6, 7, 8, 9, 12]  # wait sites of both directions (reached without rescale)
EPI_SITES = [10, 13, 14]  # the forward's epilogue handoffs (128-row query blocks)
TOL_MAX, TOL_MEAN, TOL_LSE = 2e-2, 2e-3, 1e-3


@pytest.fixture(scope="module", autouse=True)
def _lib(cuda_lib):
    return cuda_lib


def _case(block, d, growing=False):
    # More items than SMs, so that CTAs change items (site 12) several times.
    B, H, nb = 2, 8, 16
    L = nb * block
    if growing:  # later key blocks score far higher: the running max moves, O is rescaled
        q, k, v = wls.randn_qkv(B, H, L, d, seed=31, dtype=torch.float32)
        for j in range(nb):
            k[:, :, j * block:(j + 1) * block] *= 1.0 + 1.5 * j
        q, k, v = (t.to(torch.bfloat16) for t in (q, k, v))
        lay = torch.tril(torch.ones(nb, nb, dtype=torch.int32))[None].repeat(H, 1, 1)
        scale = 0.3
    else:
        q, k, v = wls.randn_qkv(B, H, L, d, seed=30)
        lay = wls.random_layout(H, nb, 0.5, 40, empty_rows=1)
        scale = 1 / math.sqrt(d)
    return q, k, v, lay, scale


def _check_oracle(q, k, v, lay, scale, block, o, lse, rel=0.0):
    """Parity bars; `rel` adds a bound proportional to |O| for inputs whose scores are
    so large that attention is nearly one-hot and |O| reaches the |v| extremes, where
    the bf16 rounding of O alone is up to 2^-8 |O|."""
    ro, rl = oracle.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                            lay.numpy(), scale, block, True)
    o, lse = o.float().cpu().numpy(), lse.cpu().numpy()
    fin = np.isfinite(rl)
    assert np.array_equal(fin, np.isfinite(lse))
    dd = np.abs(o - ro)
    assert np.all(dd <= TOL_MAX + rel * np.abs(ro)) and dd.mean() <= TOL_MEAN
    assert np.abs(lse[fin] - rl[fin]).max() <= TOL_LSE * max(1.0, rel * np.abs(rl[fin]).max())


@pytest.mark.parametrize("block,d", [(128, 128), (64, 128)])
def test_expired_wait_aborts_and_recovers(block, d):
    q, k, v, lay, scale = _case(block, d)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    lut = bsa.build_lut(lay, q.shape[0])
    o0, l0 = bsa.forward(qd, kd, vd, lut, scale, block, True)
    assert lut.device_status()[0] == 0
    o0, l0 = o0.clone(), l0.clone()
    _check_oracle(q, k, v, lay, scale, block, o0, l0)
    for site in SITES + (EPI_SITES if block == 128 else []):
        lut.debug_expire_wait(site)
        bsa.forward(qd, kd, vd, lut, scale, block, True)
        st, word = lut.device_status()
        assert st == binding.BSA_ERR_DEVICE_TIMEOUT, (site, st, hex(word))
        assert word == 0x10000 | site, (site, hex(word))
        lut.debug_expire_wait(0)
        o1, l1 = bsa.forward(qd, kd, vd, lut, scale, block, True)
        assert lut.device_status()[0] == 0
        assert torch.equal(o1, o0) and torch.equal(l1, l0), site


def test_expired_rescale_wait():
    """Site 11 (O free for a rescale) is reached only when the running max moves."""
    block, d = 128, 128
    q, k, v, lay, scale = _case(block, d, growing=True)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    lut = bsa.build_lut(lay, q.shape[0])
    o0, l0 = bsa.forward(qd, kd, vd, lut, scale, block, True)
    assert lut.device_status()[0] == 0
    o0, l0 = o0.clone(), l0.clone()
    _check_oracle(q, k, v, lay, scale, block, o0, l0, rel=2.0 ** -7)
    lut.debug_expire_wait(11)
    bsa.forward(qd, kd, vd, lut, scale, block, True)
    st, word = lut.device_status()
    assert st == binding.BSA_ERR_DEVICE_TIMEOUT and word == 0x10000 | 11, hex(word)
    lut.debug_expire_wait(0)
    o1, l1 = bsa.forward(qd, kd, vd, lut, scale, block, True)
    assert lut.device_status()[0] == 0
    assert torch.equal(o1, o0) and torch.equal(l1, l0)


@pytest.mark.parametrize("block", [128, 64])
def test_backward_expired_wait_aborts_and_recovers(block):
    """The backward's kernels take the same failure path: every wait site given up on
    in turn, then a normal backward on the same LUT equals the one before."""
    d = 128
    q, k, v, lay, scale = _case(block, d)
    qd, kd, vd = (t.cuda() for t in (q, k, v))
    do = wls.randn_qkv(q.shape[0], q.shape[1], q.shape[2], d, seed=33)[0].cuda()
    lut = bsa.build_lut(lay, q.shape[0])
    o, lse = bsa.forward(qd, kd, vd, lut, scale, block, True)
    g0 = [t.clone() for t in bsa.backward(qd, kd, vd, o, lse, do, lut, scale, block, True)]
    assert lut.device_status()[0] == 0
    for site in SITES:
        lut.debug_expire_wait(site)
        bsa.backward(qd, kd, vd, o, lse, do, lut, scale, block, True)
        st, word = lut.device_status()
        assert st == binding.BSA_ERR_DEVICE_TIMEOUT, (site, st, hex(word))
        lut.debug_expire_wait(0)
        g1 = bsa.backward(qd, kd, vd, o, lse, do, lut, scale, block, True)
        assert lut.device_status()[0] == 0
        assert all(torch.equal(a, b) for a, b in zip(g0, g1)), site
