"""Pins of the fp64 backward oracle against things other than itself (CPU only):
torch autograd through fp64 SDPA, central finite differences of the (pinned) forward
oracle, closed forms of the softmax Jacobian, and planted slips."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bsa_oracle as ob
from block_sparse_head_gb300 import workloads as wls

LIB_TOL = 1e-9


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _autograd_sdpa(q, k, v, do, scale, is_causal=False):
    t = [torch.from_numpy(np.ascontiguousarray(a)).requires_grad_(True) for a in (q, k, v)]
    o = F.scaled_dot_product_attention(*t, scale=scale, is_causal=is_causal)
    (o * torch.from_numpy(do)).sum().backward()
    return tuple(x.grad.numpy() for x in t)


def _err(a, b):
    return max(np.abs(x - y).max() for x, y in zip(a, b))


def pin_dense(bwd):
    B, H, nb, blk, d = 2, 2, 4, 8, 16
    L = nb * blk
    q, k, v, do = (_rand((B, H, L, d), s) for s in (1, 2, 3, 4))
    lay = np.ones((H, nb, nb), np.int32)
    return _err(bwd(q, k, v, do, lay, 0.37, blk, False), _autograd_sdpa(q, k, v, do, 0.37))


def pin_causal(bwd):
    B, H, nb, blk, d = 1, 3, 5, 4, 8
    L = nb * blk
    q, k, v, do = (_rand((B, H, L, d), s) for s in (5, 6, 7, 8))
    lay = np.tril(np.ones((nb, nb), np.int32))[None].repeat(H, 0)
    sc = 1 / math.sqrt(d)
    return _err(bwd(q, k, v, do, lay, sc, blk, True), _autograd_sdpa(q, k, v, do, sc, True))


def pin_block_diagonal(bwd):
    B, H, nb, blk, d = 2, 1, 4, 8, 8
    L = nb * blk
    q, k, v, do = (_rand((B, H, L, d), s) for s in (9, 10, 11, 12))
    lay = np.eye(nb, dtype=np.int32)[None]
    got = bwd(q, k, v, do, lay, 0.5, blk, False)
    err = 0.0
    for i in range(nb):
        sl = slice(i * blk, (i + 1) * blk)
        ref = _autograd_sdpa(q[:, :, sl], k[:, :, sl], v[:, :, sl], do[:, :, sl], 0.5)
        err = max(err, _err([g[:, :, sl] for g in got], ref))
    return err


def pin_finite_differences(bwd, seed=13):
    """Central differences of f = sum(O * do) through the forward oracle, on random
    layouts with empty rows and a causal diagonal, at randomly chosen entries."""
    B, H, nb, blk, d = 1, 2, 4, 3, 4
    L = nb * blk
    q, k, v, do = (_rand((B, H, L, d), seed + s) for s in range(4))
    lay = wls.random_layout(H, nb, 0.5, seed, empty_rows=1).numpy()
    lay[:, np.arange(nb), np.arange(nb)] = 1
    lay[0, 1] = 0  # one empty query block
    got = bwd(q, k, v, do, lay, 0.7, blk, True)

    def f(qq, kk, vv):
        return float((oracle.forward(qq, kk, vv, lay, 0.7, blk, True)[0] * do).sum())

    rng = np.random.default_rng(seed)
    eps = 1e-6
    err = 0.0
    for which in range(3):
        for _ in range(12):
            idx = tuple(int(rng.integers(0, n)) for n in q.shape)
            args = [q.copy(), k.copy(), v.copy()]
            args[which][idx] += eps
            fp = f(*args)
            args[which][idx] -= 2 * eps
            fm = f(*args)
            err = max(err, abs((fp - fm) / (2 * eps) - got[which][idx]))
    return err


@pytest.mark.parametrize("pin", [pin_dense, pin_causal, pin_block_diagonal])
def test_library_pins(pin):
    assert pin(oracle.backward) < LIB_TOL


def test_finite_differences():
    assert pin_finite_differences(oracle.backward) < 1e-7
    assert pin_finite_differences(oracle.backward, seed=29) < 1e-7


def test_jacobian_closed_forms():
    """Softmax rows sum to one and their Jacobian rows sum to zero: summed over keys,
    dV equals dO summed over the non-empty rows and dK sums to zero; empty rows get no
    dq, keys no row attends get no dk or dv."""
    B, H, nb, blk, d = 2, 2, 5, 4, 6
    L = nb * blk
    q, k, v, do = (_rand((B, H, L, d), s) for s in (20, 21, 22, 23))
    lay = wls.random_layout(H, nb, 0.45, 4, empty_rows=1).numpy()
    lay[:, :, 3] = 0  # key block 3 is never attended
    dq, dk, dv = oracle.backward(q, k, v, do, lay, 0.6, blk, True)
    for h in range(H):
        mask = oracle.expand_mask(lay[h], blk, L, True)
        live = mask.any(axis=1)
        for b in range(B):
            assert np.abs(dv[b, h].sum(0) - do[b, h][live].sum(0)).max() < 1e-12
            assert np.abs(dk[b, h].sum(0)).max() < 1e-12
            assert np.all(dq[b, h][~live] == 0)
            dead = ~mask.any(axis=0)
            assert np.all(dk[b, h][dead] == 0) and np.all(dv[b, h][dead] == 0)


def test_csc_is_the_transposed_csr():
    lay = wls.random_layout(3, 7, 0.4, 9, empty_rows=2).numpy()
    cp, ri, it = oracle.oracle_csc(lay, 2)
    rp, ci, it2 = oracle.oracle_lut(lay.transpose(0, 2, 1).copy(), 2)
    assert np.array_equal(cp, rp) and np.array_equal(ri, ci) and np.array_equal(it, it2)


# ------------------------------------------------------------ planted mistakes

def _no_delta(q, k, v, do, layout, scale, block, causal):
    """dS = P * dP (the row-sum term of the softmax Jacobian dropped)."""
    dq, dk, dv = ob.backward(q, k, v, do, layout, scale, block, causal)
    lay = ob.check_layout(layout)
    B, H, L, d = q.shape
    for h in range(H):
        mask = ob.expand_mask(lay[h], block, L, causal)
        for b in range(B):
            s = np.where(mask, scale * (q[b, h] @ k[b, h].T), -np.inf)
            m = np.where(mask.any(1), s.max(1), 0)[:, None]
            p = np.where(mask, np.exp(s - m), 0)
            p = p / np.maximum(p.sum(1, keepdims=True), 1e-300)
            ds = p * (do[b, h] @ v[b, h].T)
            dq[b, h] = scale * ds @ k[b, h]
    return dq, dk, dv


def _no_scale(*a):
    dq, dk, dv = ob.backward(*a)
    return dq / a[5], dk, dv


def _dv_untransposed(q, k, v, do, layout, scale, block, causal):
    """dV = P dO instead of P^T dO."""
    dq, dk, dv = ob.backward(q, k, v, do, layout, scale, block, causal)
    lay = ob.check_layout(layout)
    B, H, L, d = q.shape
    for h in range(H):
        mask = ob.expand_mask(lay[h], block, L, causal)
        for b in range(B):
            s = np.where(mask, scale * (q[b, h] @ k[b, h].T), -np.inf)
            m = np.where(mask.any(1), s.max(1), 0)[:, None]
            p = np.where(mask, np.exp(s - m), 0)
            p = p / np.maximum(p.sum(1, keepdims=True), 1e-300)
            dv[b, h] = p @ do[b, h]
    return dq, dk, dv


@pytest.mark.parametrize("mutant", [_no_delta, _no_scale, _dv_untransposed])
def test_pins_catch_planted_mistakes(mutant):
    errs = []
    for pin in (pin_dense, pin_causal, pin_block_diagonal, pin_finite_differences):
        try:
            errs.append(pin(mutant))
        except Exception:
            errs.append(math.inf)
    assert max(errs) > 1e-6


def test_block_restricted_equals_dense():
    """Skipping the entries outside the active blocks changes no gradient."""
    for seed, causal, blk in [(41, True, 4), (42, False, 3), (43, True, 5)]:
        B, H, nb, d = 2, 3, 5, 6
        L = nb * blk
        q, k, v, do = (_rand((B, H, L, d), seed * 10 + s) for s in range(4))
        lay = wls.random_layout(H, nb, 0.4, seed, empty_rows=1).numpy()
        lay[:, np.arange(nb), np.arange(nb)] = 1
        lay[1, 2] = 0
        a = oracle.backward(q, k, v, do, lay, 0.4, blk, causal)
        b = oracle.backward_blocks(q, k, v, do, lay, 0.4, blk, causal)
        assert _err(a, b) < 1e-12


def test_sampled_rows_equal_block_backward():
    """``backward_sampled`` returns exactly the chosen rows of ``backward_blocks``: dq of
    any query block, dk and dv of any key block (attended by many rows, by one, or by
    none), with and without the causal diagonal."""
    for seed, causal, blk in [(51, True, 4), (52, False, 3), (53, True, 5)]:
        B, H, nb, d = 2, 2, 6, 5
        L = nb * blk
        q, k, v, do = (_rand((B, H, L, d), seed * 10 + s) for s in range(4))
        lay = wls.random_layout(H, nb, 0.45, seed, empty_rows=1).numpy()
        lay[0, :, 1] = 1  # a column every row attends
        lay[1, :, 4] = 0  # a column no row attends
        full = oracle.backward_blocks(q, k, v, do, lay, 0.3, blk, causal)
        for b in range(B):
            for h in range(H):
                qb, kb = [0, 2, 5, 3], [1, 4, 0, 5]
                dq, dk, dv = oracle.backward_sampled(q[b, h], k[b, h], v[b, h], do[b, h], lay[h],
                                                     0.3, blk, causal, qb, kb)
                for i in qb:
                    assert np.abs(dq[i] - full[0][b, h, i * blk:(i + 1) * blk]).max() < 1e-12
                for j in kb:
                    assert np.abs(dk[j] - full[1][b, h, j * blk:(j + 1) * blk]).max() < 1e-12
                    assert np.abs(dv[j] - full[2][b, h, j * blk:(j + 1) * blk]).max() < 1e-12
                if h == 1:
                    assert not dk[4].any() and not dv[4].any()


def test_sampled_rows_planted_slip_fails():
    """A sampled backward that drops the delta term of dS disagrees with the pinned one."""
    blk, nb, d = 4, 5, 6
    L = nb * blk
    q, k, v, do = (_rand((L, d), 60 + s) for s in range(4))
    lay = np.tril(np.ones((nb, nb), np.int64))
    dq, dk, dv = oracle.backward_sampled(q, k, v, do, lay, 0.5, blk, True, [3], [1])
    s = 0.5 * (q[12:16] @ k[:16].T)
    s = np.where(np.arange(16)[None, :] > np.arange(12, 16)[:, None], -np.inf, s)
    p = np.exp(s - s.max(axis=1, keepdims=True))
    p /= p.sum(axis=1, keepdims=True)
    ds_wrong = p * (do[12:16] @ v[:16].T)  # no "- delta"
    assert np.abs(0.5 * ds_wrong @ k[:16] - dq[3]).max() > 1e-3
