"""Pins of the top-k gather attention oracle (CPU only): fp64 SDPA with the key-value
rows shared across heads, closed forms of the sink term, the duplicate-row identity,
order invariance, plain-float loops, and planted slips."""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from oracle import bsa_oracle_topk as ot

LIB_TOL = 1e-9
EXACT_TOL = 1e-12


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _case(seed, B=2, M=3, H=4, D=8, N=11, K=6):
    rng = np.random.default_rng(seed)
    q, kv = _rand((B, M, H, D), seed), _rand((B, N, D), seed + 1)
    sink = rng.standard_normal(H)
    idx = np.stack([np.stack([rng.choice(N, K, replace=False) for _ in range(M)])
                    for _ in range(B)]).astype(np.int32)
    return q, kv, sink, idx


def pin_mqa_sdpa(fn):
    """Every row listed once and a negligible sink == dense attention whose keys and
    values are the shared rows (SDPA with one key-value head broadcast to all heads)."""
    B, M, H, D, N = 2, 5, 4, 8, 9
    q, kv = _rand((B, M, H, D), 1), _rand((B, N, D), 2)
    idx = np.tile(np.arange(N, dtype=np.int32), (B, M, 1))
    out, lse = fn(q, kv, np.full(H, -1e4), idx, 0.3)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
    qt = t(q.transpose(0, 2, 1, 3))                       # [B, H, M, D]
    kt = t(kv[:, None].repeat(H, 1))                      # [B, H, N, D]
    ref = F.scaled_dot_product_attention(qt, kt, kt, scale=0.3).numpy().transpose(0, 2, 1, 3)
    lref = torch.logsumexp(0.3 * qt @ kt.transpose(-1, -2), -1).numpy().transpose(0, 2, 1)
    return max(np.abs(out - ref).max(), np.abs(lse - lref).max())


def pin_duplicates(fn):
    """Listing every row twice equals listing it once with the sink lowered by ln 2:
    both numerator and score sum double against the same sink term."""
    q, kv, sink, idx = _case(3)
    o1, l1 = fn(q, kv, sink, np.concatenate([idx, idx], axis=2), 0.5)
    o2, l2 = fn(q, kv, sink - math.log(2), idx, 0.5)
    return max(np.abs(o1 - o2).max(), np.abs(l1 - (l2 + math.log(2))).max())


def pin_scale_zero(fn):
    """scale 0: every listed row scores 0, so out = J / (J + e^sink) * mean of the rows
    and lse = ln(J + e^sink)."""
    q, kv, sink, idx = _case(4)
    idx[0, 1, 2:] = -1  # a position with J = 2
    out, lse = fn(q, kv, sink, idx, 0.0)
    err = 0.0
    B, M, H, _ = q.shape
    for b in range(B):
        for m in range(M):
            rows = [i for i in idx[b, m] if i >= 0]
            J = len(rows)
            for h in range(H):
                want = J / (J + math.exp(sink[h])) * kv[b, rows].mean(0)
                err = max(err, np.abs(out[b, m, h] - want).max(),
                          abs(lse[b, m, h] - math.log(J + math.exp(sink[h]))))
    return err


def brute(q, kv, sink, idx, scale):
    B, M, H, D = q.shape
    N = kv.shape[1]
    out = np.zeros((B, M, H, D))
    lse = np.zeros((B, M, H))
    for b in range(B):
        for m in range(M):
            rows = [int(i) for i in idx[b, m] if 0 <= i < N]
            for h in range(H):
                sc = [scale * sum(float(q[b, m, h, x]) * float(kv[b, r, x]) for x in range(D))
                      for r in rows]
                terms = sc + [float(sink[h])]
                top = max(terms)
                z = sum(math.exp(t - top) for t in terms)
                lse[b, m, h] = top + math.log(z)
                for x in range(D):
                    out[b, m, h, x] = sum(math.exp(s - lse[b, m, h]) * float(kv[b, r, x])
                                          for s, r in zip(sc, rows))
    return out, lse


def pin_brute(fn, seed=7):
    q, kv, sink, idx = _case(seed, D=5)
    idx[0, 0, 1] = -1
    idx[1, 2, :] = -1          # a position with no valid row
    idx[1, 0, 3] = idx[1, 0, 2]  # a duplicate
    idx[0, 2, 4] = 99          # out of range: unused
    out, lse = fn(q, kv, sink, idx, 0.7)
    ro, rl = brute(q, kv, sink, idx, 0.7)
    return max(np.abs(out - ro).max(), np.abs(lse - rl).max())


def test_mqa_sdpa():
    assert pin_mqa_sdpa(ot.topk_attention) < LIB_TOL


def test_duplicates():
    assert pin_duplicates(ot.topk_attention) < EXACT_TOL


def test_scale_zero():
    assert pin_scale_zero(ot.topk_attention) < EXACT_TOL


def test_brute_force():
    assert pin_brute(ot.topk_attention) < EXACT_TOL


def test_empty_position_and_order():
    q, kv, sink, idx = _case(9)
    idx[0, 0] = -1
    out, lse = ot.topk_attention(q, kv, sink, idx, 0.4)
    assert np.all(out[0, 0] == 0) and np.abs(lse[0, 0] - sink).max() < EXACT_TOL
    perm = idx[:, :, ::-1].copy()
    o2, l2 = ot.topk_attention(q, kv, sink, perm, 0.4)
    assert np.abs(o2 - out).max() < EXACT_TOL and np.abs(l2 - lse).max() < EXACT_TOL


# --------------------------------------------------------------- planted mistakes

def _wrap_negative(q, kv, sink, idx, scale):
    """-1 read as a Python index (the last row) instead of an unused slot."""
    idx = np.where(idx < 0, kv.shape[1] - 1, idx)
    return ot.topk_attention(q, kv, sink, idx, scale)


def _no_sink(q, kv, sink, idx, scale):
    return ot.topk_attention(q, kv, np.full_like(np.asarray(sink, float), -1e4), idx, scale)


def _dedup(q, kv, sink, idx, scale):
    idx = np.asarray(idx).copy()
    for b in range(idx.shape[0]):
        for m in range(idx.shape[1]):
            seen = set()
            for j in range(idx.shape[2]):
                if idx[b, m, j] in seen:
                    idx[b, m, j] = -1
                seen.add(idx[b, m, j])
    return ot.topk_attention(q, kv, sink, idx, scale)


@pytest.mark.parametrize("mutant", [_wrap_negative, _no_sink, _dedup])
def test_pins_catch_planted_mistakes(mutant):
    errs = []
    for pin in (pin_mqa_sdpa, pin_duplicates, pin_scale_zero, pin_brute):
        try:
            errs.append(pin(mutant))
        except Exception:
            errs.append(math.inf)
    assert max(errs) > 1e-6
