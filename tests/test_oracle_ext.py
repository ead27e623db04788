"""Pins of the extended oracle (ragged lengths, q_block != kv_block, sliding window,
soft-cap, sinks, segment ids) against things other than itself (CPU only).

Each pin is a library routine (torch SDPA in fp64 with a boolean mask), a closed form,
a limit, or per-element loops in plain Python floats on tiny inputs; the last test
plants plausible slips in a copy of the oracle and checks that some pin catches each.
"""

import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

import oracle
from oracle import bsa_oracle_ext as ox

LIB_TOL = 1e-9     # fp64 library reductions (threaded) against the oracle
EXACT_TOL = 1e-12  # closed forms and plain-float loops


def _rand(shape, seed):
    return np.random.default_rng(seed).standard_normal(shape)


def _sdpa(q, k, v, scale, mask=None, is_causal=False):
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a))  # noqa: E731
    m = None if mask is None else t(mask)
    return F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=m, scale=scale,
                                          is_causal=is_causal).numpy()


def _lse_masked(q, k, scale, mask=None):
    s = torch.from_numpy(scale * np.einsum("bhqd,bhkd->bhqk", q, k))
    if mask is not None:
        s = s.masked_fill(~torch.from_numpy(mask), float("-inf"))
    return torch.logsumexp(s, dim=-1).numpy()


def _lower_blocks(nbq, nbk, qb, kb):
    """Key block j active for query block i when it starts at or before the block's last row."""
    lay = np.zeros((nbq, nbk), np.int32)
    for i in range(nbq):
        for j in range(nbk):
            lay[i, j] = int(j * kb <= (i + 1) * qb - 1)
    return lay


# ------------------------------------------------------------- library reductions


def pin_dense_ragged(fwd):
    """All-ones layout over ragged lengths (Lq, Lk not multiples of the blocks)
    == dense attention."""
    B, H, Lq, Lk, d, qb, kb = 2, 2, 37, 53, 8, 8, 16
    q, k, v = _rand((B, H, Lq, d), 1), _rand((B, H, Lk, d), 2), _rand((B, H, Lk, d), 3)
    lay = np.ones((H, ox.n_blocks(Lq, qb), ox.n_blocks(Lk, kb)), np.int32)
    o, lse = fwd(q, k, v, lay, 0.4, qb, kb, False)
    return max(np.abs(o - _sdpa(q, k, v, 0.4)).max(), np.abs(lse - _lse_masked(q, k, 0.4)).max())


def pin_causal_blocks(fwd, qb=8, kb=4):
    """Block-lower layout + causal_diag over a ragged length, any block pair == causal
    dense attention."""
    B, H, L, d = 1, 2, 45, 8
    q, k, v = (_rand((B, H, L, d), s) for s in (4, 5, 6))
    lay = _lower_blocks(ox.n_blocks(L, qb), ox.n_blocks(L, kb), qb, kb)[None].repeat(H, 0)
    o, lse = fwd(q, k, v, lay, 0.35, qb, kb, True)
    tri = np.tril(np.ones((L, L), bool))
    return max(np.abs(o - _sdpa(q, k, v, 0.35, is_causal=True)).max(),
               np.abs(lse - _lse_masked(q, k, 0.35, tri)).max())


def pin_window_segments(fwd):
    """All-ones layout + window (3, 2) + packed documents == dense attention under the
    band-and-same-document mask."""
    B, H, L, d, qb, kb = 2, 1, 40, 8, 8, 8
    q, k, v = (_rand((B, H, L, d), s) for s in (7, 8, 9))
    seg = np.stack([np.repeat([0, 1, 2], [11, 17, 12]), np.repeat([5, 6], [23, 17])])
    lay = np.ones((H, 5, 5), np.int32)
    o, lse = fwd(q, k, v, lay, 0.5, qb, kb, False, window_left=3, window_right=2,
                 q_seg=seg, kv_seg=seg)
    err = 0.0
    r = np.arange(L)[:, None]
    c = np.arange(L)[None, :]
    for b in range(B):
        m = (c >= r - 3) & (c <= r + 2) & (seg[b][:, None] == seg[b][None, :])
        mm = m[None, None]
        err = max(err, np.abs(o[b:b + 1] - _sdpa(q[b:b + 1], k[b:b + 1], v[b:b + 1], 0.5, mm)).max(),
                  np.abs(lse[b:b + 1] - _lse_masked(q[b:b + 1], k[b:b + 1], 0.5, mm)).max())
    return err


def test_dense_ragged_is_sdpa():
    assert pin_dense_ragged(ox.forward_ext) < LIB_TOL


@pytest.mark.parametrize("qb,kb", [(8, 4), (4, 8), (8, 8)])
def test_causal_blocks_is_causal_sdpa(qb, kb):
    assert pin_causal_blocks(ox.forward_ext, qb, kb) < LIB_TOL


def test_window_and_segments_are_masked_sdpa():
    assert pin_window_segments(ox.forward_ext) < LIB_TOL


def test_plain_case_equals_main_oracle():
    """Without any extension (equal blocks, whole blocks) it is the main oracle's forward."""
    B, H, nb, blk, d = 2, 2, 5, 4, 8
    L = nb * blk
    q, k, v = (_rand((B, H, L, d), s) for s in (10, 11, 12))
    lay = (np.random.default_rng(3).random((H, nb, nb)) < 0.5).astype(np.int32)
    lay[0, 2] = 0
    for causal in (False, True):
        o1, l1 = ox.forward_ext(q, k, v, lay, 0.3, blk, blk, causal)
        o2, l2 = oracle.forward(q, k, v, lay, 0.3, blk, causal)
        assert np.abs(o1 - o2).max() < EXACT_TOL
        assert np.array_equal(np.isfinite(l1), np.isfinite(l2))
        fin = np.isfinite(l1)
        assert np.abs(l1[fin] - l2[fin]).max() < EXACT_TOL


# ------------------------------------------------------------ closed forms, limits


def test_window_zero_is_identity():
    """Window (0, 0): a row attends to itself only, so O = v[r] and lse = s_rr."""
    B, H, L, d = 1, 2, 19, 6
    q, k, v = (_rand((B, H, L, d), s) for s in (13, 14, 15))
    lay = np.ones((H, 5, 5), np.int32)
    o, lse = ox.forward_ext(q, k, v, lay, 0.7, 4, 4, True, window_left=0, window_right=0)
    assert np.abs(o - v).max() < EXACT_TOL
    assert np.abs(lse - 0.7 * np.einsum("bhld,bhld->bhl", q, k)).max() < EXACT_TOL


def test_softcap_limits():
    """softcap -> infinity leaves the scores unchanged; softcap -> 0 flattens them to 0,
    so O is the mean of the active value rows and lse = ln |A(r)|."""
    B, H, L, d, blk = 1, 2, 24, 5, 8
    q, k, v = (_rand((B, H, L, d), s) for s in (16, 17, 18))
    lay = np.tril(np.ones((3, 3), np.int32))[None].repeat(H, 0)
    o0, l0 = ox.forward_ext(q, k, v, lay, 0.6, blk, blk, True)
    o1, l1 = ox.forward_ext(q, k, v, lay, 0.6, blk, blk, True, softcap=1e9)
    assert np.abs(o1 - o0).max() < 1e-9 and np.abs(l1 - l0).max() < 1e-9
    o2, l2 = ox.forward_ext(q, k, v, lay, 0.6, blk, blk, True, softcap=1e-14)
    for r in range(L):
        n = r + 1  # causal over a block-lower-triangular layout: keys 0..r
        assert np.abs(o2[:, :, r] - v[:, :, :n].mean(2)).max() < EXACT_TOL
        assert np.abs(l2[:, :, r] - math.log(n)).max() < EXACT_TOL


def test_sink_closed_forms():
    """A very negative sink changes nothing; with scale 0 and sink a, O is
    n/(n + e^a) times the mean of the n active rows and lse = ln(n + e^a); an empty row
    gives O = 0 and lse = a."""
    B, H, L, d, blk = 1, 2, 16, 4, 4
    q, k, v = (_rand((B, H, L, d), s) for s in (19, 20, 21))
    lay = np.ones((H, 4, 4), np.int32)
    lay[1, 2] = 0  # rows 8..11 of head 1 have no active block
    o0, l0 = ox.forward_ext(q, k, v, lay, 0.5, blk, blk, False)
    o1, l1 = ox.forward_ext(q, k, v, lay, 0.5, blk, blk, False, sinks=np.array([-1e4, -1e4]))
    assert np.abs(o1 - o0).max() < EXACT_TOL
    fin = np.isfinite(l0)
    assert np.abs(l1[fin] - l0[fin]).max() < EXACT_TOL
    assert np.all(l1[~fin] == -1e4)  # an empty row's normaliser is the sink term alone
    a = np.array([0.3, -1.2])
    o2, l2 = ox.forward_ext(q, k, v, lay, 0.0, blk, blk, False, sinks=a)
    for h in range(H):
        for r in range(L):
            if h == 1 and 8 <= r < 12:
                assert np.all(o2[0, h, r] == 0) and abs(l2[0, h, r] - a[h]) < EXACT_TOL
                continue
            n = L
            want = n / (n + math.exp(a[h])) * v[0, h].mean(0)
            assert np.abs(o2[0, h, r] - want).max() < EXACT_TOL
            assert abs(l2[0, h, r] - math.log(n + math.exp(a[h]))) < EXACT_TOL


def test_equal_segments_change_nothing():
    B, H, L, d, blk = 2, 1, 12, 4, 4
    q, k, v = (_rand((B, H, L, d), s) for s in (22, 23, 24))
    lay = np.ones((H, 3, 3), np.int32)
    seg = np.full((B, L), 7)
    o0, l0 = ox.forward_ext(q, k, v, lay, 0.5, blk, blk, True)
    o1, l1 = ox.forward_ext(q, k, v, lay, 0.5, blk, blk, True, q_seg=seg, kv_seg=seg)
    assert np.abs(o1 - o0).max() < EXACT_TOL and np.abs(l1 - l0).max() < EXACT_TOL


# --------------------------------------------------------------------- brute force


def brute_force_ext(q, k, v, lay, scale, qb, kb, causal, wl, wr, cap, sinks, qs, ks):
    """Per-element loops in plain Python floats."""
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    o = np.zeros((B, H, Lq, d))
    lse = np.full((B, H, Lq), -math.inf)
    for b in range(B):
        for h in range(H):
            for r in range(Lq):
                keys = []
                for c in range(Lk):
                    i, j = r // qb, c // kb
                    if lay[h][i][j] != 1:
                        continue
                    overlaps = j * kb < (i + 1) * qb and (j + 1) * kb > i * qb
                    if causal and overlaps and c > r:
                        continue
                    if wl >= 0 and c < r - wl:
                        continue
                    if wr >= 0 and c > r + wr:
                        continue
                    if qs is not None and qs[b][r] != ks[b][c]:
                        continue
                    keys.append(c)
                sc = {}
                for c in keys:
                    acc = 0.0
                    for x in range(d):
                        acc += float(q[b, h, r, x]) * float(k[b, h, c, x])
                    s = scale * acc
                    sc[c] = cap * math.tanh(s / cap) if cap > 0 else s
                vals = list(sc.values()) + ([float(sinks[h])] if sinks is not None else [])
                if not vals:
                    continue
                mx = max(vals)
                tot = sum(math.exp(x - mx) for x in vals)
                lse[b, h, r] = mx + math.log(tot)
                for x in range(d):
                    o[b, h, r, x] = sum(math.exp(sc[c] - lse[b, h, r]) * float(v[b, h, c, x])
                                        for c in keys)
    return o, lse


def pin_brute_ext(fwd, seed=31):
    B, H, Lq, Lk, d, qb, kb = 2, 2, 15, 13, 3, 4, 2
    q, k, v = _rand((B, H, Lq, d), seed), _rand((B, H, Lk, d), seed + 1), _rand((B, H, Lk, d), seed + 2)
    rng = np.random.default_rng(seed)
    lay = (rng.random((H, ox.n_blocks(Lq, qb), ox.n_blocks(Lk, kb))) < 0.6).astype(np.int32)
    lay[0, 1] = 0  # an empty query block
    qs = rng.integers(0, 2, (B, Lq))
    ks = rng.integers(0, 2, (B, Lk))
    sinks = np.array([0.4, -0.8])
    args = (0.9, qb, kb, True, 4, 1, 1.5, sinks, qs, ks)
    o, lse = fwd(q, k, v, lay, *args[:4], window_left=args[4], window_right=args[5],
                 softcap=args[6], sinks=sinks, q_seg=qs, kv_seg=ks)
    ro, rl = brute_force_ext(q, k, v, lay, *args)
    fin = np.isfinite(rl)
    if not np.array_equal(fin, np.isfinite(lse)):
        return math.inf
    return max(np.abs(o - ro).max(), np.abs(lse[fin] - rl[fin]).max() if fin.any() else 0.0)


def test_brute_force_all_features():
    assert pin_brute_ext(ox.forward_ext) < EXACT_TOL
    assert pin_brute_ext(ox.forward_ext, seed=41) < EXACT_TOL


# ------------------------------------------------------------ planted mistakes


def _mutant(mask_fn=None, post=None):
    def fwd(*a, **kw):
        saved = ox.element_mask
        try:
            if mask_fn is not None:
                ox.element_mask = mask_fn
            o, lse = saved_forward(*a, **kw)
            return post(o, lse, kw) if post else (o, lse)
        finally:
            ox.element_mask = saved
    return fwd


saved_forward = ox.forward_ext
saved_mask = ox.element_mask


def _window_off_by_one(layout_h, Lq, Lk, qb, kb, causal, wl=-1, wr=-1, qs=None, ks=None):
    return saved_mask(layout_h, Lq, Lk, qb, kb, causal, wl + 1 if wl >= 0 else wl, wr, qs, ks)


def _causal_everywhere(layout_h, Lq, Lk, qb, kb, causal, wl=-1, wr=-1, qs=None, ks=None):
    m = saved_mask(layout_h, Lq, Lk, qb, kb, False, wl, wr, qs, ks)
    if causal:
        m &= np.tril(np.ones((Lq, Lk), bool))
    return m


def _causal_same_index_only(layout_h, Lq, Lk, qb, kb, causal, wl=-1, wr=-1, qs=None, ks=None):
    """Diagonal read as block j == i even when the block sizes differ."""
    m = saved_mask(layout_h, Lq, Lk, qb, kb, False, wl, wr, qs, ks)
    if causal:
        for r in range(Lq):
            for c in range(Lk):
                if r // qb == c // kb and c > r:
                    m[r, c] = False
    return m


def _segments_ignored(layout_h, Lq, Lk, qb, kb, causal, wl=-1, wr=-1, qs=None, ks=None):
    return saved_mask(layout_h, Lq, Lk, qb, kb, causal, wl, wr, None, None)


def _drop_sink_from_lse(o, lse, kw):
    return o, lse if kw.get("sinks") is None else lse + 0.01


@pytest.mark.parametrize("mutant", [
    _mutant(mask_fn=_window_off_by_one),
    _mutant(mask_fn=_causal_everywhere),
    _mutant(mask_fn=_causal_same_index_only),
    _mutant(mask_fn=_segments_ignored),
    _mutant(post=_drop_sink_from_lse),
])
def test_pins_catch_planted_mistakes(mutant):
    errs = []
    for pin in (pin_dense_ragged, pin_causal_blocks, pin_window_segments, pin_brute_ext):
        try:
            errs.append(pin(mutant))
        except Exception:
            errs.append(math.inf)
    assert max(errs) > 1e-6
