"""C-ABI library on the CPU: exported symbols, bit-exact LUT / work list against the
oracle, and argument validation (no device work: every checked call fails before it
would touch a GPU)."""

import ctypes
import os
import re

import numpy as np
import pytest

import oracle
import block_sparse_head_gb300 as bsa
from block_sparse_head_gb300 import binding
from block_sparse_head_gb300 import workloads as wls

HEADER = os.path.join(os.path.dirname(os.path.dirname(__file__)), "include", "bsa.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(bsa.library_path()):
        from block_sparse_head_gb300 import build as b

        b.build()
    return bsa.load_library()


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(bsa_[a-z_]+)\s*\(", text)))


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(binding.EXPORTED)
    assert lib.bsa_version().decode().count(".") == 2


def test_status_strings(lib):
    for code in range(0, -11, -1):
        s = lib.bsa_status_string(code).decode()
        assert s and s != "unknown status"
    assert lib.bsa_status_string(-99).decode() == "unknown status"


def _compare(layout, batch, order):
    lut = bsa.build_lut(layout, batch, order, upload=False)
    rp, ci, it = lut.export()
    orp, oci, oit = oracle.oracle_lut(np.asarray(layout), batch, order)
    assert np.array_equal(rp, orp)
    assert np.array_equal(ci, oci)
    assert np.array_equal(it, oit)
    assert lut.nnz_total == oci.size and lut.n_items == oit.shape[0]


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
@pytest.mark.parametrize("order", ["global", "grouped"])
def test_lut_bit_exact_workloads(lib, index, order):
    wl = wls.WORKLOADS[index]
    _compare(wls.layout_for(wl).numpy(), wl.B, order)


@pytest.mark.parametrize("seed", range(6))
def test_lut_bit_exact_random(lib, seed):
    rng = np.random.default_rng(seed)
    H, nb, B = int(rng.integers(1, 5)), int(rng.integers(1, 20)), int(rng.integers(1, 4))
    lay = wls.random_layout(H, nb, float(rng.uniform(0.0, 1.0)), seed,
                            empty_rows=int(rng.integers(0, nb + 1))).numpy()
    for order in ("global", "grouped"):
        _compare(lay, B, order)


def test_lut_degenerate(lib):
    for lay in (np.zeros((2, 3, 3), np.int32), np.ones((1, 1, 1), np.int32),
                np.ones((3, 5, 5), np.int32), np.eye(7, dtype=np.int32)[None]):
        for order in ("global", "grouped"):
            _compare(lay, 2, order)


def _build_status(lib, lay, H, nb, batch, order=0):
    h = ctypes.c_void_p()
    arr = None if lay is None else np.ascontiguousarray(lay, dtype=np.int32)
    st = lib.bsa_build_lut(None if arr is None else arr.ctypes.data, H, nb, batch, order,
                           ctypes.byref(h))
    if h.value:
        lib.bsa_lut_free(h)
    return st, h.value


def test_build_lut_errors(lib):
    ones = np.ones((1, 2, 2), np.int32)
    assert _build_status(lib, None, 1, 2, 1) == (-1, None)
    assert _build_status(lib, ones, 0, 2, 1)[0] == -2
    assert _build_status(lib, ones, 1, 0, 1)[0] == -2
    assert _build_status(lib, ones, 1, 2, 0)[0] == -2
    # nb >= 2^15 is refused before the layout is read (the device records pack the row
    # count and diagonal position into 16 bits each)
    assert _build_status(lib, ones, 1, 32768, 1)[0] == -2
    assert _build_status(lib, ones, 1, 2, 1, order=7)[0] == -6
    bad = ones.copy()
    bad[0, 1, 0] = 2
    assert _build_status(lib, bad, 1, 2, 1)[0] == -3
    bad[0, 1, 0] = -1
    assert _build_status(lib, bad, 1, 2, 1)[0] == -3
    assert lib.bsa_build_lut(ones.ctypes.data, 1, 2, 1, 0, None) == -1
    with pytest.raises(binding.BsaError):
        bsa.build_lut(bad, 1, upload=False)


def test_forward_validation_before_device_work(lib):
    """Every rejected call returns before touching a device; pointers here are fake."""
    lut = bsa.build_lut(np.ones((2, 4, 4), np.int32), 1, upload=False)
    A = 1 << 20  # fake, 16-byte aligned, never dereferenced
    f = lambda **kw: lib.bsa_forward(  # noqa: E731
        kw.get("q", A), kw.get("k", A), kw.get("v", A), kw.get("lut", lut.handle),
        kw.get("out", A), kw.get("lse", A), kw.get("B", 1), kw.get("H", 2), kw.get("L", 256),
        kw.get("d", 64), ctypes.c_float(kw.get("scale", 0.125)), kw.get("block", 64),
        kw.get("causal", 0), None)
    assert f(q=None) == -1 and f(lut=None) == -1 and f(lse=None) == -1
    assert f(block=32) == -6 and f(d=96) == -6 and f(scale=float("nan")) == -6
    assert f(B=2) == -2 and f(H=3) == -2 and f(L=512) == -2
    assert f(block=128, L=256) == -2  # nb = 4 blocks of 128 != 256
    assert f(q=A + 8) == -5 and f(out=A + 2) == -5 and f(lse=A + 4) == -5
    assert f() == -9  # valid arguments, but the LUT was never uploaded
    assert lib.bsa_device_status(lut.handle, None, None) == -9
    assert lib.bsa_set_wait_limit(None, 5) == -1
    assert lib.bsa_lut_info(None, None, None, None, None, None) == -1


def _check_schedule(lut, grid, by_head=False):
    _, _, items = lut.export()
    sched, start = lut.schedule(grid, by_head)
    n = lut.n_items
    if by_head:  # hand-out order: (batch, head) ascending, list order inside each pair
        order = sorted(range(n), key=lambda k: (items[k, 0], items[k, 1], k))
        items = items[order]
    assert start[0] == 0 and start[-1] == n and np.all(np.diff(start) >= 0)
    # every work-list item exactly once; within a CTA in work-list order
    key = {tuple(r): k for k, r in enumerate(items.tolist())}
    pos = np.array([key[tuple(r)] for r in sched.tolist()], dtype=np.int64)
    assert sorted(pos.tolist()) == list(range(n))
    owner = np.empty(n, np.int64)
    for c in range(grid):
        seg = pos[start[c]:start[c + 1]]
        assert np.all(np.diff(seg) > 0)
        owner[seg] = c
    # each item went to a least-loaded CTA (lowest index on ties), replayed in list order
    cost = 4 * items[:, 3].astype(np.int64) + 2
    load = np.zeros(grid, np.int64)
    for k in range(n):
        assert owner[k] == int(np.argmin(load)), (k, owner[k], load.min())
        load[owner[k]] += cost[k]
    # list scheduling bound: the busiest CTA ends at most one item past the mean
    if n:
        assert load.max() <= cost.sum() / grid + cost.max()


@pytest.mark.parametrize("index", [1, 2, 3, 4, 5])
def test_schedule_workloads(lib, index):
    wl = wls.WORKLOADS[index]
    lut = binding.Lut(wls.layout_for(wl), wl.B)
    for grid in (1, 7, 152, lut.n_items):
        for by_head in (False, True):
            _check_schedule(lut, min(grid, lut.n_items), by_head)


@pytest.mark.parametrize("seed", range(4))
def test_schedule_random_and_errors(lib, seed):
    rng = np.random.default_rng(100 + seed)
    H, nb, B = int(rng.integers(1, 5)), int(rng.integers(1, 20)), int(rng.integers(1, 4))
    lay = wls.random_layout(H, nb, float(rng.uniform(0.0, 1.0)), seed,
                            empty_rows=int(rng.integers(0, nb + 1)))
    lut = binding.Lut(lay, B)
    for grid in sorted({1, 2, 5, lut.n_items}):
        for by_head in (False, True):
            _check_schedule(lut, grid, by_head)
    for bad in (0, -1, lut.n_items + 1):
        with pytest.raises(binding.BsaError):
            lut.schedule(bad)


def test_schedule_policy_validation(lib):
    lut = binding.Lut(np.ones((1, 2, 2), np.int32), 1)
    for policy in ("auto", "list", "by_head"):
        lut.set_schedule(policy)
    assert lib.bsa_set_schedule(lut.handle, 3) == -6   # BSA_ERR_UNSUPPORTED
    assert lib.bsa_set_schedule(None, 0) == -1         # BSA_ERR_NULL


# ------------------------------------------------ rectangular layouts (bsa_build_lut_rect)


@pytest.mark.parametrize("seed", range(4))
def test_rect_lut_bit_exact(lib, seed):
    from oracle import bsa_oracle_ext as ox

    rng = np.random.default_rng(100 + seed)
    H, nbq, nbk, B = (int(rng.integers(1, 4)), int(rng.integers(1, 12)), int(rng.integers(1, 12)),
                      int(rng.integers(1, 3)))
    lay = (rng.random((H, nbq, nbk)) < rng.uniform(0.1, 0.9)).astype(np.int32)
    lay[:, rng.integers(0, nbq)] = 0  # an empty row
    for order in ("global", "grouped"):
        lut = bsa.build_lut(lay, B, order, upload=False)
        assert (lut.nb, lut.nbk) == (nbq, nbk)
        rp, ci, it = lut.export()
        orp, oci, oit = ox.lut_rect(lay, B, order)
        assert np.array_equal(rp, orp) and np.array_equal(ci, oci) and np.array_equal(it, oit)


def test_rect_lut_oracle_matches_square_oracle():
    from oracle import bsa_oracle_ext as ox

    lay = wls.random_layout(3, 9, 0.4, 8, empty_rows=2).numpy()
    for order in ("global", "grouped"):
        for a, b in zip(ox.lut_rect(lay, 2, order), oracle.oracle_lut(lay, 2, order)):
            assert np.array_equal(a, b)


def test_forward_ext_validation(lib):
    """Argument errors of bsa_forward_ext come back before any device work."""
    lay = np.ones((2, 3, 5), np.int32)  # Lq = 3 query blocks of 128, Lk = 5 key blocks of 64
    lut = bsa.build_lut(lay, 1, upload=False)
    fake = ctypes.c_void_p(1 << 20)  # 16-byte aligned, never dereferenced

    def call(Lq=300, Lk=300, qb=128, kb=64, ext=None, d=128):
        return lib.bsa_forward_ext(fake, fake, fake, lut.handle, fake, fake, 1, 2, Lq, Lk, d,
                                   ctypes.c_float(0.1), qb, kb, 1,
                                   None if ext is None else ctypes.byref(ext), None)

    seg = binding.ExtArgs(-1, -1, 0.0, None, 1 << 20, None)
    assert call(ext=seg) == -1                                 # one segment array only
    assert call(kb=32) == -6 and call(d=96) == -6              # unsupported sizes
    assert call(ext=binding.ExtArgs(-1, -1, -1.0, None, None, None)) == -6  # negative softcap
    assert call(Lk=400) == -2 and call(Lq=500) == -2           # layout / length mismatch
    assert call() == -9                                        # valid, but never uploaded


def test_backward_validation_before_device_work(lib):
    """Argument errors of bsa_backward come back before any device work (fake pointers,
    16-byte aligned, never dereferenced)."""
    lut = bsa.build_lut(np.ones((2, 4, 4), np.int32), 1, upload=False)
    A = 1 << 20

    def f(**kw):
        ptrs = [kw.get(n, A) for n in ("q", "k", "v", "out", "lse", "dout")]
        outs = [kw.get(n, A) for n in ("dq", "dk", "dv", "delta")]
        return lib.bsa_backward(*ptrs, kw.get("lut", lut.handle), *outs, kw.get("B", 1),
                                kw.get("H", 2), kw.get("L", 256), kw.get("d", 64),
                                ctypes.c_float(kw.get("scale", 0.125)), kw.get("block", 64),
                                kw.get("causal", 1), None)

    for name in ("q", "k", "v", "out", "lse", "dout", "lut", "dq", "dk", "dv", "delta"):
        assert f(**{name: None}) == -1, name
    assert f(block=32) == -6 and f(d=96) == -6 and f(scale=float("inf")) == -6
    assert f(B=2) == -2 and f(H=3) == -2 and f(L=512) == -2 and f(L=0) == -2
    for name in ("q", "dout", "dq", "delta"):
        assert f(**{name: A + 4}) == -5, name
    assert f() == -9  # valid arguments, but the LUT was never uploaded


def test_topk_validation_before_device_work(lib):
    """Argument errors of bsa_topk_forward come back before any device work."""
    A = 1 << 20

    def f(**kw):
        return lib.bsa_topk_forward(
            kw.get("q", A), kw.get("kv", A), kw.get("sink", A), kw.get("idx", A),
            kw.get("out", A), kw.get("lse", A), kw.get("status", A), kw.get("B", 1),
            kw.get("M", 16), kw.get("N", 256), kw.get("H", 64), kw.get("D", 512),
            kw.get("K", 128), ctypes.c_float(kw.get("scale", 0.05)), None)

    for name in ("q", "kv", "sink", "idx", "out", "lse", "status"):
        assert f(**{name: None}) == -1, name
    assert f(H=32) == -6 and f(D=256) == -6 and f(scale=float("nan")) == -6
    assert f(B=0) == -2 and f(M=0) == -2 and f(N=0) == -2 and f(K=0) == -2
    assert f(M=1 << 20, B=64) == -2  # B * M * H past the int32 range
    for name in ("q", "kv", "idx", "out", "lse"):
        assert f(**{name: A + 8}) == -5, name
    assert f(status=A + 2) == -5
