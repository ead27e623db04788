"""The process-pool comparison used by the full-size GPU parity tests (CPU only).

It must see every row: an error planted in one element, one lse or one empty row's
-inf anywhere in the tensor is reported."""

import numpy as np
import torch

import oracle
from block_sparse_head_gb300 import workloads as wls
from oracle_pool import compare_full


def _case():
    B, H, nb, blk, d = 2, 3, 5, 8, 16
    L = nb * blk
    lay = wls.random_layout(H, nb, 0.4, 3, empty_rows=1)
    q, k, v = wls.randn_qkv(B, H, L, d, seed=5)
    ro, rl = oracle.forward(q.double().numpy(), k.double().numpy(), v.double().numpy(),
                            lay.numpy(), 0.3, blk, True)
    o = torch.from_numpy(ro).to(torch.bfloat16)
    lse = torch.from_numpy(rl).float()
    return q, k, v, lay, blk, o, lse


def test_pool_sees_every_row():
    q, k, v, lay, blk, o, lse = _case()
    r = compare_full(q, k, v, lay.numpy(), 0.3, blk, True, o, lse, workers=2, chunk=2)
    assert r["elements"] == o.numel() and r["rows"] == lse.numel()
    # bf16 rounding: at most half an ulp, 2^-8 of the magnitude
    assert r["max_abs"] <= 2.0 ** -8 * float(o.float().abs().max())
    assert r["inf_mismatch"] == 0 and r["nonfinite"] == 0
    assert r["lse_max"] < 1e-6

    o2 = o.clone()
    o2[1, 2, -1, -1] += 0.25  # last element of the last (batch, head)
    r2 = compare_full(q, k, v, lay.numpy(), 0.3, blk, True, o2, lse, workers=2, chunk=2)
    assert r2["max_abs"] > 0.2

    fin = torch.isfinite(lse)
    idx = fin.flatten().nonzero()[-1].item()
    l2 = lse.clone().flatten()
    l2[idx] += 0.01
    r3 = compare_full(q, k, v, lay.numpy(), 0.3, blk, True, o, l2.view_as(lse), workers=2, chunk=2)
    assert r3["lse_max"] > 0.009

    empty = (~fin).flatten().nonzero()[0].item()
    l3 = lse.clone().flatten()
    l3[empty] = 0.0  # an empty row that claims a finite lse
    r4 = compare_full(q, k, v, lay.numpy(), 0.3, blk, True, o, l3.view_as(lse), workers=2, chunk=2)
    assert r4["inf_mismatch"] == 1

    o3 = o.clone()
    o3[0, 0, 3, 2] = float("nan")
    r5 = compare_full(q, k, v, lay.numpy(), 0.3, blk, True, o3, lse, workers=2, chunk=2)
    assert r5["nonfinite"] == 1
