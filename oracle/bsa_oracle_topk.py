"""Plain fp64 CPU oracle for top-k token-gather attention with an attention sink.

TEST INFRASTRUCTURE ONLY (same rule as ``bsa_oracle``): nothing on the product path
imports it; it shares no code with the CUDA path and depends on numpy only.

What it computes follows the sparse_attn kernel of the DeepSeek-V4.1 "Sparse attention
/ Weighted row sum" page: the key-value rows are shared by all heads (one row serves
as both key and value), each query position lists the rows it attends to, -1 marks an
unused slot, and each head's learned sink adds one term to the softmax denominator.
For batch b, position m, head h, with J(b, m) the list entries j whose index
idx[b, m, j] lies in [0, n) (a listed row counts once per listing):

    s_j    = scale * <q[b, m, h, :], kv[b, idx[b, m, j], :]>
    Z      = sum_{j in J} exp(s_j) + exp(sink[h])
    out[b, m, h, :] = sum_{j in J} exp(s_j) / Z * kv[b, idx[b, m, j], :]
    lse[b, m, h]    = ln Z

A position with no valid entry gives out = 0 (the page's kernel yields an all-zero
output there) and lse = sink[h].  Reading: an index outside [0, n) other than -1 is
treated like -1 (an unused slot).

Pinned by ``tests/test_oracle_topk.py``.
"""

from __future__ import annotations

import numpy as np


def topk_attention(q, kv, sink, idx, scale: float):
    """q [B, M, H, D], kv [B, N, D], sink [H], idx int [B, M, K]; fp64 result
    (out [B, M, H, D], lse [B, M, H])."""
    q = np.asarray(q, dtype=np.float64)
    kv = np.asarray(kv, dtype=np.float64)
    sink = np.asarray(sink, dtype=np.float64)
    idx = np.asarray(idx)
    B, M, H, D = q.shape
    N = kv.shape[1]
    out = np.zeros((B, M, H, D))
    lse = np.zeros((B, M, H))
    for b in range(B):
        for m in range(M):
            rows = [int(i) for i in idx[b, m] if 0 <= i < N]
            sel = kv[b, rows]                       # [J, D] (J may be 0)
            s = scale * (q[b, m] @ sel.T)           # [H, J]
            for h in range(H):
                top = max(s[h].max(), sink[h]) if rows else sink[h]
                e = np.exp(s[h] - top)
                z = e.sum() + np.exp(sink[h] - top)
                lse[b, m, h] = top + np.log(z)
                out[b, m, h] = (e / z) @ sel if rows else 0.0
    return out, lse


def topk_flops(H: int, D: int, N: int, idx) -> int:
    """Algorithmic FLOPs: 4 * H * D per valid listed row (scores and weighted sum)."""
    idx = np.asarray(idx)
    return int(4 * H * D * int(((idx >= 0) & (idx < N)).sum()))
