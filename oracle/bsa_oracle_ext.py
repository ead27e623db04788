"""Plain fp64 CPU oracle for the extended block-sparse forward: ragged lengths,
different query and key block sizes, and per-element predicates.

TEST INFRASTRUCTURE ONLY (same rule as ``bsa_oracle``): nothing on the product path
imports it; it shares no code with the CUDA path and depends on numpy only.

What it computes, for batch b, head h, query row r in [0, Lq) and key c in [0, Lk),
with query blocks of ``q_block`` rows and key blocks of ``kv_block`` keys
(nbq = ceil(Lq / q_block), nbk = ceil(Lk / kv_block); the last block of each side
may be short):

  A(r) = { c : layout[h, r // q_block, c // kv_block] == 1
               and not (causal_diag and key block c // kv_block overlaps the rows of
                        query block r // q_block and c > r)
               and (window_left  < 0 or c >= r - window_left)
               and (window_right < 0 or c <= r + window_right)
               and (no segment ids or q_segment[b, r] == kv_segment[b, c]) }
  s_c  = scale * <q[b,h,r,:], k[b,h,c,:]>;   with softcap > 0:  s_c = softcap * tanh(s_c / softcap)
  Z(r) = sum_{c in A(r)} exp(s_c)  (+ exp(sink[h]) when sinks are given)
  lse[r] = ln Z(r)     (-inf when Z(r) = 0, i.e. A(r) empty and no sink)
  O[r,:] = sum_{c in A(r)} exp(s_c - lse[r]) v[b,h,c,:]   (0 when A(r) is empty)

Sources (page title, then section):
  * "Block-Sparse Attention" (Sparse Attention Patterns chapter), section "Block
    Structure": the mask builder clips the last block of a ragged sequence to the
    sequence end, so blocks at the end may be shorter than the block size.
  * ejkernel blocksparse_attention (BlockSparseAttention class docstring and the
    ``run`` argument list): separate query and key block sizes (``q_blocksize``,
    ``kv_blocksize``), ``sliding_window`` as one size or a (left, right) pair,
    ``logits_soft_cap`` applied with tanh (Gemma-2 style), ``softmax_aux`` values
    added to the attention scores for attention sinks, and query / key-value
    segment ids for packed sequences.
  * DeepSeek-V4.1 "Sparse attention / Weighted row sum", the sparse_attn kernel: the
    head's learned sink adds one term to the softmax denominator and no value row,
    and a row with no valid key gives an all-zero output.

Readings (also in the design notes): the diagonal mask of ``causal_diag`` applies
in every active key block whose key range overlaps the query block's row range
(for equal block sizes, the block j == i); a window bound given as a negative number
is absent; ``softcap`` acts on the scaled score; the sink is a per-head logit that
takes part in the normaliser only, so lse includes it and an empty row's lse is the
sink.

Pinned by ``tests/test_oracle_ext.py``.
"""

from __future__ import annotations

import numpy as np


def n_blocks(length: int, block: int) -> int:
    return -(-length // block)


def lut_rect(layout, batch: int, order: str = "global"):
    """CSR + work list of a rectangular layout [H, nbq, nbk], by the same definition as
    ``bsa_oracle.oracle_lut`` (rows are the query blocks h * nbq + i, columns the active
    key blocks ascending; items {b, h, i, nnz} sorted by (-nnz, b, h, i) or
    (b, h, -nnz, i))."""
    lay = np.asarray(layout)
    if lay.ndim != 3 or not np.isin(lay, (0, 1)).all():
        raise ValueError("layout must be [H, nbq, nbk] of 0/1")
    H, nbq, _ = lay.shape
    row_ptr, col_idx, items = [0], [], []
    for h in range(H):
        for i in range(nbq):
            cols = [int(j) for j in np.nonzero(lay[h, i] == 1)[0]]
            col_idx.extend(cols)
            row_ptr.append(row_ptr[-1] + len(cols))
    for b in range(batch):
        for h in range(H):
            for i in range(nbq):
                r = h * nbq + i
                items.append((b, h, i, row_ptr[r + 1] - row_ptr[r]))
    key = (lambda t: (-t[3], t[0], t[1], t[2])) if order == "global" else \
        (lambda t: (t[0], t[1], -t[3], t[2]))
    items.sort(key=key)
    return (np.asarray(row_ptr, np.int32), np.asarray(col_idx, np.int32),
            np.asarray(items, np.int32).reshape(-1, 4))


def element_mask(layout_h, Lq: int, Lk: int, q_block: int, kv_block: int, causal_diag: bool,
                 window_left: int = -1, window_right: int = -1, q_seg=None, kv_seg=None):
    """Boolean [Lq, Lk] mask of one (batch, head): A(r) of every row r."""
    lay = np.asarray(layout_h)
    nbq, nbk = n_blocks(Lq, q_block), n_blocks(Lk, kv_block)
    if lay.shape != (nbq, nbk):
        raise ValueError(f"layout is {lay.shape}, expected {(nbq, nbk)}")
    mask = np.zeros((Lq, Lk), dtype=bool)
    for i in range(nbq):
        r0, r1 = i * q_block, min((i + 1) * q_block, Lq)
        for j in range(nbk):
            if lay[i, j] != 1:
                continue
            c0, c1 = j * kv_block, min((j + 1) * kv_block, Lk)
            mask[r0:r1, c0:c1] = True
            if causal_diag and c0 < (i + 1) * q_block and c1 > i * q_block:
                for r in range(r0, r1):
                    mask[r, max(c0, r + 1):c1] = False
    rows = np.arange(Lq)[:, None]
    cols = np.arange(Lk)[None, :]
    if window_left >= 0:
        mask &= cols >= rows - window_left
    if window_right >= 0:
        mask &= cols <= rows + window_right
    if q_seg is not None:
        mask &= np.asarray(q_seg)[:, None] == np.asarray(kv_seg)[None, :]
    return mask


def forward_ext(q, k, v, layout, scale: float, q_block: int, kv_block: int, causal_diag: bool,
                window_left: int = -1, window_right: int = -1, softcap: float = 0.0,
                sinks=None, q_seg=None, kv_seg=None):
    """The extended forward in fp64.  q [B,H,Lq,d], k/v [B,H,Lk,d], layout
    [H, nbq, nbk], sinks [H] or None, q_seg [B,Lq] / kv_seg [B,Lk] or None.
    Returns (O [B,H,Lq,d], lse [B,H,Lq])."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    lay = np.asarray(layout)
    if not np.isin(lay, (0, 1)).all():
        raise ValueError("layout values must be 0 or 1")
    if (q_seg is None) != (kv_seg is None):
        raise ValueError("give both segment-id arrays or neither")
    B, H, Lq, d = q.shape
    Lk = k.shape[2]
    out = np.zeros((B, H, Lq, v.shape[-1]))
    lse = np.full((B, H, Lq), -np.inf)
    for b in range(B):
        for h in range(H):
            mask = element_mask(lay[h], Lq, Lk, q_block, kv_block, causal_diag, window_left,
                                window_right, None if q_seg is None else q_seg[b],
                                None if kv_seg is None else kv_seg[b])
            s = scale * (q[b, h] @ k[b, h].T)
            if softcap > 0:
                s = softcap * np.tanh(s / softcap)
            for r in range(Lq):
                terms = s[r, mask[r]]
                vals = v[b, h][mask[r]]
                if sinks is not None:
                    a = float(sinks[h])
                    m = max(terms.max(), a) if terms.size else a
                    z = np.exp(terms - m).sum() + np.exp(a - m)
                elif terms.size:
                    m = terms.max()
                    z = np.exp(terms - m).sum()
                else:
                    continue  # O = 0, lse = -inf
                lse[b, h, r] = m + np.log(z)
                if terms.size:
                    out[b, h, r] = np.exp(terms - lse[b, h, r]) @ vals
    return out, lse
