"""Plain fp64 CPU oracle for layout-driven block-sparse multi-head attention forward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path may import or call this
module: only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` use it.  It shares no code with the CUDA
path (no kernels, headers, helpers, tables or constants); it depends on numpy only.

What it computes (the plain definition; the GPU path reaches the same result):

  For batch b, head h, query row r, with block size ``block`` and nb = L / block,
    A(r) = { c in [0, L) : layout[h, r // block, c // block] == 1
                           and not (causal_diag and r // block == c // block and c > r) }
    s_c  = scale * <q[b,h,r,:], k[b,h,c,:]>                                    (fp64)
    A(r) empty  ->  O[r,:] = 0,  lse[r] = -inf
    otherwise   ->  lse[r] = log sum_{c in A(r)} exp(s_c)   (natural log)
                    O[r,:] = sum_{c in A(r)} exp(s_c - lse[r]) * v[b,h,c,:]

Sources (page title, then section / equation):
  * "Block Sparse Attention Techniques", section 1 "Key Concepts in Attention
    Mechanisms", equation "Scaled Dot-Product Attention": softmax(Q K^T / sqrt(d_k)) V.
  * same page, section 4 "Block Sparse Attention in Large Language Models",
    the BlockSparseAttention(Q, K, V, M) equation with a binary block mask M; the
    masked logits are read as -inf (not multiplied by 0), the convention of the
    "Case Study: Longformer's Dilated Attention" equation in section 2 of the
    same page, where a masked score A_ij is -infinity.
  * "Block-Sparse Attention" (Sparse Attention Patterns chapter), section "Block
    Structure": the block layout expands to an elementwise mask by setting every
    (i*b .. (i+1)*b) x (j*b .. (j+1)*b) tile of an active block pair to True.
  * "Implementation:Deepspeedai DeepSpeed Sparse Attention Utils", section "I/O
    Contract" and "Usage Examples": the layout is int [heads x blocks_m x blocks_n]
    with 1 = compute this block and 0 = skip it.
  * DeepSeek-V4.1 "Sparse attention / Weighted row sum" page, the sparse_attn
    kernel code: a row with no valid key yields an all-zero output.
  * "Block Sparse Attention Techniques", section 3.2 "Optimizing Memory Usage with
    Block Sparsity", "Implementation with Sparse Matrix Formats": the active blocks
    are kept in compressed sparse row (CSR) form -> ``oracle_lut``.
  * "Block Sparse Attention Techniques", section 2, "Gradient Propagation in Block
    Sparse Attention": gradients flow only through the active blocks -> ``backward``,
    the gradient of the masked softmax attention above (masked entries have P = 0, so
    they pass no gradient), written out with the standard softmax Jacobian.

Readings where the pages are silent (each also listed in the design notes):
  * layout values must be exactly 0 or 1;
  * the layout is per head and shared by every batch entry;
  * ``causal_diag`` masks c > r only inside diagonal blocks (row block == column
    block); active blocks above the diagonal are not masked;
  * lse is the natural-log log-sum-exp of the *scaled* logits, -inf for an empty row;
  * CSR rows are flattened head-major (row = h * nb + i) with columns ascending;
    the work list holds one item {b, h, i, nnz} per (batch, head, query block),
    zero-count items included, stably sorted by (-nnz, b, h, i) ("global") or
    (b, h, -nnz, i) ("grouped").

Every function here is pinned by ``tests/test_oracle.py`` against library routines
(torch scaled_dot_product_attention in fp64), closed forms, invariants, brute
force loops and the cited fixtures under ``tests/golden/``.
"""

from __future__ import annotations

import numpy as np

ORDER_GLOBAL = "global"
ORDER_GROUPED = "grouped"


# --------------------------------------------------------------------------- layout


def check_layout(layout) -> np.ndarray:
    """Return the layout as an int64 array [H, nb, nb]; raise ValueError if malformed.

    Reading: the DeepSpeed utils page's I/O contract names the layout
    [heads x blocks_m x blocks_n] with 1 = compute and 0 = skip; any other value is
    rejected rather than interpreted.
    """
    lay = np.asarray(layout)
    if lay.ndim != 3 or lay.shape[1] != lay.shape[2]:
        raise ValueError(f"layout must be [H, nb, nb], got shape {lay.shape}")
    if not np.issubdtype(lay.dtype, np.integer):
        raise ValueError("layout must hold integers")
    if not np.isin(lay, (0, 1)).all():
        raise ValueError("layout values must be 0 or 1")
    return lay.astype(np.int64)


def oracle_lut(layout, batch: int, order: str = ORDER_GLOBAL):
    """CSR of active column blocks plus the (batch, head, query-block) work list.

    row_ptr[h*nb + i + 1] = row_ptr[h*nb + i] + (number of active j in row (h, i));
    col_idx lists the active j of each row in ascending order ("Block Sparse
    Attention Techniques", 3.2, CSR storage of the non-zero blocks).  The work list
    holds every (b, h, i) with its count, sorted by descending count for load
    balance; ties keep (b, h, i) order.  Returns int32 arrays
    (row_ptr [H*nb+1], col_idx [nnz], items [batch*H*nb, 4]).
    """
    lay = check_layout(layout)
    if batch < 1:
        raise ValueError("batch must be >= 1")
    if order not in (ORDER_GLOBAL, ORDER_GROUPED):
        raise ValueError(f"unknown order {order!r}")
    H, nb, _ = lay.shape
    row_ptr = [0]
    col_idx: list[int] = []
    for h in range(H):
        for i in range(nb):
            cols = [int(j) for j in np.nonzero(lay[h, i] == 1)[0]]  # ascending
            col_idx.extend(cols)
            row_ptr.append(row_ptr[-1] + len(cols))
    items = []
    for b in range(batch):
        for h in range(H):
            for i in range(nb):
                r = h * nb + i
                items.append((b, h, i, row_ptr[r + 1] - row_ptr[r]))
    if order == ORDER_GLOBAL:
        items.sort(key=lambda it: (-it[3], it[0], it[1], it[2]))
    else:
        items.sort(key=lambda it: (it[0], it[1], -it[3], it[2]))
    return (
        np.asarray(row_ptr, dtype=np.int32),
        np.asarray(col_idx, dtype=np.int32),
        np.asarray(items, dtype=np.int32).reshape(-1, 4),
    )


def expand_mask(layout_h, block: int, L: int, causal_diag: bool) -> np.ndarray:
    """Elementwise boolean mask [L, L] of one head's block layout.

    Follows the mask builder of the "Block-Sparse Attention" page (section "Block
    Structure"): each active block pair (i, j) sets the tile
    [i*block, (i+1)*block) x [j*block, (j+1)*block) to True.  With ``causal_diag``
    the entries c > r inside diagonal tiles (i == j) are then cleared.
    """
    lay = np.asarray(layout_h)
    nb = lay.shape[0]
    if nb * block != L:
        raise ValueError("L must equal nb * block")
    mask = np.zeros((L, L), dtype=bool)
    for i in range(nb):
        for j in range(nb):
            if lay[i, j] == 1:
                mask[i * block:(i + 1) * block, j * block:(j + 1) * block] = True
    if causal_diag:
        for i in range(nb):
            for rr in range(block):
                r = i * block + rr
                mask[r, r + 1:(i + 1) * block] = False
    return mask


# ------------------------------------------------------------------------ attention


def masked_attention(q, k, v, mask, scale: float):
    """Dense masked softmax attention of one (batch, head) in fp64.

    q [Lq, d], k [Lk, d], v [Lk, dv], mask [Lq, Lk] bool.  Masked logits are -inf
    before the softmax; a row with no allowed key gives O = 0 and lse = -inf.
    Returns (O [Lq, dv], lse [Lq]).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    s = scale * (q @ k.T)
    s = np.where(mask, s, -np.inf)
    out = np.zeros((q.shape[0], v.shape[1]), dtype=np.float64)
    lse = np.full(q.shape[0], -np.inf, dtype=np.float64)
    for r in range(q.shape[0]):
        if not mask[r].any():
            continue
        m = s[r].max()
        e = np.exp(s[r] - m)  # exp(-inf) = 0 on masked entries
        den = e.sum()
        lse[r] = m + np.log(den)
        out[r] = (e / den) @ v
    return out, lse


def forward_dense(q, k, v, layout, scale: float, block: int, causal_diag: bool):
    """Whole forward by materialising every head's [L, L] mask (small cases only).

    q, k, v: [B, H, L, d] arrays (any float type, computed in fp64).
    Returns (O [B, H, L, d] fp64, lse [B, H, L] fp64).
    """
    lay = check_layout(layout)
    q = np.asarray(q, dtype=np.float64)
    B, H, L, d = q.shape
    out = np.zeros((B, H, L, v.shape[-1]), dtype=np.float64)
    lse = np.zeros((B, H, L), dtype=np.float64)
    for h in range(H):
        mask = expand_mask(lay[h], block, L, causal_diag)
        for b in range(B):
            out[b, h], lse[b, h] = masked_attention(q[b, h], k[b, h], v[b, h], mask, scale)
    return out, lse


def query_block(q_bh, k_bh, v_bh, layout_h, scale: float, block: int,
                causal_diag: bool, i: int):
    """Rows [i*block, (i+1)*block) of one (batch, head), touching only active keys.

    Keys outside the active blocks carry a -inf logit, so exp() of them is 0 and
    leaving them out changes nothing (pinned against ``forward_dense``).  Returns
    (O [block, dv], lse [block]) in fp64.
    """
    lay = np.asarray(layout_h)
    nb = lay.shape[0]
    active = [j for j in range(nb) if lay[i, j] == 1]
    rows = np.arange(i * block, (i + 1) * block)
    dv = np.asarray(v_bh).shape[1]
    if not active:
        return np.zeros((block, dv)), np.full(block, -np.inf)
    cols = np.concatenate([np.arange(j * block, (j + 1) * block) for j in active])
    mask = np.ones((block, cols.size), dtype=bool)
    if causal_diag:
        mask &= ~((cols[None, :] // block == i) & (cols[None, :] > rows[:, None]))
    qb = np.asarray(q_bh)[rows].astype(np.float64)
    kb = np.asarray(k_bh)[cols].astype(np.float64)
    vb = np.asarray(v_bh)[cols].astype(np.float64)
    return masked_attention(qb, kb, vb, mask, scale)


def forward(q, k, v, layout, scale: float, block: int, causal_diag: bool):
    """Whole forward, query block by query block (mid-size cases).

    Same result as ``forward_dense`` without the [L, L] mask.  Returns
    (O [B, H, L, d] fp64, lse [B, H, L] fp64).
    """
    lay = check_layout(layout)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, H, L, d = q.shape
    nb = lay.shape[1]
    if nb * block != L:
        raise ValueError("L must equal nb * block")
    out = np.zeros((B, H, L, v.shape[-1]), dtype=np.float64)
    lse = np.zeros((B, H, L), dtype=np.float64)
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                sl = slice(i * block, (i + 1) * block)
                out[b, h, sl], lse[b, h, sl] = query_block(
                    q[b, h], k[b, h], v[b, h], lay[h], scale, block, causal_diag, i)
    return out, lse


def active_keys(layout_h, block: int, causal_diag: bool, r: int) -> np.ndarray:
    """The set A(r) of key positions query row r may attend to (ascending)."""
    lay = np.asarray(layout_h)
    i = r // block
    cols = [c for j in range(lay.shape[0]) if lay[i, j] == 1
            for c in range(j * block, (j + 1) * block)]
    if causal_diag:
        cols = [c for c in cols if not (c // block == i and c > r)]
    return np.asarray(cols, dtype=np.int64)


def block_flops(layout, batch: int, block: int, d: int) -> int:
    """Algorithmic FLOPs of one forward: 4 * block^2 * d per active block per batch.

    2*b^2*d for the b x b tile of Q K^T plus 2*b^2*d for P V; diagonal blocks
    count in full.  The block count follows the n*k*b cost of the "Block-Sparse
    Attention" page (section "Block Structure").
    """
    lay = check_layout(layout)
    return int(4 * block * block * d * int(lay.sum()) * batch)


# ------------------------------------------------------------------------- backward


def backward(q, k, v, do, layout, scale: float, block: int, causal_diag: bool):
    """Gradients (dq, dk, dv) of sum(O * do) for the forward above, in fp64.

    Per (batch, head), with P the masked softmax of the scaled scores (rows with no
    active key are all zero):
        dV = P^T dO,   dP = dO V^T,   dS = P * (dP - rowsum(P * dP)),
        dQ = scale * dS K,   dK = scale * dS^T Q.
    Masked entries have P = 0 and so pass no gradient ("Block Sparse Attention
    Techniques", section 2, gradient propagation through active blocks only).
    q, k, v, do: [B, H, L, d].  Returns (dq, dk, dv), each [B, H, L, d] fp64.
    """
    lay = check_layout(layout)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, L, d = q.shape
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for h in range(H):
        mask = expand_mask(lay[h], block, L, causal_diag)
        for b in range(B):
            s = np.where(mask, scale * (q[b, h] @ k[b, h].T), -np.inf)
            p = np.zeros((L, L))
            for r in range(L):
                if mask[r].any():
                    e = np.exp(s[r] - s[r].max())
                    p[r] = e / e.sum()
            dv[b, h] = p.T @ do[b, h]
            dp = do[b, h] @ v[b, h].T
            ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
            dq[b, h] = scale * (ds @ k[b, h])
            dk[b, h] = scale * (ds.T @ q[b, h])
    return dq, dk, dv


def backward_blocks(q, k, v, do, layout, scale: float, block: int, causal_diag: bool):
    """``backward`` computed query block by query block over the active keys only.

    Entries outside the active blocks have P = 0 and contribute nothing to any of the
    three gradients, so leaving them out changes nothing (pinned against ``backward``).
    For each query block the same formulas run on the gathered active keys; dK and dV
    rows collect the contributions of every query block that attends them."""
    lay = check_layout(layout)
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    do = np.asarray(do, dtype=np.float64)
    B, H, L, d = q.shape
    nb = lay.shape[1]
    dq, dk, dv = np.zeros_like(q), np.zeros_like(k), np.zeros_like(v)
    for b in range(B):
        for h in range(H):
            for i in range(nb):
                active = [j for j in range(nb) if lay[h, i, j] == 1]
                if not active:
                    continue
                rows = np.arange(i * block, (i + 1) * block)
                cols = np.concatenate([np.arange(j * block, (j + 1) * block) for j in active])
                mask = np.ones((block, cols.size), dtype=bool)
                if causal_diag:
                    mask &= ~((cols[None, :] // block == i) & (cols[None, :] > rows[:, None]))
                s = np.where(mask, scale * (q[b, h, rows] @ k[b, h, cols].T), -np.inf)
                e = np.exp(s - s.max(axis=1, keepdims=True))
                p = e / e.sum(axis=1, keepdims=True)
                dp = do[b, h, rows] @ v[b, h, cols].T
                ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
                dq[b, h, rows] = scale * (ds @ k[b, h, cols])
                dk[b, h, cols] += scale * (ds.T @ q[b, h, rows])
                dv[b, h, cols] += p.T @ do[b, h, rows]
    return dq, dk, dv


def backward_sampled(q_bh, k_bh, v_bh, do_bh, layout_h, scale: float, block: int,
                     causal_diag: bool, query_blocks, key_blocks):
    """Chosen rows of ``backward_blocks``'s result for one (batch, head): dq of the query
    blocks in ``query_blocks`` and dk, dv of the key blocks in ``key_blocks``, without the
    rest of the work (the full-size workloads are too large for ``backward_blocks``).

    Same source as ``backward``.  dq of query block i needs only the keys of its own
    layout row; dk and dv of key block j are sums of one term per query block i whose
    layout row lists j.  Each query block's P and dS over its active keys are formed as
    in ``backward_blocks``.  Pinned against ``backward_blocks`` in
    ``tests/test_oracle_bwd.py``.  Returns three dicts {block index: [block, d] array}."""
    lay = check_layout(np.asarray(layout_h)[None])[0]
    q = np.asarray(q_bh, dtype=np.float64)
    k = np.asarray(k_bh, dtype=np.float64)
    v = np.asarray(v_bh, dtype=np.float64)
    do = np.asarray(do_bh, dtype=np.float64)
    nb = lay.shape[0]
    d = q.shape[1]
    done = {}

    def p_ds(i):  # (rows, cols, P, dS) of query block i, or None for an empty row
        if i not in done:
            active = [j for j in range(nb) if lay[i, j] == 1]
            if not active:
                done[i] = None
            else:
                rows = np.arange(i * block, (i + 1) * block)
                cols = np.concatenate([np.arange(j * block, (j + 1) * block) for j in active])
                mask = np.ones((block, cols.size), dtype=bool)
                if causal_diag:
                    mask &= ~((cols[None, :] // block == i) & (cols[None, :] > rows[:, None]))
                s = np.where(mask, scale * (q[rows] @ k[cols].T), -np.inf)
                e = np.exp(s - s.max(axis=1, keepdims=True))
                p = e / e.sum(axis=1, keepdims=True)
                dp = do[rows] @ v[cols].T
                ds = p * (dp - (p * dp).sum(axis=1, keepdims=True))
                done[i] = (rows, cols, p, ds)
        return done[i]

    dq, dk, dv = {}, {}, {}
    for i in query_blocks:
        r = p_ds(i)
        dq[i] = np.zeros((block, d)) if r is None else scale * (r[3] @ k[r[1]])
    for j in key_blocks:
        gk, gv = np.zeros((block, d)), np.zeros((block, d))
        for i in range(nb):
            if lay[i, j] != 1:
                continue
            rows, cols, p, ds = p_ds(i)
            sel = cols // block == j
            gk += scale * (ds[:, sel].T @ q[rows])
            gv += p[:, sel].T @ do[rows]
        dk[j], dv[j] = gk, gv
    return dq, dk, dv


def oracle_csc(layout, batch: int):
    """Column view of the layout for the key-side gradients: for each (h, j) the active
    query blocks i ascending (col_ptr [H*nb+1], row_idx [nnz]) and one item
    {b, h, j, count} per (batch, head, key block), sorted by (-count, b, h, j)."""
    lay = check_layout(layout)
    H, nb, _ = lay.shape
    col_ptr = [0]
    row_idx: list[int] = []
    for h in range(H):
        for j in range(nb):
            rows = [int(i) for i in np.nonzero(lay[h, :, j] == 1)[0]]
            row_idx.extend(rows)
            col_ptr.append(col_ptr[-1] + len(rows))
    items = [(b, h, j, col_ptr[h * nb + j + 1] - col_ptr[h * nb + j])
             for b in range(batch) for h in range(H) for j in range(nb)]
    items.sort(key=lambda it: (-it[3], it[0], it[1], it[2]))
    return (np.asarray(col_ptr, np.int32), np.asarray(row_idx, np.int32),
            np.asarray(items, np.int32).reshape(-1, 4))
