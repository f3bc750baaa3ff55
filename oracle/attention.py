"""Plain double-precision attention: the definition, written out.

TEST INFRASTRUCTURE ONLY (see the package docstring): the library never
imports this module.

Shapes (all numpy float64, C-contiguous is not required):
    q, do, o, dq : [B, Hq, N, d]
    k, v, dk, dv : [B, Hkv, N, d]        Hq % Hkv == 0, G = Hq // Hkv
    lse, D       : [B, Hq, N]
Query head h reads key/value head h // G (grouped-query attention; the
Llama-2-70B-shaped workload maps 64 query heads onto 8 KV heads this way).

Causal convention: key j is visible to query i iff j <= i (the pages skip the
blocks whose key index exceeds the query index). Every function but
`backward_query_rows` and `tiled_forward` also takes keys of another length Nk
than the Nq queries
(k, v: [B, Hkv, Nk, d]); the queries are then the last Nq positions of the Nk
(bottom-right alignment): key j is visible to query i iff j <= i + (Nk - Nq),
so with Nq > Nk the first Nq - Nk query rows see no key.

A library matmul serves as the inner-product step. Rows are independent, so
computing several whole rows at once is not a change of arithmetic: no row's
max, sum or product is ever split into partial pieces, except in
`tiled_forward`, whose whole purpose is to restate the pages' tiled algorithm.
"""
from concurrent.futures import ThreadPoolExecutor

import numpy as np

# Granularity of a block mask: one 128 x 128 tile of the tiled algorithm
# ("FlashAttention技术解析" section 6.2 skips whole blocks the same way the
# causal mask skips the blocks above the diagonal).
BLOCK = 128


def _check(q, k, v):
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, Hq, N, d = q.shape
    if k.shape[0] != B or k.shape[2] != N or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, N, d] matching q")
    Hkv = k.shape[1]
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, N, d, Hq // Hkv


def _check_qk(q, k, v):
    """As _check, but k and v may hold Nk != Nq positions."""
    if q.ndim != 4 or k.ndim != 4 or v.ndim != 4:
        raise ValueError("q, k, v must be [B, H, N, d]")
    B, Hq, Nq, d = q.shape
    if k.shape[0] != B or k.shape[3] != d or v.shape != k.shape:
        raise ValueError("k and v must be [B, Hkv, Nk, d] matching q")
    Hkv, Nk = k.shape[1], k.shape[2]
    if Hkv <= 0 or Hq % Hkv != 0:
        raise ValueError("Hq must be a multiple of Hkv")
    return B, Hq, Hkv, Nq, Nk, d, Hq // Hkv


def _scores(qh, kh, scale, causal, row_index, block_mask_bh=None, off=0):
    """S = scale * q k^T for the given query rows against all keys, with the
    causal mask applied as -inf (definition; blogweb.cn section 1).

    qh: [R, d] query rows whose absolute indices are row_index [R]; kh: [Nk, d].
    Causal: key j visible to query i iff j <= i + off, off = Nk - Nq.
    block_mask_bh: optional [nq, nk] booleans; key j is visible to query i only
    if block_mask_bh[i // BLOCK, j // BLOCK] (and the causal rule holds).
    """
    s = scale * (qh @ kh.T)
    key_index = np.arange(kh.shape[0])
    if causal:
        s = np.where(key_index[None, :] <= row_index[:, None] + off, s, -np.inf)
    if block_mask_bh is not None:
        allowed = np.asarray(block_mask_bh, dtype=bool)[row_index[:, None] // BLOCK, key_index[None, :] // BLOCK]
        s = np.where(allowed, s, -np.inf)
    return s


def _softmax_rows(s):
    """Row-wise softmax and natural-log logsumexp of one whole score row at a
    time. The row max is subtracted before exp (numerical-stability advice,
    mhpq.cn section 7). A row with no visible key (possible only under a block
    mask) has P = 0 and LSE = -inf, so its output is 0."""
    vis = np.isfinite(s).any(axis=1)
    m = np.where(vis, s.max(axis=1), 0.0)
    e = np.exp(s - m[:, None])
    with np.errstate(divide="ignore"):
        lse = np.where(vis, m + np.log(np.where(vis, e.sum(axis=1), 1.0)), -np.inf)
    p = np.where(vis[:, None], np.exp(s - np.where(vis, lse, 0.0)[:, None]), 0.0)
    return p, lse


def _block_mask_bh(block_mask, B, Hq, N):
    """Broadcast an optional block mask to [B, Hq, nq, nk] booleans."""
    if block_mask is None:
        return None
    n = (N + BLOCK - 1) // BLOCK
    return np.broadcast_to(np.asarray(block_mask, dtype=bool), (B, Hq, n, n))


def forward(q, k, v, causal, scale, block_mask=None):
    """O = softmax(scale * Q K^T [+ causal mask]) V and LSE = logsumexp of the
    scaled, masked logits per query row (natural log).

    The forward stores only O and the per-row normaliser (aiknowledge.cn FA3
    section 3); LSE is that normaliser in log form. block_mask: optional
    booleans broadcastable to [B, Hq, ceil(N/128), ceil(N/128)] (see _scores).
    Returns (o [B,Hq,N,d], lse [B,Hq,N]).
    """
    B, Hq, Hkv, N, Nk, d, G = _check_qk(q, k, v)
    if block_mask is not None and Nk != N:
        raise ValueError("block masks need Nq == Nk")
    bm = _block_mask_bh(block_mask, B, Hq, N)
    o = np.empty((B, Hq, N, d))
    lse = np.empty((B, Hq, N))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            s = _scores(q[b, h], k[b, hk], scale, causal, rows, None if bm is None else bm[b, h], Nk - N)
            p, lse[b, h] = _softmax_rows(s)
            o[b, h] = p @ v[b, hk]
    return o, lse


def backward(q, k, v, do, causal, scale, block_mask=None):
    """Gradients of L = <O, dO> with respect to Q, K and V.

    The pages only say that the backward recomputes from the stored
    normaliser (aiknowledge.cn FA3 section 3; deepschool.ru "Улучшение
    backward pass"); the derivatives are the textbook ones of softmax:
        P = exp(S - LSE),  D_i = sum_c dO_ic O_ic,  dP = dO V^T,
        dS = P * (dP - D),  dQ = scale dS K,  dK = scale dS^T Q,  dV = P^T dO,
    with dK and dV summed over the G query heads that share a KV head.
    block_mask as in `forward`; a row with no visible key has dQ = 0 and adds
    nothing to dK or dV.
    Returns (o, lse, dq, dk, dv).
    """
    B, Hq, Hkv, N, Nk, d, G = _check_qk(q, k, v)
    if block_mask is not None and Nk != N:
        raise ValueError("block masks need Nq == Nk")
    bm = _block_mask_bh(block_mask, B, Hq, N)
    o = np.empty((B, Hq, N, d))
    lse = np.empty((B, Hq, N))
    dq = np.empty((B, Hq, N, d))
    dk = np.zeros((B, Hkv, Nk, d))
    dv = np.zeros((B, Hkv, Nk, d))
    rows = np.arange(N)
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            s = _scores(q[b, h], k[b, hk], scale, causal, rows, None if bm is None else bm[b, h], Nk - N)
            p, lse[b, h] = _softmax_rows(s)
            o[b, h] = p @ v[b, hk]
            D = (do[b, h] * o[b, h]).sum(axis=1)
            dp = do[b, h] @ v[b, hk].T
            ds = p * (dp - D[:, None])
            dq[b, h] = scale * (ds @ k[b, hk])
            dk[b, hk] += scale * (ds.T @ q[b, h])
            dv[b, hk] += p.T @ do[b, h]
    return o, lse, dq, dk, dv


def forward_rows(q, k, v, causal, scale, rows, block_mask=None):
    """O and LSE for selected query rows only (each row costs O(N d)).

    rows: int array [B, Hq, R] of query indices per head; block_mask as in
    `forward`.
    Returns (o [B,Hq,R,d], lse [B,Hq,R]).
    """
    B, Hq, Hkv, N, Nk, d, G = _check_qk(q, k, v)
    if block_mask is not None and Nk != N:
        raise ValueError("block masks need Nq == Nk")
    bm = _block_mask_bh(block_mask, B, Hq, N)
    R = rows.shape[2]
    o = np.empty((B, Hq, R, d))
    lse = np.empty((B, Hq, R))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            r = rows[b, h]
            s = _scores(q[b, h, r], k[b, hk], scale, causal, r, None if bm is None else bm[b, h], Nk - N)
            p, lse[b, h] = _softmax_rows(s)
            o[b, h] = p @ v[b, hk]
    return o, lse


def _slab_keys(rows, Nk, causal, off, bm_bh):
    """Keys that at least one of the given query rows may see: under the
    causal rule none past (last row + off); under a block mask only the key
    tiles some row's query tile may see. Every other key is masked for every
    row of the slab (exp(-inf) = 0), so leaving it out changes no result."""
    keys = np.arange(Nk)
    if causal:
        keys = keys[keys <= rows[-1] + off]
    if bm_bh is not None:
        tiles = np.asarray(bm_bh, dtype=bool)[np.unique(rows // BLOCK)].any(axis=0)
        keys = keys[tiles[keys // BLOCK]]
    return keys


def _scores_on(qh, kh, scale, causal, row_index, key_index, block_mask_bh=None, off=0):
    """As _scores, for the keys `key_index` only (absolute indices into kh)."""
    s = scale * (qh @ kh[key_index].T)
    if causal:
        s = np.where(key_index[None, :] <= row_index[:, None] + off, s, -np.inf)
    if block_mask_bh is not None:
        allowed = np.asarray(block_mask_bh, dtype=bool)[row_index[:, None] // BLOCK, key_index[None, :] // BLOCK]
        s = np.where(allowed, s, -np.inf)
    return s


def row_statistics(q, k, v, do, causal, scale, block=1024, threads=None, block_mask=None):
    """LSE_i and D_i = dO_i . O_i for EVERY query row, in double.

    Needed to check sampled key rows of dK/dV at lengths where the full score
    matrix does not fit: a key row's gradient sums over all query rows that
    see it, each weighted by that row's own LSE and D. The values come from
    this oracle alone, never from the GPU. Whole rows are computed together in
    batches of `block`; no row is split. Keys may be longer than queries
    (k, v: [B, Hkv, Nk, d]; bottom-right causal rule, as in `forward`), and
    block_mask is as in `forward` (Nq == Nk). A row that sees no key has
    LSE = -inf and D = 0 (its O is 0).
    Returns (lse [B,Hq,N], D [B,Hq,N]).
    """
    B, Hq, Hkv, N, Nk, d, G = _check_qk(q, k, v)
    if block_mask is not None and Nk != N:
        raise ValueError("block masks need Nq == Nk")
    bm = _block_mask_bh(block_mask, B, Hq, N)
    off = Nk - N
    lse = np.empty((B, Hq, N))
    D = np.empty((B, Hq, N))
    jobs = [(b, h, r0) for b in range(B) for h in range(Hq) for r0 in range(0, N, block)]

    def run(job):
        b, h, r0 = job
        hk = h // G
        r = np.arange(r0, min(r0 + block, N))
        bmh = None if bm is None else bm[b, h]
        keys = _slab_keys(r, Nk, causal, off, bmh)
        if keys.size == 0:
            lse[b, h, r] = -np.inf
            D[b, h, r] = 0.0
            return
        s = _scores_on(q[b, h, r], k[b, hk], scale, causal, r, keys, bmh, off)
        p, lse_r = _softmax_rows(s)
        o_r = p @ v[b, hk, keys]
        lse[b, h, r] = lse_r
        D[b, h, r] = (do[b, h, r] * o_r).sum(axis=1)

    with ThreadPoolExecutor(max_workers=threads) as ex:
        list(ex.map(run, jobs))
    return lse, D


def backward_rows(q, k, v, do, causal, scale, q_rows, k_rows, lse, D, block_mask=None):
    """dQ for selected query rows and dK, dV for selected key rows.

    q_rows: [B, Hq, R] query indices; k_rows: [B, Hkv, R2] key indices.
    lse, D: full per-row statistics [B, Hq, N] from `row_statistics` (or
    `backward`), i.e. the oracle's own values.
        dQ_i = scale sum_j P_ij (dP_ij - D_i) K_j
        dK_j = scale sum_{h in group} sum_i P_ij (dP_ij - D_i) Q_i
        dV_j = sum_{h in group} sum_i P_ij dO_i
    with P_ij = exp(S_ij - LSE_i) over the visible (i, j) and 0 elsewhere, and
    dP_ij = dO_i . V_j (see `backward`). Keys may be longer than queries
    (bottom-right causal rule) and block_mask is as in `forward`; a query row
    that sees no key (LSE = -inf) has dQ = 0 and adds nothing to dK, dV.
    Returns (dq [B,Hq,R,d], dk [B,Hkv,R2,d], dv [B,Hkv,R2,d]).
    """
    B, Hq, Hkv, N, Nk, d, G = _check_qk(q, k, v)
    if block_mask is not None and Nk != N:
        raise ValueError("block masks need Nq == Nk")
    bm = _block_mask_bh(block_mask, B, Hq, N)
    off = Nk - N
    all_rows = np.arange(N)
    dq = np.empty((B, Hq, q_rows.shape[2], d))
    dk = np.zeros((B, Hkv, k_rows.shape[2], d))
    dv = np.zeros((B, Hkv, k_rows.shape[2], d))

    def probs(s, lse_rows):
        seen = np.isfinite(lse_rows)
        return np.where(seen[:, None], np.exp(s - np.where(seen, lse_rows, 0.0)[:, None]), 0.0)

    for b in range(B):
        for h in range(Hq):
            hk = h // G
            bmh = None if bm is None else bm[b, h]
            r = q_rows[b, h]
            s = _scores(q[b, h, r], k[b, hk], scale, causal, r, bmh, off)
            p = probs(s, lse[b, h, r])
            dp = do[b, h, r] @ v[b, hk].T
            dq[b, h] = scale * ((p * (dp - D[b, h, r][:, None])) @ k[b, hk])

            c = k_rows[b, hk]
            # scores of every query row against the selected keys: [N, R2]
            st = _scores_on(q[b, h], k[b, hk], scale, causal, all_rows, c, bmh, off)
            pt = probs(st, lse[b, h])
            dpt = do[b, h] @ v[b, hk, c].T
            dst = pt * (dpt - D[b, h][:, None])
            dk[b, hk] += scale * (dst.T @ q[b, h])
            dv[b, hk] += pt.T @ do[b, h]
    return dq, dk, dv


def backward_query_rows(q, k, v, do, causal, scale, b, h, rows):
    """Everything the given query rows of head (b, h) contribute, in double:
    their O, LSE, D and dQ rows, and their additive share of dK and dV of the
    KV head they read. Summing the shares over a partition of the rows gives
    `backward`'s dK and dV; each row is computed whole (same formulas as
    `backward`). Used to time the oracle on a bounded slice of a workload.
    Returns (o [R,d], lse [R], D [R], dq [R,d], dk_part [N,d], dv_part [N,d]).
    """
    B, Hq, Hkv, N, d, G = _check(q, k, v)
    hk = h // G
    rows = np.asarray(rows)
    s = _scores(q[b, h, rows], k[b, hk], scale, causal, rows)
    p, lse = _softmax_rows(s)
    o = p @ v[b, hk]
    D = (do[b, h, rows] * o).sum(axis=1)
    dp = do[b, h, rows] @ v[b, hk].T
    ds = p * (dp - D[:, None])
    dq = scale * (ds @ k[b, hk])
    dk_part = scale * (ds.T @ q[b, h, rows])
    dv_part = p.T @ do[b, h, rows]
    return o, lse, D, dq, dk_part, dv_part


def tiled_forward(q, k, v, causal, scale, block=64, deferred=True):
    """The pages' tiled algorithm with online softmax, in double.

    Follows "FlashAttention技术解析" sections 2.1-2.2: for each block of query
    rows, stream blocks of keys; per key block compute the block scores, the
    block max m_j, p = exp(S - m_j) and l_j = rowsum(p); merge with the
    running statistics as m_new = max(m, m_j) and
    l_new = e^(m - m_new) l + e^(m_j - m_new) l_j.
      deferred=False: the section 2.1 form, which renormalises the output
        every iteration: O <- (l/l_new) e^(m-m_new) O + (e^(m_j-m_new)/l_new) p V_j.
      deferred=True: the FlashAttention-2 form ("FlashAttention v2相比于v1有哪些
        更新", section 3, "Rescale操作"): keep O unnormalised,
        O <- e^(m-m_new) O + e^(m_j-m_new) p V_j, and divide by l once at the end.
    Causal blocks entirely above the diagonal are skipped ("Flash Attention V3
    技术解析" section 2.1); partially masked entries are -inf. The page's
    operators lost in extraction are read as in the formulas above.
    Returns (o, lse) like `forward`.
    """
    B, Hq, Hkv, N, d, G = _check(q, k, v)
    o = np.empty((B, Hq, N, d))
    lse = np.empty((B, Hq, N))
    for b in range(B):
        for h in range(Hq):
            hk = h // G
            for i0 in range(0, N, block):
                ri = np.arange(i0, min(i0 + block, N))
                qi = q[b, h, ri]
                acc = np.zeros((len(ri), d))
                m = np.full(len(ri), -np.inf)
                l = np.zeros(len(ri))
                for j0 in range(0, N, block):
                    if causal and j0 > ri[-1]:
                        break                      # block fully above the diagonal
                    rj = np.arange(j0, min(j0 + block, N))
                    s = scale * (qi @ k[b, hk, rj].T)
                    if causal:
                        s = np.where(rj[None, :] <= ri[:, None], s, -np.inf)
                    m_j = s.max(axis=1)
                    p = np.exp(s - m_j[:, None])
                    l_j = p.sum(axis=1)
                    m_new = np.maximum(m, m_j)
                    alpha = np.exp(m - m_new)      # exp(-inf) = 0 on the first block
                    beta = np.exp(m_j - m_new)
                    l_new = alpha * l + beta * l_j
                    pv = p @ v[b, hk, rj]
                    if deferred:
                        acc = alpha[:, None] * acc + beta[:, None] * pv
                    else:
                        acc = ((l / l_new) * alpha)[:, None] * acc + (beta / l_new)[:, None] * pv
                    m, l = m_new, l_new
                o[b, h, ri] = acc / l[:, None] if deferred else acc
                lse[b, h, ri] = m + np.log(l)
    return o, lse


__all__ = [
    "forward", "backward", "forward_rows", "row_statistics", "backward_rows",
    "backward_query_rows", "tiled_forward",
]
