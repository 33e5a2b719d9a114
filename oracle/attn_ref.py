"""Plain fp64 CPU oracle for exact scaled-dot-product attention, forward and backward.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports or calls this
module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / reference arm may.  It shares no code with the CUDA path.

What it computes, per (batch b, head h), on inputs already rounded to bf16 and
upcast exactly to float64:

  1. ``S = scale * Q K^T``  (Nq x Nk).  Scale applied after the dot product, as in
     "FlashAttention-2实现与优化：高效注意力机制详解" §3.1/§3.2
     (``S = q k^T * scale``).
  2. Causal: ``S[i, j] = -inf`` for ``j > i`` on absolute indices (top-left
     alignment; the pages' mask keeps ``q_idx >= k_idx``, §4.3 因果掩码实现).
     The pages fill with -1e6; -inf is the exact zero-weight reading.
  3. Row-wise stable softmax ``P = exp(S - m) / sum exp(S - m)`` with
     ``m = rowmax S`` ("FlashAttention技术演进全景图" §2.3 stable_softmax),
     ``O = P V`` and the row logsumexp ``L = m + log(sum exp(S - m))``
     (natural log, same page as 1., §3.1: ``L = m + log(l)``).
  4. Backward for an upstream gradient dO, the softmax Jacobian written out
     (the pages name the backward only as "recompute instead of store",
     "解释FlashAttention的显存优化原理" §2(2) 重计算, and list it as future work in
     §7 of the FlashAttention-2 page):
        dV = P^T dO;  dP = dO V^T;  delta_i = sum_j P_ij dP_ij;
        dS = P o (dP - delta);  dQ = scale dS K;  dK = scale dS^T Q.
     ``delta`` is taken from P and dP (not from O and dO) so the oracle does
     not share the GPU path's route.

Queries are processed in chunks of at most ``row_chunk`` rows to bound memory;
each chunk still materialises its full score rows.  In causal mode a chunk
skips the key columns that no row of the chunk can see: their weight is
exactly zero, so the result is unchanged.

Parity pins for every function here live in ``tests/test_oracle_pins.py``.
"""
from __future__ import annotations

import numpy as np

NEG_INF = -np.inf


def _check(q, k, v):
    assert q.dtype == np.float64 and k.dtype == np.float64 and v.dtype == np.float64
    assert q.ndim == 4 and k.shape == v.shape and q.shape[:2] == k.shape[:2]
    assert q.shape[3] == k.shape[3]


def _scores(qc, k, scale, causal, row0):
    """Scaled, masked score rows for the query chunk starting at absolute row row0."""
    s = scale * (qc @ k.T)
    if causal:
        rows = np.arange(row0, row0 + qc.shape[0])[:, None]
        cols = np.arange(k.shape[0])[None, :]
        s = np.where(cols > rows, NEG_INF, s)
    return s


def _softmax_rows(s):
    """Stable softmax of each row plus the row logsumexp (natural log)."""
    m = s.max(axis=1)
    e = np.exp(s - m[:, None])
    l = e.sum(axis=1)
    return e / l[:, None], m + np.log(l)


def _visible_keys(row_end, nk, causal):
    # keys j <= row_end-1 are the only ones a causal chunk ending at row_end-1 sees
    return min(nk, row_end) if causal else nk


def forward_head(q, k, v, scale, causal, rows=None, row_chunk=1024):
    """O and L for one head.  q:[Nq,D], k,v:[Nk,D] float64.

    ``rows``: optional sorted array of query indices; only those rows are
    computed (used for sampled checks at large N).  Returns (o, lse) with
    shapes [len(rows) or Nq, D] and [len(rows) or Nq].
    """
    nq = q.shape[0]
    idx = np.arange(nq) if rows is None else np.asarray(rows)
    o = np.empty((idx.size, v.shape[1]), np.float64)
    lse = np.empty(idx.size, np.float64)
    for c0 in range(0, idx.size, row_chunk):
        ci = idx[c0:c0 + row_chunk]
        nkv = _visible_keys(int(ci.max()) + 1, k.shape[0], causal)
        s = scale * (q[ci] @ k[:nkv].T)
        if causal:
            s = np.where(np.arange(nkv)[None, :] > ci[:, None], NEG_INF, s)
        p, l = _softmax_rows(s)
        o[c0:c0 + ci.size] = p @ v[:nkv]
        lse[c0:c0 + ci.size] = l
    return o, lse


def attention_forward(q, k, v, scale, causal, row_chunk=1024):
    """O [B,H,Nq,D] and L [B,H,Nq] for contiguous [B,H,N,D] float64 inputs."""
    _check(q, k, v)
    B, H, Nq, D = q.shape
    o = np.empty((B, H, Nq, v.shape[3]), np.float64)
    lse = np.empty((B, H, Nq), np.float64)
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal,
                                              row_chunk=row_chunk)
    return o, lse


def backward_head(q, k, v, do, scale, causal, q_rows=None, k_range=None, row_chunk=1024):
    """dQ, dK, dV for one head via the explicit softmax Jacobian.

    Full outputs by default.  For sampled checks at large N:
      * ``q_rows``: only these dQ rows are computed (each needs only its own
        score row);
      * ``k_range=(k0, k1)``: only dK/dV rows k0..k1-1 are computed (they need
        every query row that can see them).
    With either given, the other outputs are returned as None unless also
    requested.
    """
    nq, nk = q.shape[0], k.shape[0]
    full = q_rows is None and k_range is None
    dq = dk = dv = None

    if full:
        # one pass over row chunks yields every output
        dq = np.empty_like(q)
        dk = np.zeros_like(k)
        dv = np.zeros_like(v)
        for r0 in range(0, nq, row_chunk):
            r1 = min(nq, r0 + row_chunk)
            nkv = _visible_keys(r1, nk, causal)
            s = _scores(q[r0:r1], k[:nkv], scale, causal, r0)
            p, _ = _softmax_rows(s)
            dp = do[r0:r1] @ v[:nkv].T
            delta = (p * dp).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dq[r0:r1] = scale * (ds @ k[:nkv])
            dv[:nkv] += p.T @ do[r0:r1]
            dk[:nkv] += scale * (ds.T @ q[r0:r1])
        return dq, dk, dv

    # dQ rows (sampled)
    if q_rows is not None:
        idx = np.asarray(q_rows)
        dq = np.empty((idx.size, q.shape[1]), np.float64)
        for c0 in range(0, idx.size, row_chunk):
            ci = idx[c0:c0 + row_chunk]
            nkv = _visible_keys(int(ci.max()) + 1, nk, causal)
            s = scale * (q[ci] @ k[:nkv].T)
            if causal:
                s = np.where(np.arange(nkv)[None, :] > ci[:, None], NEG_INF, s)
            p, _ = _softmax_rows(s)
            dp = do[ci] @ v[:nkv].T
            delta = (p * dp).sum(axis=1)
            ds = p * (dp - delta[:, None])
            dq[c0:c0 + ci.size] = scale * (ds @ k[:nkv])

    # dK / dV rows (a contiguous key range)
    if k_range is not None:
        k0, k1 = k_range
        dk = np.zeros((k1 - k0, k.shape[1]), np.float64)
        dv = np.zeros((k1 - k0, v.shape[1]), np.float64)
        first_q = k0 if causal else 0  # causal: rows i < k0 never see keys >= k0
        for r0 in range(first_q, nq, row_chunk):
            r1 = min(nq, r0 + row_chunk)
            nkv = _visible_keys(r1, nk, causal)
            s = _scores(q[r0:r1], k[:nkv], scale, causal, r0)
            p, _ = _softmax_rows(s)
            dp = do[r0:r1] @ v[:nkv].T
            delta = (p * dp).sum(axis=1)
            ds = p * (dp - delta[:, None])
            hi = min(k1, nkv)
            if hi <= k0:
                continue
            dv[:hi - k0] += p[:, k0:hi].T @ do[r0:r1]
            dk[:hi - k0] += scale * (ds[:, k0:hi].T @ q[r0:r1])
    return dq, dk, dv


def attention_backward(q, k, v, do, scale, causal, row_chunk=1024):
    """dQ, dK, dV [B,H,N,D] for contiguous float64 inputs."""
    _check(q, k, v)
    B, H = q.shape[:2]
    dq = np.empty_like(q)
    dk = np.empty_like(k)
    dv = np.empty_like(v)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(
                q[b, h], k[b, h], v[b, h], do[b, h], scale, causal, row_chunk=row_chunk)
    return dq, dk, dv


def attention_varlen(q, k, v, do, cu_q, cu_k, scale, causal, backward=True, row_chunk=1024):
    """Packed variable-length batch: sequence b is tokens cu_q[b]..cu_q[b+1]-1 of q/do
    ([total_q, H, D]) and cu_k[b]..cu_k[b+1]-1 of k/v ([total_k, H, D]); each (sequence,
    head) is attended independently (causal: top-left within the sequence).  A sequence
    with queries but no keys gets O = 0, L = -inf and zero gradients.
    Returns (o [total_q,H,D], lse [H,total_q], dq, dk, dv) (gradients None if not backward)."""
    total_q, H, D = q.shape
    o = np.zeros((total_q, H, v.shape[2]))
    lse = np.full((H, total_q), -np.inf)
    dq = np.zeros_like(q) if backward else None
    dk = np.zeros_like(k) if backward else None
    dv = np.zeros_like(v) if backward else None
    for b in range(len(cu_q) - 1):
        q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])
        if q1 <= q0 or k1 <= k0:
            continue
        for h in range(H):
            oo, ll = forward_head(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], scale, causal, row_chunk=row_chunk)
            o[q0:q1, h], lse[h, q0:q1] = oo, ll
            if backward:
                gq, gk, gv = backward_head(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], scale, causal,
                                           row_chunk=row_chunk)
                dq[q0:q1, h], dk[k0:k1, h], dv[k0:k1, h] = gq, gk, gv
    return o, lse, dq, dk, dv
