"""Plain fp64 CPU oracle for attention under a local-window + global-token mask.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports or calls this
module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / reference arm may.  It shares no code with the CUDA path.

The pages name this variant without defining it: "sparse attention combining
local windows and global tokens" ("FlashAttention-2实现与优化：高效注意力机制详解"
§7 扩展与进阶方向) and "sparse attention (local blocks + global key points)" for
100K-long sequences ("解释FlashAttention的显存优化原理", case 2).  The reading
taken here, an exact mask on absolute indices (top-left, as the causal mask of
§4.3 of the first page), is: query i may attend key j iff

    j < Nk
    and (not causal or j <= i)
    and (  (window_left  < 0 or j >= i - window_left)
           and (window_right < 0 or j <= i + window_right)
        or j < n_global          # global keys are seen by every query
        or i < n_global )        # global queries see every key

A negative window bound is unbounded.  Everything else is the plain definition
of ``attn_ref``: ``S = scale Q K^T``, masked entries get zero weight, row
softmax, ``O = P V``, ``L = m + log sum exp(S - m)``, and the softmax Jacobian
for the backward.  A query row with no allowed key has ``O = 0``, ``L = -inf``
and zero gradient (the same convention as a sequence with no keys).

Rows are processed in chunks of ``row_chunk`` queries; each chunk materialises
its full score rows over all keys (no key skipping), so the mask is applied by
its definition alone.  Pins: ``tests/test_oracle_masked_pins.py``.
"""
from __future__ import annotations

import numpy as np


def allowed(qi, kj, nk, causal, window_left, window_right, n_global):
    """Boolean mask for query indices ``qi`` (column vector) and key indices ``kj``
    (row vector), by the definition in the module docstring."""
    qi = np.asarray(qi)[:, None] if np.ndim(qi) == 1 else np.asarray(qi)
    kj = np.asarray(kj)[None, :] if np.ndim(kj) == 1 else np.asarray(kj)
    ok = kj < nk
    if causal:
        ok = ok & (kj <= qi)
    local = np.ones(np.broadcast(qi, kj).shape, bool)
    if window_left >= 0:
        local &= kj >= qi - window_left
    if window_right >= 0:
        local &= kj <= qi + window_right
    return ok & (local | (kj < n_global) | (qi < n_global))


def _softmax_masked(s, ok):
    """Row softmax over the allowed entries; empty rows give P = 0 and L = -inf."""
    empty = ~ok.any(axis=1)
    s = np.where(ok, s, -np.inf)
    m = np.where(empty, 0.0, s.max(axis=1, initial=-np.inf))
    e = np.where(ok, np.exp(s - m[:, None]), 0.0)
    l = e.sum(axis=1)
    p = e / np.where(empty, 1.0, l)[:, None]
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m + np.log(np.where(empty, 1.0, l)))
    return p, lse


def forward_head(q, k, v, scale, causal, window_left, window_right, n_global, rows=None, row_chunk=1024):
    """O and L for one head (q [Nq,D], k, v [Nk,D] float64); ``rows`` selects query rows."""
    nq, nk = q.shape[0], k.shape[0]
    idx = np.arange(nq) if rows is None else np.asarray(rows)
    o = np.empty((idx.size, v.shape[1]))
    lse = np.empty(idx.size)
    keys = np.arange(nk)
    for c0 in range(0, idx.size, row_chunk):
        ci = idx[c0:c0 + row_chunk]
        ok = allowed(ci, keys, nk, causal, window_left, window_right, n_global)
        p, l = _softmax_masked(scale * (q[ci] @ k.T), ok)
        o[c0:c0 + ci.size] = p @ v
        lse[c0:c0 + ci.size] = l
    return o, lse


def backward_head(q, k, v, do, scale, causal, window_left, window_right, n_global,
                  q_rows=None, k_range=None, row_chunk=1024):
    """dQ, dK, dV for one head via the softmax Jacobian.  Full outputs by default;
    ``q_rows`` computes only those dQ rows, ``k_range=(k0, k1)`` only dK/dV rows
    k0..k1-1 (from every query row that may attend one of them)."""
    nq, nk = q.shape[0], k.shape[0]
    keys = np.arange(nk)
    mask = (window_left, window_right, n_global)

    def grads(ci):
        ok = allowed(ci, keys, nk, causal, *mask)
        p, _ = _softmax_masked(scale * (q[ci] @ k.T), ok)
        dp = do[ci] @ v.T
        delta = (p * dp).sum(axis=1)
        return p, p * (dp - delta[:, None])

    if q_rows is None and k_range is None:
        dq, dk, dv = np.empty_like(q), np.zeros_like(k), np.zeros_like(v)
        for r0 in range(0, nq, row_chunk):
            ci = np.arange(r0, min(nq, r0 + row_chunk))
            p, ds = grads(ci)
            dq[ci] = scale * (ds @ k)
            dv += p.T @ do[ci]
            dk += scale * (ds.T @ q[ci])
        return dq, dk, dv

    dq = dk = dv = None
    if q_rows is not None:
        idx = np.asarray(q_rows)
        dq = np.empty((idx.size, q.shape[1]))
        for c0 in range(0, idx.size, row_chunk):
            ci = idx[c0:c0 + row_chunk]
            _, ds = grads(ci)
            dq[c0:c0 + ci.size] = scale * (ds @ k)
    if k_range is not None:
        k0, k1 = k_range
        dk = np.zeros((k1 - k0, k.shape[1]))
        dv = np.zeros((k1 - k0, v.shape[1]))
        # the query rows that may attend at least one key of the range, by the definition
        sees = np.zeros(nq, bool)
        for r0 in range(0, nq, 4 * row_chunk):
            r = np.arange(r0, min(nq, r0 + 4 * row_chunk))
            sees[r] = allowed(r, np.arange(k0, k1), nk, causal, *mask).any(axis=1)
        idx = np.nonzero(sees)[0]
        for c0 in range(0, idx.size, row_chunk):
            ci = idx[c0:c0 + row_chunk]
            p, ds = grads(ci)
            dv += p[:, k0:k1].T @ do[ci]
            dk += scale * (ds[:, k0:k1].T @ q[ci])
    return dq, dk, dv


def attention_forward(q, k, v, scale, causal, window_left, window_right, n_global, row_chunk=1024):
    """O [B,H,Nq,D] and L [B,H,Nq] for contiguous [B,H,N,D] float64 inputs."""
    B, H, Nq, _ = q.shape
    o = np.empty((B, H, Nq, v.shape[3]))
    lse = np.empty((B, H, Nq))
    for b in range(B):
        for h in range(H):
            o[b, h], lse[b, h] = forward_head(q[b, h], k[b, h], v[b, h], scale, causal, window_left,
                                              window_right, n_global, row_chunk=row_chunk)
    return o, lse


def attention_backward(q, k, v, do, scale, causal, window_left, window_right, n_global, row_chunk=1024):
    """dQ, dK, dV [B,H,N,D] for contiguous float64 inputs."""
    B, H = q.shape[:2]
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    for b in range(B):
        for h in range(H):
            dq[b, h], dk[b, h], dv[b, h] = backward_head(q[b, h], k[b, h], v[b, h], do[b, h], scale, causal,
                                                         window_left, window_right, n_global, row_chunk=row_chunk)
    return dq, dk, dv
