"""Tiled online-softmax forward in fp64: the pages' algorithm, step by step.

TEST INFRASTRUCTURE ONLY (same rules as ``oracle.attn_ref``).

This restates the tiled forward of "FlashAttention-2实现与优化：高效注意力机制详解"
§3.1 (PyTorch基础实现) in plain numpy, in the page's order and notation:
Q is cut into tiles of Bq rows and K, V into tiles of Bk rows (the page leaves
Bq, Bk free); for each query tile the running statistics (m, l, o_acc) start
at (-inf, 0, 0) and, for each key tile j,

    S      = q_i k_j^T * scale            (masked to -inf where k > q if causal)
    m_new  = max(m, rowmax S)
    P      = exp(S - m_new)
    l_new  = exp(m - m_new) * l + rowsum P
    o_acc  = exp(m - m_new) * o_acc + P v_j

and the epilogue writes O = o_acc / l and L = m + log l.

Readings (the page is silent or garbled here):
  * mask fill -inf instead of the page's -1e6 (exact zero weight);
  * keys beyond Nk in a ragged last tile do not exist here (numpy slicing), so
    the page's zero-padded-key issue does not arise;
  * a key tile that a causal row cannot see at all leaves m = -inf; the
    subtrahend is then taken as 0 so exp(-inf - 0) = 0 (no NaN).

It exists to pin the algebra of the online update against the plain
definition in ``oracle.attn_ref`` (they agree to ~1e-12 for any Bq, Bk).
"""
from __future__ import annotations

import numpy as np


def tiled_forward_head(q, k, v, scale, causal, Bq, Bk):
    nq, d = q.shape
    nk = k.shape[0]
    o = np.empty((nq, v.shape[1]), np.float64)
    L = np.empty(nq, np.float64)
    for i in range(0, nq, Bq):
        q_i = q[i:i + Bq]
        rows = q_i.shape[0]
        m = np.full(rows, -np.inf)
        l = np.zeros(rows)
        o_acc = np.zeros((rows, v.shape[1]))
        for j in range(0, nk, Bk):
            k_j = k[j:j + Bk]
            v_j = v[j:j + Bk]
            S = (q_i @ k_j.T) * scale
            if causal:
                qi = np.arange(i, i + rows)[:, None]
                kj = np.arange(j, j + k_j.shape[0])[None, :]
                S = np.where(qi >= kj, S, -np.inf)
            m_new = np.maximum(m, S.max(axis=1))
            sub = np.where(np.isneginf(m_new), 0.0, m_new)
            P = np.exp(S - sub[:, None])
            alpha = np.exp(m - sub)
            l = alpha * l + P.sum(axis=1)
            o_acc = alpha[:, None] * o_acc + P @ v_j
            m = m_new
        o[i:i + rows] = o_acc / l[:, None]
        L[i:i + rows] = m + np.log(l)
    return o, L
