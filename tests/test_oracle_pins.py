"""Pins for the CPU oracle: it is checked against things other than itself.

* hand-derived closed-form cases (tests/golden/handworked.json);
* closed forms: Q=0 (uniform weights / causal prefix means), Nk=1, causal row 0;
* brute force with scalar Python loops on tiny inputs;
* PyTorch's float64 CPU scaled_dot_product_attention and autograd (a library
  routine for the same definition, top-left causal) and torch.logsumexp;
* central finite differences of sum(O * dO);
* invariants: key permutation, constant key shift, sum_j dK_j = 0,
  sum_j dV_j = sum_i dO_i;
* the tiled online-softmax restatement at several tile sizes.

``test_planted_mistakes_are_caught`` plants plausible mistakes in a copy of
the oracle (on the CPU) and checks that at least one pin fails for each.
"""
import json
import math
import os
import types

import numpy as np
import pytest
import torch

from oracle import attn_ref, tiled_ref

HERE = os.path.dirname(os.path.abspath(__file__))


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


# --------------------------------------------------------------------------------------
# pin functions: each takes an oracle module (the real one, or a planted-mistake copy)
# and returns True when the pin holds.
# --------------------------------------------------------------------------------------

def pin_handworked(ref):
    data = json.load(open(os.path.join(HERE, "golden", "handworked.json")))
    ok = True
    for c in data["cases"]:
        q, k, v = (np.array(c[x], np.float64) for x in ("q", "k", "v"))
        o, lse = ref.forward_head(q, k, v, c["scale"], c["causal"])
        ok &= np.allclose(o, c["o"], rtol=0, atol=1e-12) and np.allclose(lse, c["lse"], rtol=0, atol=1e-12)
        if "dq" in c:
            do = np.array(c["do"], np.float64)
            dq, dk, dv = ref.backward_head(q, k, v, do, c["scale"], c["causal"])
            ok &= np.allclose(dq, c["dq"], atol=1e-12) and np.allclose(dk, c["dk"], atol=1e-12)
            ok &= np.allclose(dv, c["dv"], atol=1e-12)
    return bool(ok)


def pin_closed_forms(ref):
    ok = True
    nk, d = 9, 4
    k, v = rnd((nk, d), 1), rnd((nk, d), 2)
    # Q = 0: uniform weights over the visible keys
    q0 = np.zeros((nk, d))
    o, lse = ref.forward_head(q0, k, v, 0.7, False)
    ok &= np.allclose(o, v.mean(0)[None, :].repeat(nk, 0), atol=1e-13)
    ok &= np.allclose(lse, math.log(nk), atol=1e-13)
    o, lse = ref.forward_head(q0, k, v, 0.7, True)
    prefix = np.cumsum(v, 0) / np.arange(1, nk + 1)[:, None]
    ok &= np.allclose(o, prefix, atol=1e-13)
    ok &= np.allclose(lse, np.log(np.arange(1, nk + 1)), atol=1e-13)
    # Nk = 1: O = v_0 and L = scale q.k_0, for every row, causal or not
    q = rnd((5, d), 3)
    for causal in (False, True):
        o, lse = ref.forward_head(q, k[:1], v[:1], 0.3, causal)
        ok &= np.allclose(o, v[:1].repeat(5, 0), atol=1e-13)
        ok &= np.allclose(lse, 0.3 * q @ k[0], atol=1e-13)
    # causal row 0 sees only key 0
    q = rnd((nk, d), 4)
    o, lse = ref.forward_head(q, k, v, 0.5, True)
    ok &= np.allclose(o[0], v[0], atol=1e-13) and abs(lse[0] - 0.5 * q[0] @ k[0]) < 1e-13
    return bool(ok)


def _brute_head(q, k, v, do, scale, causal):
    """Scalar-loop reference: O, L, dQ, dK, dV with math.exp only."""
    nq, nk, d = q.shape[0], k.shape[0], q.shape[1]
    O = np.zeros((nq, v.shape[1])); L = np.zeros(nq)
    dQ = np.zeros_like(q); dK = np.zeros_like(k); dV = np.zeros_like(v)
    for i in range(nq):
        vis = [j for j in range(nk) if (not causal) or j <= i]
        s = {j: scale * sum(q[i, t] * k[j, t] for t in range(d)) for j in vis}
        mx = max(s.values())
        den = sum(math.exp(s[j] - mx) for j in vis)
        p = {j: math.exp(s[j] - mx) / den for j in vis}
        L[i] = mx + math.log(den)
        for j in vis:
            O[i] += p[j] * v[j]
        dp = {j: sum(do[i, t] * v[j, t] for t in range(v.shape[1])) for j in vis}
        delta = sum(p[j] * dp[j] for j in vis)
        for j in vis:
            ds = p[j] * (dp[j] - delta)
            dQ[i] += scale * ds * k[j]
            dK[j] += scale * ds * q[i]
            dV[j] += p[j] * do[i]
    return O, L, dQ, dK, dV


def pin_brute_force(ref):
    ok = True
    for (nq, nk, d, causal, seed) in [(4, 6, 3, False, 10), (6, 6, 2, True, 11), (3, 7, 3, True, 12),
                                      (7, 3, 2, True, 13)]:
        q, k, v, do = rnd((nq, d), seed), rnd((nk, d), seed + 1), rnd((nk, d), seed + 2), rnd((nq, d), seed + 3)
        O, L, dQ, dK, dV = _brute_head(q, k, v, do, 0.6, causal)
        o, lse = ref.forward_head(q, k, v, 0.6, causal)
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.6, causal)
        for a, b in ((o, O), (lse, L), (dq, dQ), (dk, dK), (dv, dV)):
            ok &= np.allclose(a, b, rtol=1e-12, atol=1e-12)
    return bool(ok)


def pin_torch_library(ref):
    ok = True
    for (B, H, nq, nk, d, causal, seed) in [(2, 3, 17, 17, 8, False, 20), (2, 2, 33, 33, 16, True, 21),
                                            (1, 2, 9, 21, 4, True, 22), (1, 1, 21, 9, 4, True, 23),
                                            (1, 2, 13, 40, 8, False, 24)]:
        q, k, v, do = (rnd((B, H, n, d), seed + i) for i, n in enumerate((nq, nk, nk, nq)))
        sc = 1.0 / math.sqrt(d)
        tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
        to = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal, scale=sc)
        to.backward(torch.tensor(do))
        s = (torch.tensor(q) @ torch.tensor(k).transpose(-1, -2)) * sc
        if causal:
            s = s.masked_fill(torch.ones(nq, nk, dtype=torch.bool).tril().logical_not(), float("-inf"))
        tl = torch.logsumexp(s, dim=-1)
        o, lse = ref.attention_forward(q, k, v, sc, causal)
        dq, dk, dv = ref.attention_backward(q, k, v, do, sc, causal)
        ok &= np.allclose(o, to.detach().numpy(), rtol=1e-11, atol=1e-12)
        ok &= np.allclose(lse, tl.numpy(), rtol=1e-12, atol=1e-12)
        ok &= np.allclose(dq, tq.grad.numpy(), rtol=1e-10, atol=1e-11)
        ok &= np.allclose(dk, tk.grad.numpy(), rtol=1e-10, atol=1e-11)
        ok &= np.allclose(dv, tv.grad.numpy(), rtol=1e-10, atol=1e-11)
    return bool(ok)


def pin_finite_differences(ref):
    ok = True
    h = 1e-6
    for (nq, nk, d, causal, seed) in [(5, 7, 3, False, 30), (6, 6, 4, True, 31), (4, 7, 2, True, 32)]:
        q, k, v, do = rnd((nq, d), seed), rnd((nk, d), seed + 1), rnd((nk, d), seed + 2), rnd((nq, d), seed + 3)
        sc = 0.8

        def f(qq, kk, vv):
            return float((ref.forward_head(qq, kk, vv, sc, causal)[0] * do).sum())

        dq, dk, dv = ref.backward_head(q, k, v, do, sc, causal)
        for which, g in ((0, dq), (1, dk), (2, dv)):
            num = np.zeros_like(g)
            for idx in np.ndindex(*g.shape):
                args_p = [q.copy(), k.copy(), v.copy()]
                args_m = [q.copy(), k.copy(), v.copy()]
                args_p[which][idx] += h
                args_m[which][idx] -= h
                num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
            err = np.abs(num - g).max() / max(np.abs(g).max(), 1e-30)
            ok &= err <= 1e-7
    return bool(ok)


def pin_invariants(ref):
    ok = True
    nq = nk = 12
    d = 5
    q, k, v, do = rnd((nq, d), 40), rnd((nk, d), 41), rnd((nk, d), 42), rnd((nq, d), 43)
    # permuting keys and values together leaves a non-causal O unchanged
    perm = np.random.default_rng(44).permutation(nk)
    o1, l1 = ref.forward_head(q, k, v, 0.4, False)
    o2, l2 = ref.forward_head(q, k[perm], v[perm], 0.4, False)
    ok &= np.allclose(o1, o2, atol=1e-13) and np.allclose(l1, l2, atol=1e-13)
    # adding a constant vector c to every key: O unchanged, L_i shifts by scale q_i.c
    c = rnd((d,), 45)
    for causal in (False, True):
        o1, l1 = ref.forward_head(q, k, v, 0.4, causal)
        o2, l2 = ref.forward_head(q, k + c[None, :], v, 0.4, causal)
        ok &= np.allclose(o1, o2, atol=1e-12) and np.allclose(l2 - l1, 0.4 * q @ c, atol=1e-12)
        # gradient invariants
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.4, causal)
        ok &= np.allclose(dk.sum(0), 0.0, atol=1e-12)
        ok &= np.allclose(dv.sum(0), do.sum(0), atol=1e-12)
    # softmax rows sum to one: O of V = ones is ones
    o, _ = ref.forward_head(q, k, np.ones((nk, 3)), 0.4, True)
    ok &= np.allclose(o, 1.0, atol=1e-14)
    return bool(ok)


def pin_sampled_equals_full(ref):
    ok = True
    nq, nk, d = 50, 50, 4
    q, k, v, do = rnd((nq, d), 50), rnd((nk, d), 51), rnd((nk, d), 52), rnd((nq, d), 53)
    for causal in (False, True):
        o, lse = ref.forward_head(q, k, v, 0.5, causal, row_chunk=7)
        rows = np.array([0, 3, 17, 49])
        o2, l2 = ref.forward_head(q, k, v, 0.5, causal, rows=rows, row_chunk=3)
        ok &= np.allclose(o[rows], o2, atol=1e-13) and np.allclose(lse[rows], l2, atol=1e-13)
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.5, causal, row_chunk=11)
        dq2, _, _ = ref.backward_head(q, k, v, do, 0.5, causal, q_rows=rows, row_chunk=2)
        _, dk2, dv2 = ref.backward_head(q, k, v, do, 0.5, causal, k_range=(20, 37), row_chunk=6)
        ok &= np.allclose(dq[rows], dq2, atol=1e-12)
        ok &= np.allclose(dk[20:37], dk2, atol=1e-12) and np.allclose(dv[20:37], dv2, atol=1e-12)
    return bool(ok)


PINS = [pin_handworked, pin_closed_forms, pin_brute_force, pin_torch_library,
        pin_finite_differences, pin_invariants, pin_sampled_equals_full]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    assert pin(attn_ref)


# --------------------------------------------------------------------------------------
# tiled restatement of the online softmax vs the plain definition
# --------------------------------------------------------------------------------------

@pytest.mark.parametrize("Bq,Bk", [(1, 1), (3, 3), (16, 16), (5, 16), (16, 7), (128, 128)])
@pytest.mark.parametrize("causal", [False, True])
def test_tiled_online_softmax_matches_plain(Bq, Bk, causal):
    for (nq, nk) in [(37, 37), (37, 53), (53, 37), (1, 9)]:
        q, k, v = rnd((nq, 8), 60, 3.0), rnd((nk, 8), 61, 3.0), rnd((nk, 8), 62)
        o, lse = attn_ref.forward_head(q, k, v, 0.35, causal)
        o2, l2 = tiled_ref.tiled_forward_head(q, k, v, 0.35, causal, Bq, Bk)
        assert np.allclose(o, o2, rtol=0, atol=1e-12)
        assert np.allclose(lse, l2, rtol=0, atol=1e-12)


def pin_tiled(ref):
    # the tiled online update equals the plain definition for any tile sizes
    ok = True
    for Bq, Bk in [(1, 1), (3, 3), (5, 16), (16, 7), (128, 128)]:
        for causal in (False, True):
            for (nq, nk) in [(37, 37), (37, 53), (53, 37)]:
                q, k, v = rnd((nq, 8), 60, 3.0), rnd((nk, 8), 61, 3.0), rnd((nk, 8), 62)
                o, lse = attn_ref.forward_head(q, k, v, 0.35, causal)
                o2, l2 = ref.tiled_forward_head(q, k, v, 0.35, causal, Bq, Bk)
                ok &= bool(np.allclose(o, o2, rtol=0, atol=1e-12) and np.allclose(lse, l2, rtol=0, atol=1e-12))
    return ok


TILED_MUTATIONS = [
    ("alpha not applied to l", "l = alpha * l + P.sum(axis=1)", "l = l + P.sum(axis=1)"),
    ("o_acc not rescaled", "o_acc = alpha[:, None] * o_acc + P @ v_j", "o_acc = o_acc + P @ v_j"),
    ("running max not kept", "            m = m_new\n", "            m = S.max(axis=1)\n"),
    ("causal mask off by one", "S = np.where(qi >= kj, S, -np.inf)", "S = np.where(qi > kj, S, -np.inf)"),
    ("missing max term in L", "L[i:i + rows] = m + np.log(l)", "L[i:i + rows] = np.log(l)"),
]


@pytest.mark.parametrize("name,old,new", TILED_MUTATIONS, ids=[m[0] for m in TILED_MUTATIONS])
def test_tiled_planted_mistakes_are_caught(name, old, new):
    src = open(tiled_ref.__file__).read()
    assert old in src, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("tiled_ref_mutant")
    exec(compile(src.replace(old, new, 1), "tiled_ref_mutant", "exec"), mod.__dict__)
    try:
        with np.errstate(all="ignore"):  # a broken update may produce NaN: that is the point
            caught = not pin_tiled(mod)
    except Exception:  # a crash is also a caught mistake
        caught = True
    assert caught, f"planted mistake '{name}' passed the tiled pin"


def test_tiled_pin_holds():
    assert pin_tiled(tiled_ref)


def test_tiled_matches_torch_library():
    q, k, v = rnd((1, 1, 40, 8), 70), rnd((1, 1, 40, 8), 71), rnd((1, 1, 40, 8), 72)
    to = torch.nn.functional.scaled_dot_product_attention(
        torch.tensor(q), torch.tensor(k), torch.tensor(v), is_causal=True, scale=0.3)
    o, _ = tiled_ref.tiled_forward_head(q[0, 0], k[0, 0], v[0, 0], 0.3, True, 16, 16)
    assert np.allclose(o, to[0, 0].numpy(), atol=1e-12)


def test_large_logits_stable():
    # logits of several hundred (the x8 stability variant's range) stay finite
    q, k, v = rnd((64, 16), 80, 8.0), rnd((64, 16), 81, 8.0), rnd((64, 16), 82)
    o, lse = attn_ref.forward_head(q, k, v, 0.25, True)
    assert np.isfinite(o).all() and np.isfinite(lse).all() and np.abs(lse).max() > 100
    dq, dk, dv = attn_ref.backward_head(q, k, v, rnd((64, 16), 83), 0.25, True)
    assert np.isfinite(dq).all() and np.isfinite(dk).all()


# --------------------------------------------------------------------------------------
# planted mistakes: each must make at least one pin fail
# --------------------------------------------------------------------------------------

MUTATIONS = [
    ("sign of dS", "ds = p * (dp - delta[:, None])", "ds = p * (dp + delta[:, None])"),
    ("dropped scale in dQ", "dq[c0:c0 + ci.size] = scale * (ds @ k[:nkv])", "dq[c0:c0 + ci.size] = (ds @ k[:nkv])"),
    ("dropped scale in dK", "dk[:hi - k0] += scale * (ds[:, k0:hi].T @ q[r0:r1])", "dk[:hi - k0] += (ds[:, k0:hi].T @ q[r0:r1])"),
    ("causal mask off by one (fwd)", "s = np.where(np.arange(nkv)[None, :] > ci[:, None], NEG_INF, s)\n        p, l = _softmax_rows(s)",
     "s = np.where(np.arange(nkv)[None, :] > ci[:, None] + 1, NEG_INF, s)\n        p, l = _softmax_rows(s)"),
    ("causal mask off by one (bwd)", "s = np.where(cols > rows, NEG_INF, s)", "s = np.where(cols > rows + 1, NEG_INF, s)"),
    ("missing max term in L", "return e / l[:, None], m + np.log(l)", "return e / l[:, None], np.log(l)"),
    ("unnormalised P", "return e / l[:, None], m + np.log(l)", "return e, m + np.log(l)"),
    ("dQ multiplies V instead of K", "dq[c0:c0 + ci.size] = scale * (ds @ k[:nkv])", "dq[c0:c0 + ci.size] = scale * (ds @ v[:nkv])"),
    ("keys reversed in dP", "dp = do[r0:r1] @ v[:nkv].T", "dp = do[r0:r1] @ v[:nkv][::-1].T"),
    ("delta from wrong axis", "delta = (p * dp).sum(axis=1)\n            ds = p * (dp - delta[:, None])\n            hi",
     "delta = (p * dp).sum(axis=1) * 0\n            ds = p * (dp - delta[:, None])\n            hi"),
    ("dropped scale in full-pass dQ", "dq[r0:r1] = scale * (ds @ k[:nkv])", "dq[r0:r1] = (ds @ k[:nkv])"),
    ("full-pass dK without scale", "dk[:nkv] += scale * (ds.T @ q[r0:r1])", "dk[:nkv] += (ds.T @ q[r0:r1])"),
    ("full-pass dV scaled", "dv[:nkv] += p.T @ do[r0:r1]", "dv[:nkv] += 1.01 * (p.T @ do[r0:r1])"),
    ("dV uses dP instead of dO", "dv[:hi - k0] += p[:, k0:hi].T @ do[r0:r1]", "dv[:hi - k0] += p[:, k0:hi].T @ (do[r0:r1] * 1.5)"),
    ("no causal key skipping bound", "return min(nk, row_end) if causal else nk", "return min(nk, row_end - 1) if causal else nk"),
    ("scale applied twice", "s = scale * (q[ci] @ k[:nkv].T)\n        if causal:\n            s = np.where(np.arange(nkv)[None, :] > ci[:, None], NEG_INF, s)\n        p, l",
     "s = scale * scale * (q[ci] @ k[:nkv].T)\n        if causal:\n            s = np.where(np.arange(nkv)[None, :] > ci[:, None], NEG_INF, s)\n        p, l"),
]


def _mutant(src, old, new):
    assert old in src, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("attn_ref_mutant")
    exec(compile(src.replace(old, new, 1), "attn_ref_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(name, old, new):
    src = open(attn_ref.__file__).read()
    mut = _mutant(src, old, new)
    results = {}
    for pin in PINS:
        try:
            results[pin.__name__] = pin(mut)
        except Exception:  # a crash is also a caught mistake
            results[pin.__name__] = False
    assert not all(results.values()), f"planted mistake '{name}' passed every pin"


# --------------------------------------------------------------------------------------
# packed variable-length batches: each sequence attended on its own
# --------------------------------------------------------------------------------------

def pin_varlen_equal_lengths(ref):
    # equal lengths: the packed layout of the dense oracle's result
    B, H, N, D = 3, 2, 11, 4
    q, k, v, do = (rnd((B, H, N, D), 90 + i) for i in range(4))
    cu = np.arange(B + 1) * N
    pack = lambda x: x.transpose(0, 2, 1, 3).reshape(B * N, H, D)  # noqa: E731
    ok = True
    for causal in (False, True):
        o, lse, dq, dk, dv = ref.attention_varlen(pack(q), pack(k), pack(v), pack(do), cu, cu, 0.4, causal)
        ro, rl = attn_ref.attention_forward(q, k, v, 0.4, causal)
        rdq, rdk, rdv = attn_ref.attention_backward(q, k, v, do, 0.4, causal)
        ok &= bool(np.allclose(o, pack(ro), atol=1e-13))
        ok &= bool(np.allclose(lse, rl.transpose(1, 0, 2).reshape(H, B * N), atol=1e-13))
        for a_, r in ((dq, rdq), (dk, rdk), (dv, rdv)):
            ok &= bool(np.allclose(a_, pack(r), atol=1e-12))
    return ok


def pin_varlen_brute_force(ref):
    # ragged and cross lengths with empty sequences, each (sequence, head) by brute force
    lens_q, lens_k = [3, 0, 5, 1], [4, 2, 5, 0]
    cu_q, cu_k = np.concatenate([[0], np.cumsum(lens_q)]), np.concatenate([[0], np.cumsum(lens_k)])
    H, D = 2, 3
    q, do = rnd((cu_q[-1], H, D), 95), rnd((cu_q[-1], H, D), 96)
    k, v = rnd((cu_k[-1], H, D), 97), rnd((cu_k[-1], H, D), 98)
    ok = True
    for causal in (False, True):
        o, lse, dq, dk, dv = ref.attention_varlen(q, k, v, do, cu_q, cu_k, 0.6, causal)
        for b in range(4):
            q0, q1, k0, k1 = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
            for h in range(H):
                if q1 == q0:
                    continue
                if k1 == k0:
                    ok &= bool(np.all(o[q0:q1, h] == 0) and np.all(np.isneginf(lse[h, q0:q1])))
                    continue
                O, L, dQ, dK, dV = _brute_head(q[q0:q1, h], k[k0:k1, h], v[k0:k1, h], do[q0:q1, h], 0.6, causal)
                ok &= bool(np.allclose(o[q0:q1, h], O, atol=1e-12) and np.allclose(lse[h, q0:q1], L, atol=1e-12))
                ok &= bool(np.allclose(dq[q0:q1, h], dQ, atol=1e-12) and np.allclose(dk[k0:k1, h], dK, atol=1e-12))
                ok &= bool(np.allclose(dv[k0:k1, h], dV, atol=1e-12))
    return ok


VARLEN_PINS = [pin_varlen_equal_lengths, pin_varlen_brute_force]


@pytest.mark.parametrize("pin", VARLEN_PINS, ids=[p.__name__ for p in VARLEN_PINS])
def test_varlen_oracle_pin(pin):
    assert pin(attn_ref)


VARLEN_MUTATIONS = [
    ("keys of a sequence taken at the query offsets",
     "q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_k[b]), int(cu_k[b + 1])",
     "q0, q1, k0, k1 = int(cu_q[b]), int(cu_q[b + 1]), int(cu_q[b]), int(cu_q[b + 1])"),
    ("last sequence dropped", "for b in range(len(cu_q) - 1):", "for b in range(len(cu_q) - 2):"),
    ("L of every head written to head 0", "o[q0:q1, h], lse[h, q0:q1] = oo, ll", "o[q0:q1, h], lse[0, q0:q1] = oo, ll"),
    ("sequences without keys not skipped", "if q1 <= q0 or k1 <= k0:", "if q1 <= q0:"),
    ("dK written to the query rows", "dq[q0:q1, h], dk[k0:k1, h], dv[k0:k1, h] = gq, gk, gv",
     "dq[q0:q1, h], dk[q0:q0 + (k1 - k0), h], dv[k0:k1, h] = gq, gk, gv"),
]


@pytest.mark.parametrize("name,old,new", VARLEN_MUTATIONS, ids=[m[0] for m in VARLEN_MUTATIONS])
def test_varlen_planted_mistakes_are_caught(name, old, new):
    mut = _mutant(open(attn_ref.__file__).read(), old, new)
    results = {}
    for pin in VARLEN_PINS:
        try:
            results[pin.__name__] = pin(mut)
        except Exception:  # a crash is also a caught mistake
            results[pin.__name__] = False
    assert not all(results.values()), f"planted mistake '{name}' passed every varlen pin"
