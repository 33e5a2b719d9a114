"""Pins for the local-window + global-token oracle (``oracle.masked_ref``).

Checked against things other than itself:
* brute force with scalar Python loops and the mask written as its own predicate;
* reductions to the plain oracle (itself pinned): unbounded windows without global
  tokens, every token global, windows wider than the sequence;
* closed forms: a zero-width window (O = V, L = scale q.k, dV = dO, dQ = dK = 0) and
  Q = 0 (uniform weights over the allowed keys, whose count has a closed form);
* central finite differences of sum(O * dO);
* invariants: sum_j dK_j = 0 and sum_j dV_j = sum of dO over rows with a key;
* sampled rows / key ranges equal the full computation.
``test_planted_mistakes_are_caught`` plants plausible mistakes in a copy of the
oracle and checks that at least one pin fails for each.
"""
import math
import types

import numpy as np
import pytest

from oracle import attn_ref, masked_ref


def rnd(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _visible(i, j, nk, causal, wl, wr, g):
    if j >= nk or (causal and j > i):
        return False
    in_window = (wl < 0 or i - j <= wl) and (wr < 0 or j - i <= wr)
    return in_window or j < g or i < g


def _brute(q, k, v, do, scale, causal, wl, wr, g):
    nq, nk, d = q.shape[0], k.shape[0], q.shape[1]
    O = np.zeros((nq, v.shape[1])); L = np.full(nq, -math.inf)
    dQ = np.zeros_like(q); dK = np.zeros_like(k); dV = np.zeros_like(v)
    for i in range(nq):
        vis = [j for j in range(nk) if _visible(i, j, nk, causal, wl, wr, g)]
        if not vis:
            continue
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


def _same_lse(a, b, atol=1e-12):
    a, b = np.asarray(a), np.asarray(b)
    return bool(np.array_equal(np.isneginf(a), np.isneginf(b)) and
                np.allclose(a[np.isfinite(b)], b[np.isfinite(b)], atol=atol))


BRUTE_CASES = [
    # nq, nk, d, causal, wl, wr, g, seed
    (9, 9, 3, True, 2, -1, 0, 1),
    (9, 9, 3, False, 1, 2, 0, 2),
    (10, 10, 2, True, 1, -1, 2, 3),
    (10, 10, 2, False, 0, 0, 3, 4),
    (7, 11, 3, False, 2, 1, 1, 5),
    (11, 6, 2, True, 3, -1, 1, 6),
    (9, 4, 2, False, 1, 0, 0, 7),     # rows 6..8 have no key
    (6, 8, 2, True, -1, -1, 0, 8),
    (8, 8, 3, False, -1, 2, 2, 9),
]


def pin_brute_force(ref):
    ok = True
    for (nq, nk, d, causal, wl, wr, g, seed) in BRUTE_CASES:
        q, k, v, do = rnd((nq, d), seed), rnd((nk, d), seed + 10), rnd((nk, d), seed + 20), rnd((nq, d), seed + 30)
        O, L, dQ, dK, dV = _brute(q, k, v, do, 0.7, causal, wl, wr, g)
        o, lse = ref.forward_head(q, k, v, 0.7, causal, wl, wr, g, row_chunk=4)
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.7, causal, wl, wr, g, row_chunk=3)
        ok &= np.allclose(o, O, atol=1e-12) and _same_lse(lse, L)
        ok &= np.allclose(dq, dQ, atol=1e-12) and np.allclose(dk, dK, atol=1e-12) and np.allclose(dv, dV, atol=1e-12)
    return bool(ok)


def pin_reduces_to_plain(ref):
    ok = True
    for (nq, nk, causal) in [(13, 13, True), (13, 13, False), (9, 14, True), (14, 9, False)]:
        q, k, v, do = rnd((nq, 4), 40), rnd((nk, 4), 41), rnd((nk, 4), 42), rnd((nq, 4), 43)
        o0, l0 = attn_ref.forward_head(q, k, v, 0.5, causal)
        g0 = attn_ref.backward_head(q, k, v, do, 0.5, causal)
        for (wl, wr, g) in [(-1, -1, 0), (-1, -1, 5), (0, 0, max(nq, nk)), (nq + nk, nq + nk, 0), (nq + nk, -1, 2)]:
            o, lse = ref.forward_head(q, k, v, 0.5, causal, wl, wr, g)
            gr = ref.backward_head(q, k, v, do, 0.5, causal, wl, wr, g)
            ok &= np.allclose(o, o0, atol=1e-13) and np.allclose(lse, l0, atol=1e-13)
            ok &= all(np.allclose(a, b, atol=1e-12) for a, b in zip(gr, g0))
    return bool(ok)


def pin_closed_forms(ref):
    ok = True
    n, d = 12, 5
    q, k, v, do = rnd((n, d), 50), rnd((n, d), 51), rnd((n, d), 52), rnd((n, d), 53)
    # zero-width window: each query sees only its own key
    for causal, wr in ((False, 0), (True, -1)):
        o, lse = ref.forward_head(q, k, v, 0.4, causal, 0, wr, 0)
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.4, causal, 0, wr, 0)
        ok &= np.allclose(o, v, atol=1e-14) and np.allclose(lse, 0.4 * (q * k).sum(1), atol=1e-13)
        ok &= np.allclose(dv, do, atol=1e-14) and np.abs(dq).max() < 1e-14 and np.abs(dk).max() < 1e-14
    # Q = 0: uniform weights over the allowed keys.  Window [i-wl, i+wr] clipped to [0, nk):
    # count = min(nk-1, i+wr) - max(0, i-wl) + 1, O_i = mean of those V rows.
    q0 = np.zeros((n, d))
    for wl, wr in ((2, 1), (0, 3), (4, 0)):
        o, lse = ref.forward_head(q0, k, v, 0.9, False, wl, wr, 0)
        for i in range(n):
            a, b = max(0, i - wl), min(n - 1, i + wr)
            ok &= np.allclose(o[i], v[a:b + 1].mean(0), atol=1e-13) and abs(lse[i] - math.log(b - a + 1)) < 1e-13
    # Q = 0, causal, window 0, G global tokens: row i < G sees keys 0..i; row i >= G sees 0..G-1 and i
    g = 3
    o, lse = ref.forward_head(q0, k, v, 0.9, True, 0, -1, g)
    for i in range(n):
        cols = list(range(i + 1)) if i < g else list(range(g)) + [i]
        ok &= np.allclose(o[i], v[cols].mean(0), atol=1e-13) and abs(lse[i] - math.log(len(cols))) < 1e-13
    # rows with no allowed key: O = 0, L = -inf, dQ = 0
    o, lse = ref.forward_head(q[:, :], k[:4], v[:4], 0.5, False, 1, 0, 0)
    dq, _, _ = ref.backward_head(q, k[:4], v[:4], do, 0.5, False, 1, 0, 0)
    ok &= bool(np.all(o[6:] == 0) and np.all(np.isneginf(lse[6:])) and np.all(dq[6:] == 0))
    ok &= bool(np.isfinite(lse[:5]).all())
    return bool(ok)


def pin_finite_differences(ref):
    ok = True
    nq, nk, d = 8, 10, 3
    q, k, v, do = rnd((nq, d), 60), rnd((nk, d), 61), rnd((nk, d), 62), rnd((nq, d), 63)
    for causal, wl, wr, g in ((True, 2, -1, 1), (False, 1, 2, 2)):
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.6, causal, wl, wr, g)

        def f(q_, k_, v_):
            o, _ = ref.forward_head(q_, k_, v_, 0.6, causal, wl, wr, g)
            return float((o * do).sum())
        h = 1e-6
        for name, x, gx in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
            num = np.zeros_like(x)
            for idx in np.ndindex(*x.shape):
                xp, xm = x.copy(), x.copy()
                xp[idx] += h
                xm[idx] -= h
                args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
                args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
                num[idx] = (f(*args_p) - f(*args_m)) / (2 * h)
            ok &= np.allclose(num, gx, atol=1e-7)
    return bool(ok)


def pin_invariants(ref):
    ok = True
    nq, nk, d = 30, 24, 4
    q, k, v, do = rnd((nq, d), 70), rnd((nk, d), 71), rnd((nk, d), 72), rnd((nq, d), 73)
    for causal, wl, wr, g in ((True, 5, -1, 3), (False, 3, 2, 0), (False, 2, 1, 4)):
        _, lse = ref.forward_head(q, k, v, 0.5, causal, wl, wr, g)
        _, dk, dv = ref.backward_head(q, k, v, do, 0.5, causal, wl, wr, g)
        has_key = np.isfinite(lse)
        ok &= np.allclose(dk.sum(0), 0.0, atol=1e-12)
        ok &= np.allclose(dv.sum(0), do[has_key].sum(0), atol=1e-12)
    return bool(ok)


def pin_sampled_equals_full(ref):
    ok = True
    nq, nk, d = 50, 45, 3
    q, k, v, do = rnd((nq, d), 80), rnd((nk, d), 81), rnd((nk, d), 82), rnd((nq, d), 83)
    rows = np.array([0, 3, 17, 31, 49])
    for causal, wl, wr, g in ((True, 6, -1, 2), (False, 4, 3, 1)):
        o, lse = ref.forward_head(q, k, v, 0.5, causal, wl, wr, g, row_chunk=7)
        o2, l2 = ref.forward_head(q, k, v, 0.5, causal, wl, wr, g, rows=rows, row_chunk=2)
        ok &= np.allclose(o[rows], o2, atol=1e-13) and _same_lse(lse[rows], l2)
        dq, dk, dv = ref.backward_head(q, k, v, do, 0.5, causal, wl, wr, g, row_chunk=9)
        dq2, _, _ = ref.backward_head(q, k, v, do, 0.5, causal, wl, wr, g, q_rows=rows, row_chunk=2)
        _, dk2, dv2 = ref.backward_head(q, k, v, do, 0.5, causal, wl, wr, g, k_range=(20, 33), row_chunk=4)
        ok &= np.allclose(dq[rows], dq2, atol=1e-12)
        ok &= np.allclose(dk[20:33], dk2, atol=1e-12) and np.allclose(dv[20:33], dv2, atol=1e-12)
    return bool(ok)


PINS = [pin_brute_force, pin_reduces_to_plain, pin_closed_forms, pin_finite_differences, pin_invariants,
        pin_sampled_equals_full]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_masked_oracle_pin(pin):
    assert pin(masked_ref)


def test_batched_wrappers_match_heads():
    q, k, v, do = rnd((2, 3, 17, 4), 90), rnd((2, 3, 17, 4), 91), rnd((2, 3, 17, 4), 92), rnd((2, 3, 17, 4), 93)
    o, lse = masked_ref.attention_forward(q, k, v, 0.5, True, 3, -1, 2)
    dq, dk, dv = masked_ref.attention_backward(q, k, v, do, 0.5, True, 3, -1, 2)
    for b in range(2):
        for h in range(3):
            oh, lh = masked_ref.forward_head(q[b, h], k[b, h], v[b, h], 0.5, True, 3, -1, 2)
            gh = masked_ref.backward_head(q[b, h], k[b, h], v[b, h], do[b, h], 0.5, True, 3, -1, 2)
            assert np.array_equal(o[b, h], oh) and np.array_equal(lse[b, h], lh)
            assert all(np.array_equal(a, g) for a, g in zip((dq[b, h], dk[b, h], dv[b, h]), gh))


MUTATIONS = [
    ("window left off by one", "local &= kj >= qi - window_left", "local &= kj > qi - window_left"),
    ("window right sign", "local &= kj <= qi + window_right", "local &= kj <= qi - window_right"),
    ("global keys dropped", "return ok & (local | (kj < n_global) | (qi < n_global))",
     "return ok & (local | (qi < n_global))"),
    ("global queries dropped", "return ok & (local | (kj < n_global) | (qi < n_global))",
     "return ok & (local | (kj < n_global))"),
    ("global tokens override causality", "return ok & (local | (kj < n_global) | (qi < n_global))",
     "return (ok & local) | (kj < n_global) | (qi < n_global)"),
    ("empty rows get L = 0", "lse = np.where(empty, -np.inf, m + np.log(np.where(empty, 1.0, l)))",
     "lse = np.where(empty, 0.0, m + np.log(np.where(empty, 1.0, l)))"),
    ("sign of dS", "return p, p * (dp - delta[:, None])", "return p, p * (dp + delta[:, None])"),
    ("dK without scale", "dk += scale * (ds.T @ q[ci])", "dk += (ds.T @ q[ci])"),
    ("sampled dK misses global rows", "sees[r] = allowed(r, np.arange(k0, k1), nk, causal, *mask).any(axis=1)",
     "sees[r] = allowed(r, np.arange(k0, k1), nk, causal, mask[0], mask[1], 0).any(axis=1)"),
    ("masked entries keep weight", "e = np.where(ok, np.exp(s - m[:, None]), 0.0)",
     "e = np.exp(np.where(ok, s, m[:, None] - 3.0) - m[:, None])"),
]


def _mutant(src, old, new):
    assert old in src, f"mutation anchor not found: {old!r}"
    mod = types.ModuleType("masked_ref_mutant")
    exec(compile(src.replace(old, new, 1), "masked_ref_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(name, old, new):
    mut = _mutant(open(masked_ref.__file__).read(), old, new)
    results = {}
    for pin in PINS:
        try:
            results[pin.__name__] = pin(mut)
        except Exception:  # a crash is also a caught mistake
            results[pin.__name__] = False
    assert not all(results.values()), f"planted mistake '{name}' passed every pin"


@pytest.mark.parametrize("nq,nk,causal,wl,wr,g", [(40, 40, True, 5, -1, 0), (40, 40, True, 7, -1, 3),
                                                  (33, 50, False, 4, 9, 6), (50, 33, False, 0, 0, 0),
                                                  (30, 30, False, -1, 2, 40), (45, 20, True, 3, -1, 25)])
def test_bench_pair_count_matches_the_mask(nq, nk, causal, wl, wr, g):
    # the FLOP count bench.py reports for local-window rows counts exactly the allowed pairs
    import bench
    want = int(masked_ref.allowed(np.arange(nq), np.arange(nk), nk, causal, wl, wr, g).sum())
    assert bench.window_pairs(nq, nk, causal, wl, wr, g) == want
