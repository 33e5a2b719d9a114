"""GPU parity for the local-window + global-token mask (fa_fwd_window / fa_bwd_window).

Same acceptance as the dense parity tests (O, dQ, dK, dV relative-L2 <= 1e-2 and
max-abs <= 2e-2 * max|ref|; L within 1e-3; rows without a visible key exactly O = 0,
L = -inf).  The oracle is ``oracle.masked_ref``, the mask written out by definition.
Cases cover windows narrower and wider than a tile, tile-aligned and ragged edges,
global tokens inside one tile and across several, non-causal windows with a right
extent, Nq != Nk, rows with no visible key, degenerate masks that reduce to the
plain ones (compared bitwise with fa_fwd/fa_bwd), exact zero weight outside the
mask, and a long sequence where the oracle checks sampled rows and key ranges.
"""
import numpy as np
import pytest
import torch

import oracle
from oracle import masked_ref
from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300 import inputs as I
from tiled_attention_11_gb300.build import build

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_FRAC = 2e-2
LSE_ABS = 1e-3
ZERO_REF_ABS = 1e-4


@pytest.fixture(scope="module", autouse=True)
def _lib_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    _lib.lib()
    _lib.fa_device_status(reset=True)
    yield
    rc, site = _lib.fa_device_status()
    assert rc == _lib.FA_OK, f"device status word set: {rc} at wait site {site}"


def f64(t):
    return t.detach().to("cpu", torch.float64).numpy()


def assert_close(name, got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert got.shape == ref.shape and np.isfinite(got).all(), name
    err = got - ref
    nref = np.linalg.norm(ref)
    rl2 = np.linalg.norm(err) / nref if nref > 0 else np.linalg.norm(err)
    ma = np.abs(err).max() if err.size else 0.0
    rmax = np.abs(ref).max() if ref.size else 0.0
    lim = MAX_FRAC * rmax if rmax > 0 else ZERO_REF_ABS
    assert rl2 <= REL_L2 and ma <= lim, f"{name}: rel_l2={rl2:.3e} max_abs={ma:.3e} limit={lim:.3e}"


def assert_lse(name, got, ref):
    got, ref = np.asarray(got, np.float64), np.asarray(ref, np.float64)
    assert np.array_equal(np.isneginf(got), np.isneginf(ref)), f"{name}: -inf pattern"
    fin = np.isfinite(ref)
    assert np.isfinite(got[fin]).all()
    if fin.any():
        e = np.abs(got[fin] - ref[fin]).max()
        assert e <= LSE_ABS, f"{name}: max_abs={e:.3e}"


def run_window(p, q, k, v, do, wl, wr, g, sentinel=float("nan")):
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o = torch.full_like(qg, sentinel)
    lse = torch.full((p.B, p.H, p.Nq), sentinel, dtype=torch.float32, device=dev)
    _lib.fa_fwd_window(qg, kg, vg, o, lse, p.causal, wl, wr, g, p.scale)
    dq, dk, dv = (torch.full_like(t, sentinel) for t in (qg, kg, vg))
    _lib.fa_bwd_window(qg, kg, vg, o, lse, dog, dq, dk, dv, p.causal, wl, wr, g, p.scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def check_window(p, wl, wr, g, seed=0):
    q, k, v, do = I.draw(p, seed)
    o, lse, dq, dk, dv = run_window(p, q, k, v, do, wl, wr, g)
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    ro, rl = masked_ref.attention_forward(qd, kd, vd, p.scale, p.causal, wl, wr, g)
    rdq, rdk, rdv = masked_ref.attention_backward(qd, kd, vd, dod, p.scale, p.causal, wl, wr, g)
    tag = f"{p.name()} wl{wl} wr{wr} g{g} s{seed}"
    assert_close(tag + " O", f64(o), ro)
    assert_lse(tag + " L", f64(lse), rl)
    assert_close(tag + " dQ", f64(dq), rdq)
    assert_close(tag + " dK", f64(dk), rdk)
    assert_close(tag + " dV", f64(dv), rdv)


CASES = [
    # (problem, window_left, window_right, n_global)
    (I.Problem(2, 2, 700, 700, 128, True), 100, -1, 0),      # window narrower than a tile
    (I.Problem(2, 2, 700, 700, 128, True), 256, -1, 0),      # tile-aligned window
    (I.Problem(1, 2, 1000, 1000, 64, True), 300, -1, 5),     # global tokens inside one tile
    (I.Problem(1, 2, 1000, 1000, 64, True), 130, -1, 200),   # global tokens across two tiles
    (I.Problem(1, 2, 900, 900, 128, False), 150, 70, 0),     # non-causal, both extents
    (I.Problem(1, 2, 900, 900, 32, False), 64, 200, 129),    # non-causal with global
    (I.Problem(1, 1, 513, 513, 16, True), 0, -1, 0),         # each query sees itself only
    (I.Problem(1, 2, 600, 333, 64, False), 50, 40, 0),       # Nq > Nk: rows past the keys see none
    (I.Problem(1, 2, 333, 600, 128, True), 90, -1, 3),       # Nq < Nk
    (I.Problem(2, 1, 1025, 1025, 128, True), 511, -1, 64),   # ragged tail, several tiles
    (I.Problem(1, 2, 800, 800, 64, False), -1, 0, 0),        # window_right only (= causal)
    (I.Problem(1, 2, 800, 800, 128, False), 0, -1, 17),      # look-ahead only plus global
]


@pytest.mark.parametrize("p,wl,wr,g", CASES, ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in CASES])
def test_window_parity(p, wl, wr, g):
    check_window(p, wl, wr, g)


def test_window_large_logits():
    p = I.Problem(1, 2, 640, 640, 128, True, qk_factor=8.0)
    check_window(p, 200, -1, 32, seed=3)


BITWISE_CASES = [
    # (B, H, Nq, Nk, D, causal).  Causal grids of at most one wave fold their query-tile
    # pairs in fa_fwd (tile t with tile n-1-t); the local-mask kernel never does, so these
    # also check the fold bit for bit: odd tile counts (the middle tile alone), even ones,
    # and Nq != Nk both ways.
    (2, 2, 333, 333, 64, False),
    (2, 2, 333, 333, 64, True),
    (1, 2, 1100, 1100, 128, True),
    (1, 2, 1536, 1536, 64, True),
    (1, 1, 700, 1500, 128, True),
    (1, 1, 1500, 700, 32, True),
]


@pytest.mark.parametrize("B,H,Nq,Nk,D,causal", BITWISE_CASES,
                         ids=[f"B{c[0]}H{c[1]}q{c[2]}k{c[3]}D{c[4]}{'c' if c[5] else 'n'}" for c in BITWISE_CASES])
def test_unbounded_mask_matches_plain_path_bitwise(B, H, Nq, Nk, D, causal):
    # window_left = window_right = -1 and no global tokens is the plain mask: the same
    # tiles in the same order, so the outputs agree bit for bit with fa_fwd / fa_bwd
    p = I.Problem(B, H, Nq, Nk, D, causal)
    q, k, v, do = I.draw(p, 5)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = _lib.forward(qg, kg, vg, causal, p.scale)
    dq, dk, dv = _lib.backward(qg, kg, vg, o, lse, dog, causal, p.scale)
    wo, wl_, wdq, wdk, wdv = run_window(p, q, k, v, do, -1, -1, 0)
    assert torch.equal(wo, o) and torch.equal(wl_, lse)
    assert torch.equal(wdk, dk) and torch.equal(wdv, dv)
    assert_close("dQ", f64(wdq), f64(dq))  # dQ adds across CTAs in any order


def test_all_global_equals_plain():
    p = I.Problem(1, 2, 300, 300, 128, True)
    q, k, v, do = I.draw(p, 6)
    o, lse, dq, dk, dv = run_window(p, q, k, v, do, 3, -1, 300)
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    ro, rl = oracle.attention_forward(qd, kd, vd, p.scale, True)
    assert_close("O", f64(o), ro)
    assert_lse("L", f64(lse), rl)


def test_masked_keys_have_zero_weight():
    # changing K and V outside every query's window (and not global) leaves O and L bitwise unchanged
    p = I.Problem(1, 1, 512, 512, 64, True)
    q, k, v, _ = I.draw(p, 7)
    wl, g = 64, 16
    dev = torch.device("cuda")
    qg, kg, vg = (t.to(dev) for t in (q, k, v))
    o1 = torch.empty_like(qg)
    l1 = torch.empty((1, 1, 512), device=dev)
    _lib.fa_fwd_window(qg, kg, vg, o1, l1, True, wl, -1, g, p.scale)
    # rows 400..511 see keys [i-64, i] and 0..15: keys 16..335 are invisible to them
    k2, v2 = kg.clone(), vg.clone()
    k2[0, 0, 16:336] = 30.0
    v2[0, 0, 16:336] = -7.0
    o2 = torch.empty_like(qg)
    l2 = torch.empty_like(l1)
    _lib.fa_fwd_window(qg, k2, v2, o2, l2, True, wl, -1, g, p.scale)
    torch.cuda.synchronize()
    assert torch.equal(o1[0, 0, 400:], o2[0, 0, 400:]) and torch.equal(l1[0, 0, 400:], l2[0, 0, 400:])


def test_long_window_sampled():
    # 16384 tokens, window 1024, 64 global tokens: sampled query rows and key ranges
    p = I.Problem(1, 2, 16384, 16384, 128, True)
    wl, g = 1024, 64
    q, k, v, do = I.draw(p, 8)
    o, lse, dq, dk, dv = run_window(p, q, k, v, do, wl, -1, g)
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    rows = np.array([0, 63, 64, 1087, 1088, 8191, 16383])
    for h in range(p.H):
        ro, rl = masked_ref.forward_head(qd[0, h], kd[0, h], vd[0, h], p.scale, True, wl, -1, g, rows=rows)
        assert_close(f"h{h} O", f64(o)[0, h][rows], ro)
        assert_lse(f"h{h} L", f64(lse)[0, h][rows], rl)
        rdq, _, _ = masked_ref.backward_head(qd[0, h], kd[0, h], vd[0, h], dod[0, h], p.scale, True, wl, -1, g,
                                             q_rows=rows)
        assert_close(f"h{h} dQ", f64(dq)[0, h][rows], rdq)
        for k0, k1 in ((0, 128), (8000, 8128), (16256, 16384)):
            _, rdk, rdv = masked_ref.backward_head(qd[0, h], kd[0, h], vd[0, h], dod[0, h], p.scale, True, wl, -1,
                                                   g, k_range=(k0, k1))
            assert_close(f"h{h} dK[{k0}:{k1}]", f64(dk)[0, h, k0:k1], rdk)
            assert_close(f"h{h} dV[{k0}:{k1}]", f64(dv)[0, h, k0:k1], rdv)
    # invariants over every key: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i (every row sees a key)
    dkl, dvl, dol = dk.double().cpu(), dv.double().cpu(), do.double()
    assert ((dkl.sum(2).abs() / dkl.abs().sum(2).clamp_min(1e-30)).max() < 5e-3)
    assert (((dvl.sum(2) - dol.sum(2)).abs() / dol.abs().sum(2).clamp_min(1e-30)).max() < 5e-3)


SPLIT_CASES = [
    # non-causal, global tokens, key range > 32 tiles: the global query tiles split into
    # chunks of 16 key tiles and merged (rows of the same tiles that are not global see
    # nothing in far chunks)
    (I.Problem(1, 2, 5000, 5000, 64, False), 100, 100, 40),
    (I.Problem(1, 1, 4500, 4500, 128, False), 64, 0, 300),     # two global pairs
    (I.Problem(2, 1, 600, 5000, 128, False), 50, 50, 17),      # Nq != Nk
    (I.Problem(1, 1, 4300, 4300, 32, False), -1, 30, 129),     # look-back unbounded
]


@pytest.mark.parametrize("p,wl,wr,g", SPLIT_CASES, ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in SPLIT_CASES])
def test_window_split_global_rows(p, wl, wr, g):
    assert _lib.fa_fwd_window_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D, p.causal, wl, wr, g) > 0
    check_window(p, wl, wr, g)


def test_window_split_large_logits():
    p = I.Problem(1, 1, 4400, 4400, 128, False, qk_factor=8.0)
    assert _lib.fa_fwd_window_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D, p.causal, 200, 200, 64) > 0
    check_window(p, 200, 200, 64, seed=4)


BWD_SPLIT_CASES = [
    # more than 64 query steps with global keys: the global key tiles split into chunks
    # of 32 query steps whose partial dK, dV add up in an fp32 workspace
    (I.Problem(1, 2, 4500, 4500, 64, True), 200, -1, 40),      # causal, one global key tile
    (I.Problem(1, 1, 4200, 4200, 128, True), 128, -1, 300),    # three global key tiles, ragged
    (I.Problem(1, 1, 4200, 4500, 128, True), 300, -1, 130),    # causal, Nq < Nk
    (I.Problem(1, 1, 5000, 2000, 64, False), 100, 100, 17),    # Nq > Nk
    (I.Problem(1, 2, 4200, 200, 64, False), 10, 10, 500),      # every key global
]


@pytest.mark.parametrize("p,wl,wr,g", BWD_SPLIT_CASES,
                         ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in BWD_SPLIT_CASES])
def test_window_split_global_keys(p, wl, wr, g):
    assert (_lib.fa_bwd_window_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D, wl, wr, g) >
            _lib.fa_bwd_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D))
    check_window(p, wl, wr, g)


# Beyond one wave of query-tile pairs the forward of an unsplit mask (causal, or no global
# rows to split) runs persistent CTAs by default: same per-row arithmetic and key order as
# one CTA per pair, so O and L agree bit for bit.  Ragged tails (a pair whose second tile is
# past the rows), Nq > Nk (tiles whose rows see no key), globals across two tiles, D 16-128.
PERSIST_CASES = [
    (I.Problem(1, 32, 1100, 1100, 128, True), 300, -1, 64, True),
    (I.Problem(2, 40, 700, 700, 64, False), 100, 50, 0, False),
    (I.Problem(1, 64, 600, 333, 32, False), 50, 40, 0, True),
    (I.Problem(1, 48, 1000, 1000, 16, False), 64, 64, 100, False),
    (I.Problem(1, 32, 1300, 900, 128, True), 200, -1, 130, False),
]


@pytest.mark.parametrize("p,wl,wr,g,with_oracle", PERSIST_CASES,
                         ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in PERSIST_CASES])
def test_window_forward_persistent_equals_one_cta_per_pair(p, wl, wr, g, with_oracle):
    q, k, v, _ = I.draw(p, 4)
    dev = torch.device("cuda")
    qg, kg, vg = (t.to(dev) for t in (q, k, v))
    outs = {}
    prev = _lib.fa_set_fwd_persistent(True)
    try:
        for on in (True, False):
            _lib.fa_set_fwd_persistent(on)
            o = torch.full_like(qg, float("nan"))
            lse = torch.full((p.B, p.H, p.Nq), float("nan"), dtype=torch.float32, device=dev)
            _lib.fa_fwd_window(qg, kg, vg, o, lse, p.causal, wl, wr, g, p.scale)
            torch.cuda.synchronize()
            outs[on] = (o, lse)
    finally:
        _lib.fa_set_fwd_persistent(prev)
    assert torch.equal(outs[True][0], outs[False][0]), "O"
    assert torch.equal(outs[True][1], outs[False][1]), "L"
    if with_oracle:
        qd, kd, vd = (I.as_f64(t) for t in (q, k, v))
        ro, rl = masked_ref.attention_forward(qd, kd, vd, p.scale, p.causal, wl, wr, g)
        assert_close("persistent O", f64(outs[True][0]), ro)
        assert_lse("persistent L", f64(outs[True][1]), rl)


# The backward of an unsplit mask (no global key tiles split over query chunks) also runs
# persistent CTAs beyond one wave: dK and dV bitwise those of one CTA per key tile, dQ (fp32
# reductions in another order) within the parity tolerance.  Adds key tiles no query sees
# (Nq < Nk causal: zero dK, dV) and D = 64 (dQ^T of two steps per UMMA group).
BWD_PERSIST_CASES = PERSIST_CASES[:4] + [
    (I.Problem(1, 32, 900, 1300, 128, True), 200, -1, 130, True),
    (I.Problem(1, 16, 2000, 2000, 64, True), 256, -1, 0, False),
]


@pytest.mark.parametrize("p,wl,wr,g,with_oracle", BWD_PERSIST_CASES,
                         ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in BWD_PERSIST_CASES])
def test_window_backward_persistent_equals_one_cta_per_tile(p, wl, wr, g, with_oracle):
    q, k, v, do = I.draw(p, 8)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qg)
    lse = torch.empty((p.B, p.H, p.Nq), dtype=torch.float32, device=dev)
    _lib.fa_fwd_window(qg, kg, vg, o, lse, p.causal, wl, wr, g, p.scale)
    outs = {}
    prev = _lib.fa_set_bwd_persistent(True)
    try:
        for on in (True, False):
            _lib.fa_set_bwd_persistent(on)
            dq, dk, dv = (torch.full_like(t, float("nan")) for t in (qg, kg, vg))
            _lib.fa_bwd_window(qg, kg, vg, o, lse, dog, dq, dk, dv, p.causal, wl, wr, g, p.scale)
            torch.cuda.synchronize()
            outs[on] = (dq, dk, dv)
    finally:
        _lib.fa_set_bwd_persistent(prev)
    assert torch.equal(outs[True][1], outs[False][1]), "dK"
    assert torch.equal(outs[True][2], outs[False][2]), "dV"
    assert_close("persistent dQ vs one CTA per tile", f64(outs[True][0]), f64(outs[False][0]))
    if with_oracle:
        qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
        rdq, rdk, rdv = masked_ref.attention_backward(qd, kd, vd, dod, p.scale, p.causal, wl, wr, g)
        assert_close("persistent dQ", f64(outs[True][0]), rdq)
        assert_close("persistent dK", f64(outs[True][1]), rdk)
        assert_close("persistent dV", f64(outs[True][2]), rdv)


# Split global key tiles (global tokens, more than 64 query steps) in the persistent
# backward: their chunks add partial dK, dV into the fp32 area in no fixed order, so those
# rows (the first ceil(G/128) key tiles) agree within tolerance; every other row bitwise.
BWD_PERSIST_SPLIT_CASES = [
    (I.Problem(1, 8, 4200, 4200, 64, True), 300, -1, 64),
    (I.Problem(1, 5, 4500, 4500, 128, False), 200, 100, 150),
]


@pytest.mark.parametrize("p,wl,wr,g", BWD_PERSIST_SPLIT_CASES,
                         ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in BWD_PERSIST_SPLIT_CASES])
def test_window_backward_persistent_with_split_key_tiles(p, wl, wr, g):
    assert _lib.fa_bwd_window_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D, wl, wr, g) > \
        _lib.fa_bwd_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D), "the case must split"
    q, k, v, do = I.draw(p, 9)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o = torch.empty_like(qg)
    lse = torch.empty((p.B, p.H, p.Nq), dtype=torch.float32, device=dev)
    _lib.fa_fwd_window(qg, kg, vg, o, lse, p.causal, wl, wr, g, p.scale)
    outs = {}
    prev = _lib.fa_set_bwd_persistent(True)
    try:
        for on in (True, False):
            _lib.fa_set_bwd_persistent(on)
            dq, dk, dv = (torch.full_like(t, float("nan")) for t in (qg, kg, vg))
            _lib.fa_bwd_window(qg, kg, vg, o, lse, dog, dq, dk, dv, p.causal, wl, wr, g, p.scale)
            torch.cuda.synchronize()
            outs[on] = (dq, dk, dv)
    finally:
        _lib.fa_set_bwd_persistent(prev)
    ks = (g + 127) // 128 * 128  # rows of the split global key tiles
    for n, i in (("dK", 1), ("dV", 2)):
        a, b = outs[True][i], outs[False][i]
        assert torch.equal(a[:, :, ks:], b[:, :, ks:]), f"{n} outside the split tiles"
        assert_close(f"{n} of the split tiles", f64(a[:, :, :ks]), f64(b[:, :, :ks]))
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    rdq, rdk, rdv = masked_ref.attention_backward(qd, kd, vd, dod, p.scale, p.causal, wl, wr, g)
    assert_close("persistent dQ", f64(outs[True][0]), rdq)
    assert_close("persistent dK", f64(outs[True][1]), rdk)
    assert_close("persistent dV", f64(outs[True][2]), rdv)


# Split global query rows (non-causal, global tokens, more than 32 key tiles) in the
# persistent forward: the key chunks' partial records are the one-CTA kernel's and
# combine_kernel merges them in a fixed order, so O and L agree bit for bit.
FWD_PERSIST_SPLIT_CASES = [
    (I.Problem(1, 24, 4500, 4500, 64, False), 200, 200, 128, True),
    (I.Problem(2, 10, 4200, 4200, 128, False), 300, 100, 300, False),
]


@pytest.mark.parametrize("p,wl,wr,g,with_oracle", FWD_PERSIST_SPLIT_CASES,
                         ids=[f"{c[0].name()}-wl{c[1]}-wr{c[2]}-g{c[3]}" for c in FWD_PERSIST_SPLIT_CASES])
def test_window_forward_persistent_with_split_rows(p, wl, wr, g, with_oracle):
    assert _lib.fa_fwd_window_workspace_size(p.B, p.H, p.Nq, p.Nk, p.D, p.causal, wl, wr, g) > 0, "must split"
    test_window_forward_persistent_equals_one_cta_per_pair(p, wl, wr, g, with_oracle)
