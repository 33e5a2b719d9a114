"""GPU parity for packed variable-length batches (fa_fwd_varlen / fa_bwd_varlen).

Same acceptance as the dense parity tests: O, dQ, dK, dV relative-L2 <= 1e-2 and
max-abs <= 2e-2 * max|ref| per output, the row logsumexp within 1e-3.  The oracle
attends each (sequence, head) on its own in fp64.  Length mixes cover single-token
sequences, tile edges (127/128/129), several tiles with a ragged tail, empty
sequences, and cross attention with different query and key lengths.
"""
import numpy as np
import pytest
import torch

import oracle
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


def run_varlen(q, k, v, do, cu_q, cu_k, causal, scale, sentinel=float("nan")):
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    cq, ck = cu_q.to(dev), cu_k.to(dev)
    lens_q, lens_k = np.diff(cu_q.numpy()), np.diff(cu_k.numpy())
    mq, mk = max(int(lens_q.max()), 1), max(int(lens_k.max()), 1)
    # outputs start as NaN so that a row the kernels never write shows up
    o = torch.full_like(qg, sentinel)
    lse = torch.full((q.shape[1], q.shape[0]), sentinel, dtype=torch.float32, device=dev)
    _lib.fa_fwd_varlen(qg, kg, vg, o, lse, cq, ck, mq, mk, causal, scale)
    dq, dk, dv = (torch.full_like(t, sentinel) for t in (qg, kg, vg))
    _lib.fa_bwd_varlen(qg, kg, vg, o, lse, dog, dq, dk, dv, cq, ck, mq, mk, causal, scale)
    torch.cuda.synchronize()
    return o, lse, dq, dk, dv


def check_varlen(lens_q, lens_k, H, D, causal, seed, factor=1.0):
    q, k, v, do, cu_q, cu_k = I.draw_varlen(lens_q, lens_k, H, D, seed, factor)
    scale = 1.0 / np.sqrt(D)
    o, lse, dq, dk, dv = run_varlen(q, k, v, do, cu_q, cu_k, causal, scale)
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    ro, rl, rdq, rdk, rdv = oracle.attention_varlen(qd, kd, vd, dod, cu_q.numpy(), cu_k.numpy(), scale, causal)
    tag = f"q{lens_q}k{lens_k}H{H}D{D}{'c' if causal else 'n'}s{seed}"
    assert_close(tag + " O", f64(o), ro)
    gl = f64(lse)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(gl), ~fin), f"{tag}: -inf pattern of L"
    if fin.any():
        e = np.abs(gl[fin] - rl[fin]).max()
        assert e <= LSE_ABS, f"{tag} L: max_abs={e:.3e}"
    assert_close(tag + " dQ", f64(dq), rdq)
    assert_close(tag + " dK", f64(dk), rdk)
    assert_close(tag + " dV", f64(dv), rdv)


MIX = [1, 127, 128, 129, 300, 1000]


@pytest.mark.parametrize("D", [16, 64, 128])
@pytest.mark.parametrize("causal", [False, True])
def test_length_mix(D, causal):
    check_varlen(MIX, MIX, 2, D, causal, seed=D)


@pytest.mark.parametrize("causal", [False, True])
def test_cross_lengths(causal):
    # different query and key lengths per sequence, both directions
    check_varlen([200, 77, 1, 513], [77, 200, 300, 129], 3, 64, causal, seed=5)


@pytest.mark.parametrize("D", [32, 128])
def test_empty_sequences(D):
    # empty sequences at the start, middle and end; one with queries but no keys
    check_varlen([0, 5, 0, 130, 64, 0], [0, 5, 7, 130, 0, 3], 2, D, True, seed=11)
    check_varlen([0, 5, 0, 130, 64, 0], [0, 5, 7, 130, 0, 3], 2, D, False, seed=12)


def test_many_short_sequences():
    rng = np.random.default_rng(3)
    lens = rng.integers(1, 90, size=40).tolist()
    check_varlen(lens, lens, 2, 128, True, seed=13)


def test_thousands_of_sequences():
    # more than 1024 sequences (three rounds of the kernels' 32-way slot search), empty
    # ones among them
    rng = np.random.default_rng(4)
    lens = rng.integers(0, 40, size=1100).tolist()
    check_varlen(lens, lens, 2, 64, True, seed=15)


# more (slot, head) units than SMs: forward and backward run persistent CTAs by default
PERSIST_VARLEN = [(MIX, MIX, 16, 128, True), (MIX, MIX, 16, 64, False),
                  ([0, 5, 0, 130, 64, 0], [0, 5, 7, 130, 0, 3], 40, 32, True),
                  ([200, 77, 1, 513], [77, 200, 300, 129], 40, 16, True),
                  (I.doc_lengths(4096, seed=9), I.doc_lengths(4096, seed=9), 8, 128, True)]


@pytest.mark.parametrize("case", PERSIST_VARLEN, ids=[f"H{c[2]}D{c[3]}{'c' if c[4] else 'n'}-{i}"
                                                      for i, c in enumerate(PERSIST_VARLEN)])
def test_persistent_equals_one_cta_per_unit(case):
    # the persistent schedule changes which SM runs a unit, never its arithmetic: O, L, dK
    # and dV bitwise equal to one CTA per slot, dQ equal up to the order in which key tiles
    # add into it, and all of them match the oracle
    lens_q, lens_k, H, D, causal = case
    q, k, v, do, cu_q, cu_k = I.draw_varlen(lens_q, lens_k, H, D, 17, 1.0)
    assert (sum(lens_q) // 256 + len(lens_q)) * H > 152 and (sum(lens_k) // 128 + len(lens_k)) * H > 152
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    cq, ck = cu_q.to(dev), cu_k.to(dev)
    mq, mk = max(max(lens_q), 1), max(max(lens_k), 1)
    scale = 1.0 / np.sqrt(D)
    outs = []
    prev = (_lib.fa_set_fwd_persistent(False), _lib.fa_set_bwd_persistent(False))
    try:
        for on in (False, True):
            _lib.fa_set_fwd_persistent(on)
            _lib.fa_set_bwd_persistent(on)
            o = torch.full_like(qg, float("nan"))
            lse = torch.full((H, q.shape[0]), float("nan"), dtype=torch.float32, device=dev)
            _lib.fa_fwd_varlen(qg, kg, vg, o, lse, cq, ck, mq, mk, causal, scale)
            dq, dk, dv = (torch.full_like(t, float("nan")) for t in (qg, kg, vg))
            _lib.fa_bwd_varlen(qg, kg, vg, o, lse, dog, dq, dk, dv, cq, ck, mq, mk, causal, scale)
            outs.append((o, lse, dq, dk, dv))
        torch.cuda.synchronize()
    finally:
        _lib.fa_set_fwd_persistent(prev[0])
        _lib.fa_set_bwd_persistent(prev[1])
    (o1, l1, dq1, dk1, dv1), (o2, l2, dq2, dk2, dv2) = outs
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    assert torch.equal(dk1, dk2) and torch.equal(dv1, dv2)
    err = (dq1.float() - dq2.float()).abs().max().item()
    assert err <= 1e-2 * max(dq1.float().abs().max().item(), 1e-30), err
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    ro, rl, rdq, rdk, rdv = oracle.attention_varlen(qd, kd, vd, dod, cu_q.numpy(), cu_k.numpy(), scale, causal)
    tag = f"H{H}D{D}"
    assert_close(tag + " O", f64(o2), ro)
    gl = f64(l2)
    fin = np.isfinite(rl)
    assert np.array_equal(np.isneginf(gl), ~fin)
    if fin.any():
        assert np.abs(gl[fin] - rl[fin]).max() <= LSE_ABS
    assert_close(tag + " dQ", f64(dq2), rdq)
    assert_close(tag + " dK", f64(dk2), rdk)
    assert_close(tag + " dV", f64(dv2), rdv)


def test_scaled_inputs_peaked_softmax():
    check_varlen([129, 700, 33], [129, 700, 33], 2, 128, True, seed=14, factor=8.0)


def test_equal_lengths_match_dense_path():
    # a packed batch of equal lengths computes exactly what the dense layout does:
    # the same kernels on the same tiles, so the bf16 outputs agree bit for bit
    p = I.Problem(3, 2, 300, 300, 64, True)
    q, k, v, do = I.draw(p, 21)
    dev = torch.device("cuda")
    qg, kg, vg, dog = (t.to(dev) for t in (q, k, v, do))
    o, lse = _lib.forward(qg, kg, vg, True, p.scale)
    dq, dk, dv = _lib.backward(qg, kg, vg, o, lse, dog, True, p.scale)
    pack = lambda t: t.transpose(1, 2).reshape(p.B * p.Nq, p.H, p.D).contiguous()  # noqa: E731
    cu = torch.arange(p.B + 1, dtype=torch.int32) * p.Nq
    vo, vl, vdq, vdk, vdv = run_varlen(*(pack(t).cpu() for t in (q, k, v, do)), cu, cu, True, p.scale)
    assert torch.equal(vo, pack(o))
    assert torch.equal(vl, lse.transpose(0, 1).reshape(p.H, p.B * p.Nq))
    assert torch.equal(vdq, pack(dq)) and torch.equal(vdk, pack(dk)) and torch.equal(vdv, pack(dv))


def test_long_sequence_sampled_rows():
    # one long sequence between two short ones: check sampled query rows of the long one
    lens = [50, 8300, 70]
    H, D = 2, 128
    q, k, v, do, cu_q, cu_k = I.draw_varlen(lens, lens, H, D, 31)
    scale = 1.0 / np.sqrt(D)
    o, lse, dq, dk, dv = run_varlen(q, k, v, do, cu_q, cu_k, True, scale)
    qd, kd, vd, dod = (I.as_f64(t) for t in (q, k, v, do))
    a, b = 50, 8350
    rows = np.array([0, 127, 128, 4095, 8191, 8192, 8299])
    for h in range(H):
        ro, rl = oracle.forward_head(qd[a:b, h], kd[a:b, h], vd[a:b, h], scale, True, rows=rows)
        assert_close(f"long h{h} O", f64(o)[a:b, h][rows], ro)
        assert np.abs(f64(lse)[h, a:b][rows] - rl).max() <= LSE_ABS
    # the short neighbours in full
    for lo, hi in ((0, 50), (8350, 8420)):
        ro, rl, rdq, rdk, rdv = oracle.attention_varlen(qd[lo:hi], kd[lo:hi], vd[lo:hi], dod[lo:hi],
                                                        [0, hi - lo], [0, hi - lo], scale, True)
        assert_close(f"nb{lo} O", f64(o)[lo:hi], ro)
        assert_close(f"nb{lo} dQ", f64(dq)[lo:hi], rdq)
        assert_close(f"nb{lo} dK", f64(dk)[lo:hi], rdk)
        assert_close(f"nb{lo} dV", f64(dv)[lo:hi], rdv)
    # properties over the long sequence: sum_j dK_j = 0, sum_j dV_j = sum_i dO_i
    dkl, dvl, dol = (t.double()[a:b] for t in (dk.cpu(), dv.cpu(), do))
    assert ((dkl.sum(0).abs() / dkl.abs().sum(0).clamp_min(1e-30)).max() < 5e-3)
    assert (((dvl.sum(0) - dol.sum(0)).abs() / dol.abs().sum(0).clamp_min(1e-30)).max() < 5e-3)


def test_varlen_validation_on_device():
    dev = torch.device("cuda")
    q = torch.zeros(10, 2, 64, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(2, 10, device=dev)
    cu = torch.tensor([0, 4, 10], dtype=torch.int32, device=dev)
    with pytest.raises(RuntimeError):
        _lib.fa_fwd_varlen(q, q, q, q, lse, cu, cu, 6, 6, True)  # o aliases q
    with pytest.raises(RuntimeError):
        _lib.fa_fwd_varlen(q, q, q, o, lse, cu, cu, 0, 6, True)  # max_seqlen_q = 0
    _lib.fa_fwd_varlen(q, q, q, o, lse, cu, cu, 6, 6, True)
    torch.cuda.synchronize()
    assert torch.all(o == 0)  # zero V
