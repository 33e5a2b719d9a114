"""GPU parity for the FP8 (e4m3) path: per-tensor quantisation and the FP8 forward.

* Quantisation is byte work: fa_quantize_e4m3 / _transposed must produce the oracle's
  codes bit for bit, and the same fp32 descale.
* The FP8 forward runs on codes made by the oracle (uploaded, so no oracle input comes
  from the CUDA path) and is compared with the oracle's attention on the dequantised
  inputs.  Tolerance, derived from the arithmetic: P is rounded to e4m3 (relative step
  up to 2^-4), which moves O by ~2-3% RMS on rows spread over many keys; so O rel-L2
  <= 5e-2 and max-abs <= 6e-2 * max|ref|.  S is exact up to fp32 accumulation, so L
  keeps the 1e-3 bound.  Rows dominated by one key (x8 logits) must come out far
  tighter: rel-L2 <= 1e-2.
"""
import numpy as np
import pytest
import torch

from oracle import fp8_ref
from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300 import inputs as I
from tiled_attention_11_gb300.build import build

pytestmark = pytest.mark.gpu

REL_L2 = 5e-2
MAX_FRAC = 6e-2
LSE_ABS = 1e-3


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


def err(got, ref):
    e = np.asarray(got, np.float64) - ref
    return np.linalg.norm(e) / np.linalg.norm(ref), np.abs(e).max() / np.abs(ref).max()


def oracle_codes(x_bf16):
    return fp8_ref.quantize_per_tensor(x_bf16.to(torch.float32).numpy())


@pytest.mark.parametrize("shape,mult", [((2, 3, 100, 64), 1.0), ((1, 1, 1, 128), 3.0), ((1, 2, 257, 128), 1e-3),
                                        ((3, 1, 33, 64), 700.0)])
def test_quantize_bit_exact(shape, mult):
    g = torch.Generator().manual_seed(sum(shape))
    x = (torch.randn(shape, generator=g) * mult).to(torch.bfloat16)
    codes, amax, descale = _lib.quantize_e4m3(x.cuda())
    want, wd = oracle_codes(x)
    torch.cuda.synchronize()
    assert np.array_equal(codes.cpu().numpy(), want)
    assert descale.cpu().numpy()[0].view(np.uint32) == np.float32(wd).view(np.uint32)
    assert amax.cpu().item() == np.abs(x.to(torch.float32).numpy()).max()


def test_quantize_flat_tail_and_zeros():
    x = torch.zeros(1003, dtype=torch.bfloat16)  # not a multiple of 8; all zero
    codes, _, descale = _lib.quantize_e4m3(x.cuda())
    torch.cuda.synchronize()
    assert int(codes.cpu().max()) == 0 and descale.item() == 1.0
    x[1002] = -3.0
    codes, _, descale = _lib.quantize_e4m3(x.cuda())
    want, wd = oracle_codes(x)
    assert np.array_equal(codes.cpu().numpy(), want) and descale.item() == wd


@pytest.mark.parametrize("shape", [(2, 2, 100, 64), (1, 3, 129, 128), (1, 1, 16, 128), (2, 1, 1000, 64)])
def test_quantize_transposed_bit_exact(shape):
    g = torch.Generator().manual_seed(7 + sum(shape))
    v = torch.randn(shape, generator=g).to(torch.bfloat16)
    codes_t, ldt, _, descale = _lib.quantize_e4m3_transposed(v.cuda())
    want, wd = oracle_codes(v)
    N = shape[2]
    got = codes_t.cpu().numpy()[..., :N]
    assert ldt % 16 == 0 and ldt >= N
    assert np.array_equal(got, want.transpose(0, 1, 3, 2))
    assert descale.item() == wd


# the three tensors of one call in one launch pair: Nq != Nk, ragged key slabs (not a
# multiple of 128 or of 16), a single key, an all-zero tensor, wide value ranges
QKV_CASES = [((2, 3, 257, 1000, 128), (1.0, 1.0, 1.0)), ((1, 2, 100, 129, 64), (3.0, 1e-3, 700.0)),
             ((1, 1, 1, 1, 128), (1.0, 2.0, 0.5)), ((3, 2, 4099, 300, 64), (0.0, 1.0, 5.0)),
             ((1, 4, 64, 4096, 128), (1.0, 0.0, 0.0))]


@pytest.mark.parametrize("shape,mults", QKV_CASES)
def test_quantize_qkv_bit_exact(shape, mults):
    B, H, Nq, Nk, D = shape
    g = torch.Generator().manual_seed(3 + sum(shape))
    q, k, v = ((torch.randn((B, H, n, D), generator=g) * m).to(torch.bfloat16)
               for n, m in ((Nq, mults[0]), (Nk, mults[1]), (Nk, mults[2])))
    q8, k8, vt8, ldv, amax, descale = _lib.quantize_qkv_e4m3(q.cuda(), k.cuda(), v.cuda())
    torch.cuda.synchronize()
    assert ldv % 16 == 0 and Nk <= ldv < Nk + 16
    vt = vt8.cpu().numpy()
    for t, (x, got) in enumerate(((q, q8.cpu().numpy()), (k, k8.cpu().numpy()), (v, vt[..., :Nk]))):
        want, wd = oracle_codes(x)
        if t == 2:
            want = want.transpose(0, 1, 3, 2)
            assert int(vt[..., Nk:].max(initial=0)) == 0  # keys past Nk up to ldv: zero codes
        assert np.array_equal(got, want), f"tensor {t}"
        assert descale.cpu().numpy()[t].view(np.uint32) == np.float32(wd).view(np.uint32)
        assert amax.cpu().numpy()[t] == np.abs(x.to(torch.float32).numpy()).max()


def test_quantize_qkv_equals_separate_calls():
    p = I.Problem(2, 8, 1500, 1500, 128, True)
    q, k, v = (t.cuda() for t in I.draw(p, 5)[:3])
    q8, k8, vt8, ldv, _, descale = _lib.quantize_qkv_e4m3(q, k, v)
    sq, _, dq = _lib.quantize_e4m3(q)
    sk, _, dk = _lib.quantize_e4m3(k)
    svt, sldv, _, dv = _lib.quantize_e4m3_transposed(v)
    torch.cuda.synchronize()
    assert ldv == sldv
    assert torch.equal(q8, sq) and torch.equal(k8, sk) and torch.equal(vt8, svt)
    assert torch.equal(descale, torch.cat([dq, dk, dv]))


def run_fp8(p, seed):
    q, k, v, _ = I.draw(p, seed)
    (q8, qd), (k8, kd), (v8, vd) = oracle_codes(q), oracle_codes(k), oracle_codes(v)
    dev = torch.device("cuda")
    ldv = (p.Nk + 15) // 16 * 16
    vt = np.zeros((p.B, p.H, p.D, ldv), np.uint8)
    vt[..., :p.Nk] = v8.transpose(0, 1, 3, 2)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    sc = lambda d: torch.tensor([d], dtype=torch.float32, device=dev)  # noqa: E731
    o = torch.full((p.B, p.H, p.Nq, p.D), float("nan"), dtype=torch.bfloat16, device=dev)
    lse = torch.full((p.B, p.H, p.Nq), float("nan"), dtype=torch.float32, device=dev)
    _lib.fa_fwd_fp8(t(q8), t(k8), t(vt), ldv, sc(qd), sc(kd), sc(vd), o, lse, p.causal, p.scale)
    torch.cuda.synchronize()
    return (q8, k8, v8, qd, kd, vd), f64(o), f64(lse)


def check_fp8(p, seed=0, rel=REL_L2, frac=MAX_FRAC):
    (q8, k8, v8, qd, kd, vd), o, lse = run_fp8(p, seed)
    ro, rl = fp8_ref.forward(q8, k8, v8, qd, kd, vd, p.scale, p.causal)
    assert np.isfinite(o).all() and np.isfinite(lse).all()
    r, a = err(o, ro)
    assert r <= rel and a <= frac, f"{p.name()}: O rel_l2={r:.3e} max_frac={a:.3e}"
    e = np.abs(lse - rl).max()
    assert e <= LSE_ABS, f"{p.name()}: L max_abs={e:.3e}"
    return r, a


CASES = [I.Problem(1, 2, n, n, d, c) for d in (64, 128) for c in (False, True) for n in (1, 127, 128, 129, 300, 1000)]
CASES += [I.Problem(2, 3, 200, 77, 128, True), I.Problem(2, 3, 77, 200, 64, True), I.Problem(1, 2, 77, 513, 128, False),
          I.Problem(2, 2, 4096, 4096, 128, True)]


@pytest.mark.parametrize("p", CASES, ids=[p.name() for p in CASES])
def test_fp8_forward(p):
    check_fp8(p)


@pytest.mark.parametrize("D", [64, 128])
def test_fp8_peaked_rows_are_tight(D):
    # x8 logits: every row is dominated by one key, whose weight the e4m3 normalisation
    # keeps exact; the remaining error is bf16 rounding and the neighbours' tiny weights
    check_fp8(I.Problem(1, 2, 640, 640, D, True, qk_factor=8.0), seed=3, rel=1e-2, frac=2e-2)


def test_fp8_end_to_end_from_bf16():
    # bf16 -> the GPU quantisers -> FP8 forward, against the oracle on the oracle's codes
    p = I.Problem(1, 4, 700, 700, 128, True)
    q, k, v, _ = I.draw(p, 9)
    dev = torch.device("cuda")
    o, lse = _lib.forward_fp8(q.to(dev), k.to(dev), v.to(dev), True, p.scale)
    torch.cuda.synchronize()
    (q8, qd), (k8, kd), (v8, vd) = oracle_codes(q), oracle_codes(k), oracle_codes(v)
    ro, rl = fp8_ref.forward(q8, k8, v8, qd, kd, vd, p.scale, True)
    r, a = err(f64(o), ro)
    assert r <= REL_L2 and a <= MAX_FRAC and np.abs(f64(lse) - rl).max() <= LSE_ABS


def test_fp8_long_sampled_rows():
    p = I.Problem(1, 2, 16384, 16384, 128, True)
    q, k, v, _ = I.draw(p, 11)
    (q8, k8, v8, qd, kd, vd), o, lse = run_fp8(p, 11)
    rows = np.array([0, 1, 127, 128, 8191, 16383])
    for h in range(p.H):
        ro, rl = fp8_ref.forward_head(q8[0, h], k8[0, h], v8[0, h], qd, kd, vd, p.scale, True, rows=rows)
        r, a = err(o[0, h][rows], ro)
        assert r <= REL_L2 and a <= MAX_FRAC, f"h{h}: rel {r:.3e} frac {a:.3e}"
        assert np.abs(lse[0, h][rows] - rl).max() <= LSE_ABS


# more (query-tile pair, head) units than SMs: the FP8 forward runs persistent CTAs by default
PERSIST_CASES = [I.Problem(2, 16, 2048, 2048, 128, True), I.Problem(4, 16, 1100, 1100, 64, False),
                 I.Problem(8, 32, 300, 300, 128, True), I.Problem(4, 16, 700, 1500, 64, True)]


@pytest.mark.parametrize("p", PERSIST_CASES, ids=[p.name() for p in PERSIST_CASES])
def test_fp8_persistent_equals_one_cta_per_unit(p):
    # the persistent schedule changes which SM runs a unit, never its arithmetic: O and L
    # bitwise equal to one CTA per unit, and the oracle agrees on the first and last head
    assert p.B * p.H * ((p.Nq + 255) // 256) > 152
    q, k, v, _ = I.draw(p, 19)
    (q8, qd), (k8, kd), (v8, vd) = oracle_codes(q), oracle_codes(k), oracle_codes(v)
    dev = torch.device("cuda")
    ldv = (p.Nk + 15) // 16 * 16
    vt = np.zeros((p.B, p.H, p.D, ldv), np.uint8)
    vt[..., :p.Nk] = v8.transpose(0, 1, 3, 2)
    t = lambda a: torch.from_numpy(np.ascontiguousarray(a)).to(dev)  # noqa: E731
    sc = lambda d: torch.tensor([d], dtype=torch.float32, device=dev)  # noqa: E731
    args = (t(q8), t(k8), t(vt), ldv, sc(qd), sc(kd), sc(vd))
    outs = []
    prev = _lib.fa_set_fwd_persistent(False)
    try:
        for on in (False, True):
            _lib.fa_set_fwd_persistent(on)
            o = torch.full((p.B, p.H, p.Nq, p.D), float("nan"), dtype=torch.bfloat16, device=dev)
            lse = torch.full((p.B, p.H, p.Nq), float("nan"), dtype=torch.float32, device=dev)
            _lib.fa_fwd_fp8(*args, o, lse, p.causal, p.scale)
            outs.append((o, lse))
        torch.cuda.synchronize()
    finally:
        _lib.fa_set_fwd_persistent(prev)
    (o1, l1), (o2, l2) = outs
    assert torch.equal(o1, o2) and torch.equal(l1, l2)
    for (b, h) in ((0, 0), (p.B - 1, p.H - 1)):
        ro, rl = fp8_ref.forward_head(q8[b, h], k8[b, h], v8[b, h], qd, kd, vd, p.scale, p.causal)
        r, a = err(f64(o2[b, h]), ro)
        assert r <= REL_L2 and a <= MAX_FRAC, f"{p.name()} b{b}h{h}: rel {r:.3e} frac {a:.3e}"
        assert np.abs(f64(l2[b, h]) - rl).max() <= LSE_ABS
