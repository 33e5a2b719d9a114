"""Pins for the FP8 (e4m3) oracle (``oracle.fp8_ref``).

* the e4m3 value table against hand-derived values and against PyTorch's
  float8_e4m3fn (a library routine for the same format), all 256 codes;
* encoding: every finite code round-trips, midpoints between neighbours go to the
  even code, out-of-range values saturate, and random float32 values encode as
  PyTorch rounds them;
* per-tensor quantisation: the largest magnitude maps to +-448, the dequantised
  error stays within half a unit in the last place, exactly representable inputs
  come back unchanged, an all-zero tensor is handled;
* the FP8 forward on exactly representable inputs equals the plain oracle.
``test_planted_mistakes_are_caught`` plants mistakes in a copy of the module.
"""
import types

import numpy as np
import pytest
import torch

from oracle import attn_ref, fp8_ref


def torch_values(codes):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def pin_value_table(ref):
    codes = np.arange(256, dtype=np.uint8)
    mine, lib = ref.e4m3_value(codes), torch_values(codes)
    ok = np.array_equal(np.isnan(mine), np.isnan(lib)) and np.array_equal(mine[~np.isnan(mine)], lib[~np.isnan(lib)])
    hand = {0x00: 0.0, 0x01: 2.0 ** -9, 0x07: 7 * 2.0 ** -9, 0x08: 2.0 ** -6, 0x38: 1.0, 0x3C: 1.5, 0x7E: 448.0,
            0x80: -0.0, 0xB8: -1.0, 0xFE: -448.0}
    ok &= all(ref.e4m3_value(np.uint8(c)) == v for c, v in hand.items())
    ok &= bool(np.isnan(ref.e4m3_value(np.uint8(0x7F))) and np.isnan(ref.e4m3_value(np.uint8(0xFF))))
    return bool(ok)


def pin_encode(ref):
    ok = True
    finite = np.array([c for c in range(256) if c not in (0x7F, 0xFF)], np.uint8)
    vals = ref.e4m3_value(finite)
    ok &= np.array_equal(ref.e4m3_encode(vals), finite)  # includes -0 -> 0x80
    # midpoints between neighbouring positive values: ties go to the even code
    pos = ref.e4m3_value(np.arange(0x7F, dtype=np.uint8))
    mids = (pos[:-1] + pos[1:]) / 2
    lo_codes = np.arange(0x7E, dtype=np.uint8)
    want = np.where(lo_codes % 2 == 0, lo_codes, lo_codes + 1).astype(np.uint8)
    ok &= np.array_equal(ref.e4m3_encode(mids), want)
    ok &= np.array_equal(ref.e4m3_encode(-mids), want | 0x80)
    # saturation and NaN
    ok &= np.array_equal(ref.e4m3_encode(np.array([448.0, 460.0, 1e6, -1e30])), np.array([0x7E, 0x7E, 0x7E, 0xFE], np.uint8))
    ok &= ref.e4m3_encode(np.array([np.nan]))[0] == 0x7F
    # random float32 values inside the range encode as PyTorch rounds them (nearest-even)
    rng = np.random.default_rng(0)
    x = (rng.standard_normal(20000) * np.exp(rng.uniform(-9, 6, 20000))).astype(np.float32)
    x = x[np.abs(x) <= 440]
    lib = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ok &= np.array_equal(ref.e4m3_encode(x), lib)
    return bool(ok)


def pin_quantize(ref):
    ok = True
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((3, 50)) * 3.0).astype(np.float32)
    codes, descale = ref.quantize_per_tensor(x)
    amax = np.abs(x).max()
    ok &= descale.dtype == np.float32 and descale == np.float32(amax / np.float32(448))
    i = np.unravel_index(np.argmax(np.abs(x)), x.shape)
    ok &= codes[i] == (0x7E if x[i] > 0 else 0xFE)
    # dequantised error: at most half a unit in the last place of the scaled value
    y = x.astype(np.float64) * np.float64(np.float32(448 / amax))
    err = np.abs(ref.e4m3_value(codes) - y)
    ulp = np.where(np.abs(y) >= 2 ** -6, 2.0 ** (np.floor(np.log2(np.maximum(np.abs(y), 2 ** -6))) - 3), 2.0 ** -9)
    ok &= bool(np.all(err <= ulp / 2 * (1 + 1e-6)))
    # values already on the e4m3 grid with amax 448 come back unchanged
    grid = ref.e4m3_value(np.array([0x7E, 0x38, 0xBC, 0x01, 0x80, 0x45], np.uint8)).astype(np.float32)
    c2, d2 = ref.quantize_per_tensor(grid)
    ok &= d2 == np.float32(1.0) and np.array_equal(ref.e4m3_value(c2), grid.astype(np.float64))
    # all zeros: codes 0, descale 1
    c3, d3 = ref.quantize_per_tensor(np.zeros(7, np.float32))
    ok &= bool(np.all(c3 == 0)) and d3 == np.float32(1.0)
    return bool(ok)


def pin_forward_on_grid(ref):
    # inputs on the e4m3 grid quantise exactly, so the FP8 forward equals the plain oracle
    rng = np.random.default_rng(2)
    codes = [rng.integers(0, 0x7F, (1, 2, 9, 4)).astype(np.uint8) | (rng.integers(0, 2, (1, 2, 9, 4)) * 0x80).astype(np.uint8)
             for _ in range(3)]
    for c in codes:
        c[0, 0, 0, 0] = 0x7E  # amax 448 -> descale 1
    x = [ref.e4m3_value(c) for c in codes]
    q8, qs = ref.quantize_per_tensor(x[0])
    k8, ks = ref.quantize_per_tensor(x[1])
    v8, vs = ref.quantize_per_tensor(x[2])
    o, lse = ref.forward(q8, k8, v8, qs, ks, vs, 0.01, True)
    o2, l2 = attn_ref.attention_forward(x[0], x[1], x[2], 0.01, True)
    ok = np.array_equal(q8, codes[0]) and np.allclose(o, o2, atol=1e-13) and np.allclose(lse, l2, atol=1e-13)
    # descales multiply the values
    o3, l3 = ref.forward(q8, k8, v8, np.float32(2.0), np.float32(0.5), np.float32(4.0), 0.01, True)
    ok &= np.allclose(o3, 4.0 * o2, atol=1e-12) and np.allclose(l3, l2, atol=1e-12)
    return bool(ok)


PINS = [pin_value_table, pin_encode, pin_quantize, pin_forward_on_grid]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_fp8_oracle_pin(pin):
    assert pin(fp8_ref)


MUTATIONS = [
    ("exponent bias 8", "normal = s * np.ldexp(1.0 + m / 8.0, e - 7)", "normal = s * np.ldexp(1.0 + m / 8.0, e - 8)"),
    ("subnormal scale 2^-7", "sub = s * np.ldexp(m / 8.0, -6)", "sub = s * np.ldexp(m / 8.0, -7)"),
    ("ties away from zero", "pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))",
     "pick_hi = (d_hi <= d_lo)"),
    ("largest code excluded", "hi = np.clip(np.searchsorted(_POS_VALUES, a, side=\"left\"), 0, 126)",
     "hi = np.clip(np.searchsorted(_POS_VALUES, a, side=\"left\"), 0, 125)"),
    ("descale inverted", "descale = np.float32(amax / np.float32(E4M3_MAX))",
     "descale = np.float32(np.float32(E4M3_MAX) / amax)"),
    ("sign dropped", "code = np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)",
     "code = code.astype(np.uint8)"),
    ("v descale ignored", "v = dequantize(v_codes, v_descale)", "v = dequantize(v_codes, 1.0)"),
    ("truncation instead of rounding", "pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))",
     "pick_hi = d_hi == 0"),
]


def _mutant(src, old, new):
    assert old in src, f"mutation anchor not found: {old!r}"
    src = src.replace(old, new, 1).replace("from . import attn_ref", "from oracle import attn_ref")
    mod = types.ModuleType("fp8_ref_mutant")
    exec(compile(src, "fp8_ref_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistakes_are_caught(name, old, new):
    mut = _mutant(open(fp8_ref.__file__).read(), old, new)
    results = {}
    for pin in PINS:
        try:
            results[pin.__name__] = pin(mut)
        except Exception:  # a crash is also a caught mistake
            results[pin.__name__] = False
    assert not all(results.values()), f"planted mistake '{name}' passed every pin"
