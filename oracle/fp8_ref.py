"""Plain CPU oracle for the FP8 (e4m3) forward with per-tensor scales.

TEST INFRASTRUCTURE ONLY.  Nothing on the product path imports or calls this
module: only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py``'s
``cpu_baseline`` / reference arm may.  It shares no code with the CUDA path.

The pages name FP8 only as a direction: combining the method with quantised
formats such as FP8 ("FlashAttention技术演进全景图" §5.3 未来优化方向).  The reading
taken here is the usual per-tensor one:

  * e4m3 ("fn" variant): 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits;
    exponent field 0 holds the subnormals m/8 * 2^-6; exponent 15 with mantissa 7
    is NaN; there is no infinity; the largest finite value is 448.
  * Per-tensor quantisation of a tensor x (values taken in float32):
        amax = max |x|;  mult = float32(448 / amax);  descale = float32(amax / 448)
        code = e4m3(float32(x * mult))   (round to nearest, ties to even, saturating)
    so that x ~= descale * value(code).  An all-zero tensor uses mult = descale = 1.
    Both divisions and the product are single IEEE float32 operations, so the codes
    are fixed bit for bit.
  * Attention on the quantised inputs: Q, K, V are taken as descale * value(code)
    (exact in float64) and the plain definition of ``attn_ref`` is applied to them,
    with the caller's softmax scale.

Pins: ``tests/test_oracle_fp8_pins.py``.
"""
from __future__ import annotations

import numpy as np

from . import attn_ref

E4M3_MAX = 448.0


def e4m3_value(code):
    """Value of each e4m3 code (uint8 array), from the bit fields; NaN for the NaN codes."""
    c = np.asarray(code, np.uint8).astype(np.int64)
    s = np.where(c & 0x80, -1.0, 1.0)
    e = (c >> 3) & 0xF
    m = c & 0x7
    normal = s * np.ldexp(1.0 + m / 8.0, e - 7)
    sub = s * np.ldexp(m / 8.0, -6)
    v = np.where(e == 0, sub, normal)
    return np.where((e == 15) & (m == 7), np.nan, v)


# the 127 non-negative finite values, ascending, with their codes 0x00..0x7E
_POS_CODES = np.arange(0x7F, dtype=np.uint8)
_POS_VALUES = e4m3_value(_POS_CODES)


def e4m3_encode(x):
    """Round float values to e4m3 codes: nearest, ties to the even code, saturating at
    +-448; NaN maps to 0x7F.  Works on any float array (the float32 values the kernels see)."""
    x = np.asarray(x, np.float64)
    a = np.minimum(np.abs(x), E4M3_MAX)
    hi = np.clip(np.searchsorted(_POS_VALUES, a, side="left"), 0, 126)  # first value >= a
    lo = np.maximum(hi - 1, 0)
    d_hi = _POS_VALUES[hi] - a
    d_lo = a - _POS_VALUES[lo]
    pick_hi = (d_hi < d_lo) | ((d_hi == d_lo) & (_POS_CODES[hi] % 2 == 0))
    code = np.where(pick_hi, _POS_CODES[hi], _POS_CODES[lo]).astype(np.uint8)
    code = np.where(np.signbit(x) & (code != 0), code | 0x80, code).astype(np.uint8)
    code = np.where(np.signbit(x) & (code == 0), np.uint8(0x80), code).astype(np.uint8)
    return np.where(np.isnan(x), np.uint8(0x7F), code).astype(np.uint8)


def quantize_per_tensor(x):
    """(codes uint8, descale float32) for a float tensor, as the module docstring defines."""
    x32 = np.asarray(x, np.float32)
    amax = np.float32(np.max(np.abs(x32))) if x32.size else np.float32(0)
    if amax == 0:
        mult = descale = np.float32(1.0)
    else:
        mult = np.float32(np.float32(E4M3_MAX) / amax)
        descale = np.float32(amax / np.float32(E4M3_MAX))
    y = (x32 * mult).astype(np.float32)  # one float32 multiply per element
    return e4m3_encode(y), descale


def dequantize(codes, descale):
    """descale * value(code), exact in float64."""
    return np.float64(descale) * e4m3_value(codes)


def forward(q_codes, k_codes, v_codes, q_descale, k_descale, v_descale, scale, causal, row_chunk=1024):
    """O [B,H,Nq,D] and L [B,H,Nq] of attention on the dequantised inputs."""
    q = dequantize(q_codes, q_descale)
    k = dequantize(k_codes, k_descale)
    v = dequantize(v_codes, v_descale)
    return attn_ref.attention_forward(q, k, v, scale, causal, row_chunk=row_chunk)


def forward_head(q_codes, k_codes, v_codes, q_descale, k_descale, v_descale, scale, causal, rows=None,
                 row_chunk=1024):
    """One head ([N, D] code arrays); ``rows`` selects query rows."""
    return attn_ref.forward_head(dequantize(q_codes, q_descale), dequantize(k_codes, k_descale),
                                 dequantize(v_codes, v_descale), scale, causal, rows=rows, row_chunk=row_chunk)
