"""The measurement library (libta11_probe.so): its exports and argument checks on the
host, and on the GPU the two roof probes (exp2 rate, UMMA rate)."""
import ctypes
import os
import re

import pytest

from tiled_attention_11_gb300 import probe
from tiled_attention_11_gb300.build import build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
PROBE_H = os.path.join(ROOT, "tiled_attention_11_gb300", "csrc", "probe.h")


def _device_present() -> bool:
    import torch
    return torch.cuda.is_available() or os.path.exists("/dev/nvidiactl")


@pytest.fixture(scope="module")
def P():
    build()
    return probe.lib()


def test_probe_header_matches_exports(P):
    text = re.sub(r"/\*.*?\*/", "", open(PROBE_H).read(), flags=re.S)
    declared = sorted(set(re.findall(r"\b(ta11_probe_[a-z_0-9]+)\s*\(", text)))
    assert declared == sorted(probe.EXPORTED)
    for name in declared:
        assert hasattr(P, name)


def test_attention_library_exports_no_probe():
    from tiled_attention_11_gb300 import _lib
    L = _lib.lib()
    for name in ("fa_ex2_probe", "fa_umma_probe"):
        assert not hasattr(L, name)


def test_probe_argument_checks(P):
    vp = ctypes.c_void_p
    fake = vp(1 << 40)
    assert P.ta11_probe_ex2(None, 4, 8, None) == 1
    assert P.ta11_probe_ex2(fake, 0, 8, None) == 1
    assert P.ta11_probe_ex2(fake, 65536, 8, None) == 1
    assert P.ta11_probe_ex2(fake, 4, 0, None) == 1
    assert P.ta11_probe_ex2(fake, 4, (1 << 20) + 1, None) == 1
    assert P.ta11_probe_ex2(vp((1 << 40) + 2), 4, 8, None) == 3
    assert P.ta11_probe_umma(0, 8, 1000, None) == 1
    assert P.ta11_probe_umma(65536, 8, 1000, None) == 1
    assert P.ta11_probe_umma(4, 0, 1000, None) == 1
    assert P.ta11_probe_umma(4, (1 << 16) + 1, 1000, None) == 1
    if not _device_present():
        assert P.ta11_probe_ex2(fake, 4, 8, None) == 5
        assert P.ta11_probe_umma(4, 8, 1000, None) == 5


@pytest.mark.gpu
def test_ex2_probe_rate_and_values():
    # every chain x <- 2^(-x) contracts to the fixed point x* = 2^(-x*) ~ 0.6412; the rate
    # is the special-function units' (about 32 per SM-clock x 152 SMs x ~2 GHz ~ 1e13 per
    # second; a wide band)
    import torch
    x = 0.5
    for _ in range(200):
        x = 2.0 ** -x
    out = probe.ex2_values(152, 256)
    torch.cuda.synchronize()
    assert torch.allclose(out.double().cpu(), torch.full((152 * 512,), 8 * x, dtype=torch.float64), atol=1e-4)
    assert 1e12 < probe.ex2_rate() < 1e14


@pytest.mark.gpu
def test_umma_probe_rate():
    # the score GEMM's UMMA shape back to back on every SM: within the hardware's range
    # (8192 bf16 FLOP per SM-clock x 152 SMs x ~2 GHz ~ 2.5 PFLOP/s), no timeout recorded
    probe.status(reset=True)
    rate = probe.umma_rate(iters=256)
    assert probe.status() == 0
    assert 1.0e15 < rate < 3.5e15, rate
