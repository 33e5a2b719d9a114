"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Some callers cannot call cudaMalloc or hand the library a workspace: a serving
process whose device memory budget is fixed at start-up, or a plug-in whose
host framework owns the allocator and passes only input and output buffers.
fa_bwd_noalloc serves them with a fixed 32 MiB scratch array inside the
library.  These tests call it through the C ABI and check it against the fp64
oracle and against the workspace entry point fa_bwd, within the parity
tolerances used by every GPU test here, on consecutive calls that reuse the
shared scratch, up to a problem that fills it.

This file is collected last on purpose, and passes both alone in a fresh
process and after the rest of the GPU suite.
"""
import ctypes

import numpy as np

import oracle
import pytest
import torch

from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300 import inputs as I
from tiled_attention_11_gb300.build import build

pytestmark = pytest.mark.gpu

REL_L2 = 1e-2
MAX_FRAC = 2e-2


def close(name, got, ref):
    g = got.to("cpu", torch.float64).numpy()
    r = ref.to("cpu", torch.float64).numpy()
    rl2 = np.linalg.norm(g - r) / max(np.linalg.norm(r), 1e-30)
    ma = np.abs(g - r).max()
    assert np.isfinite(g).all(), f"{name}: non-finite"
    assert rl2 <= REL_L2 and ma <= MAX_FRAC * np.abs(r).max(), f"{name}: rel_l2={rl2:.3e} max_abs={ma:.3e}"


def test_noalloc_backward_matches_oracle_and_workspace_backward_on_consecutive_calls():
    assert torch.cuda.is_available(), "needs a CUDA device"
    build()
    _lib.lib()
    dev = torch.device("cuda")
    # consecutive calls of different sizes share the scratch; the third repeats the first
    # after a smaller problem has overwritten part of it, the last fills the array
    # (1008 heads of 64 queries at D = 128: 33546240 of its 33554432 bytes)
    problems = [(I.Problem(2, 3, 300, 257, 64, True), 0), (I.Problem(1, 2, 200, 200, 128, False), 1),
                (I.Problem(2, 3, 300, 257, 64, True), 0), (I.Problem(1, 1008, 64, 64, 128, True), 2)]
    assert _lib.fa_bwd_workspace_size(1, 1008, 64, 64, 128) > 33_500_000
    for n, (p, seed) in enumerate(problems):
        qc, kc, vc, doc = I.draw(p, seed)
        q, k, v, do = (t.to(dev) for t in (qc, kc, vc, doc))
        o, lse = _lib.forward(q, k, v, p.causal, p.scale)
        dq_ref, dk_ref, dv_ref = _lib.backward(q, k, v, o, lse, do, p.causal, p.scale)
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
        _lib.fa_bwd_noalloc(q, k, v, o, lse, do, dq, dk, dv, p.causal, p.scale)
        torch.cuda.synchronize()
        tag = f"call {n} {p.name()}"
        close(tag + " dQ vs fa_bwd", dq, dq_ref)
        close(tag + " dK vs fa_bwd", dk, dk_ref)
        close(tag + " dV vs fa_bwd", dv, dv_ref)
        odq, odk, odv = oracle.attention_backward(*(I.as_f64(t) for t in (qc, kc, vc, doc)), p.scale, p.causal)
        for name, got, ref in (("dQ", dq, odq), ("dK", dk, odk), ("dV", dv, odv)):
            close(tag + f" {name} vs oracle", got, torch.from_numpy(ref))
    assert _lib.fa_device_status()[0] == _lib.FA_OK


def test_noalloc_rejects_problems_beyond_its_scratch():
    L = _lib.lib()
    vp = ctypes.c_void_p
    ptrs = [vp(0x10000000 * (i + 1)) for i in range(9)]
    # the multi-head layer needs ~270 MB of scratch: refused before any launch
    rc = L.fa_bwd_noalloc(*ptrs, 4, 32, 4096, 4096, 128, 0.088, 1, None)
    assert rc == _lib.FA_ERR_SCRATCH_LIMIT
    assert "32 MiB" in _lib.strerror(rc)
