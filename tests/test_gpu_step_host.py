"""fa_step_host: a forward + backward step from pinned host buffers.

The host-buffer step must give what fa_fwd + fa_bwd give on device copies of the same
inputs (O, L, dK, dV bitwise; dQ adds across CTAs in any order, so within the parity
tolerance), and two steps in flight on two streams with separate device buffers must
both land intact.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300 import inputs as I
from tiled_attention_11_gb300.build import build

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib_ready():
    assert torch.cuda.is_available(), "GPU tests need a CUDA device"
    build()
    _lib.lib()
    _lib.fa_device_status(reset=True)
    yield
    rc, site = _lib.fa_device_status()
    assert rc == _lib.FA_OK, f"device status word set: {rc} at wait site {site}"


def host_outputs(p):
    mk = lambda shape, dt: torch.full(shape, float("nan"), dtype=dt).pin_memory()  # noqa: E731
    return [mk((p.B, p.H, p.Nq, p.D), torch.bfloat16), mk((p.B, p.H, p.Nq), torch.float32),
            mk((p.B, p.H, p.Nq, p.D), torch.bfloat16), mk((p.B, p.H, p.Nk, p.D), torch.bfloat16),
            mk((p.B, p.H, p.Nk, p.D), torch.bfloat16)]


@pytest.mark.parametrize("p", [I.Problem(2, 2, 300, 300, 64, True), I.Problem(1, 3, 129, 77, 128, False)],
                         ids=lambda p: p.name())
def test_step_host_matches_device_calls(p):
    q, k, v, do = I.draw(p, 4)
    pin = [t.pin_memory() for t in (q, k, v, do)]
    outs = host_outputs(p)
    buf = torch.empty(_lib.step_host_device_bytes(p.B, p.H, p.Nq, p.Nk, p.D), dtype=torch.uint8, device="cuda")
    _lib.step_host(*pin, *outs, buf, p.causal, p.scale)
    torch.cuda.synchronize()
    qg, kg, vg, dog = (t.cuda() for t in (q, k, v, do))
    o, lse = _lib.forward(qg, kg, vg, p.causal, p.scale)
    dq, dk, dv = _lib.backward(qg, kg, vg, o, lse, dog, p.causal, p.scale)
    torch.cuda.synchronize()
    assert torch.equal(outs[0], o.cpu()) and torch.equal(outs[1], lse.cpu())
    assert torch.equal(outs[3], dk.cpu()) and torch.equal(outs[4], dv.cpu())
    ref = dq.double().cpu().numpy()
    got = outs[2].double().numpy()
    assert np.linalg.norm(got - ref) / np.linalg.norm(ref) < 1e-2


def test_two_steps_in_flight():
    p = I.Problem(1, 4, 1024, 1024, 128, True)
    q, k, v, do = I.draw(p, 5)
    pin = [t.pin_memory() for t in (q, k, v, do)]
    n = _lib.step_host_device_bytes(p.B, p.H, p.Nq, p.Nk, p.D)
    lanes = [(torch.cuda.Stream(), torch.empty(n, dtype=torch.uint8, device="cuda"), host_outputs(p)) for _ in range(2)]
    for i in range(6):
        st, buf, outs = lanes[i % 2]
        _lib.step_host(*pin, *outs, buf, p.causal, p.scale, stream=st)
    torch.cuda.synchronize()
    qd, kd, vd = (I.as_f64(t) for t in (q, k, v))
    ro, rl = oracle.attention_forward(qd, kd, vd, p.scale, True)
    for _, _, outs in lanes:
        o = outs[0].double().numpy()
        assert np.linalg.norm(o - ro) / np.linalg.norm(ro) < 1e-2
        assert np.abs(outs[1].double().numpy() - rl).max() < 1e-3
    assert torch.equal(lanes[0][2][3], lanes[1][2][3])  # dK deterministic across lanes


def test_step_host_rejects_device_tensors_and_short_buffer():
    p = I.Problem(1, 1, 64, 64, 64, False)
    q, k, v, do = I.draw(p, 6)
    outs = host_outputs(p)
    buf = torch.empty(_lib.step_host_device_bytes(1, 1, 64, 64, 64), dtype=torch.uint8, device="cuda")
    with pytest.raises(ValueError):
        _lib.step_host(q.cuda(), k, v, do, *outs, buf, False)
    with pytest.raises(RuntimeError):
        _lib.step_host(q, k, v, do, *outs, buf[:1024], False)
