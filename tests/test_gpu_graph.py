"""CUDA Graph capture of one forward + backward step (C fa_graph_create/launch/destroy).

The graph replays the same four kernels as the direct calls, so O, L, dK and dV must be
bitwise identical to fa_fwd/fa_bwd on the same inputs; dQ (fp32 reduction order) within
the parity tolerance.  A replay reads the buffers' current contents.
"""
import numpy as np
import pytest
import torch

import oracle
from tiled_attention_11_gb300 import _lib
from tiled_attention_11_gb300 import inputs as I
from tiled_attention_11_gb300.build import build

pytestmark = pytest.mark.gpu


def _close(name, got, ref):
    g = got.to("cpu", torch.float64).numpy()
    r = np.asarray(ref, np.float64)
    rl2 = np.linalg.norm(g - r) / np.linalg.norm(r)
    assert rl2 <= 1e-2 and np.abs(g - r).max() <= 2e-2 * np.abs(r).max(), f"{name}: rel_l2={rl2:.3e}"


@pytest.mark.parametrize("p", [I.SMALL, I.Problem(2, 3, 300, 257, 128, True)], ids=lambda p: p.name())
def test_graph_step_matches_direct_calls(p):
    build()
    dev = torch.device("cuda")
    q, k, v, do = (t.to(dev) for t in I.draw(p, 0))
    o, lse = _lib.forward(q, k, v, p.causal, p.scale)
    dq, dk, dv = _lib.backward(q, k, v, o, lse, do, p.causal, p.scale)
    go, glse = torch.empty_like(o), torch.empty_like(lse)
    gdq, gdk, gdv = torch.empty_like(dq), torch.empty_like(dk), torch.empty_like(dv)
    g = _lib.StepGraph(q, k, v, go, glse, do, gdq, gdk, gdv, p.causal, p.scale)
    for _ in range(3):
        go.zero_(); gdk.zero_()
        g.launch()
        torch.cuda.synchronize()
        assert torch.equal(go, o) and torch.equal(glse, lse)
        assert torch.equal(gdk, dk) and torch.equal(gdv, dv)
        _close("graph dQ", gdq, dq.double().cpu().numpy())
    # new contents in the same buffers: the replay computes on them
    q2, k2, v2, do2 = I.draw(p, 7)
    for dst, src in zip((q, k, v, do), (q2, k2, v2, do2)):
        dst.copy_(src)
    g.launch()
    torch.cuda.synchronize()
    qd, kd, vd, dod = (I.as_f64(t) for t in (q2, k2, v2, do2))
    ro, rl = oracle.attention_forward(qd, kd, vd, p.scale, p.causal)
    rdq, rdk, rdv = oracle.attention_backward(qd, kd, vd, dod, p.scale, p.causal)
    _close("graph O", go, ro)
    assert np.abs(glse.double().cpu().numpy() - rl).max() <= 1e-3
    _close("graph dQ", gdq, rdq)
    _close("graph dK", gdk, rdk)
    _close("graph dV", gdv, rdv)
    g.close()


def test_graph_create_rejects_bad_arguments():
    build()
    q = torch.zeros(1, 1, 64, 48, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(_lib.FAError) as e:
        _lib.StepGraph(q, q.clone(), q.clone(), torch.empty_like(q), torch.empty(1, 1, 64, device="cuda"),
                       q.clone(), torch.empty_like(q), torch.empty_like(q), torch.empty_like(q), True)
    assert e.value.code == _lib.FA_ERR_UNSUPPORTED_D
