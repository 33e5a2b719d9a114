"""CPU oracle for tiled attention — TEST INFRASTRUCTURE, not part of the product.

Only ``tests/``, ``__graft_entry__.smoke()`` and ``bench.py`` (its
``cpu_baseline`` leg and ``--impl reference`` arm) may import anything here.
The CUDA library and its Python binding never do, and this package never
imports them.  Everything is float64 numpy.

Modules:
  * ``attn_ref``  — the plain definition (materialised S, stable softmax,
    explicit softmax-Jacobian backward); the oracle proper.
  * ``tiled_ref`` — the pages' tile-by-tile online-softmax forward restated in
    fp64, used only to pin the online-update algebra.

Pins: every function is checked in ``tests/test_oracle_pins.py`` against
closed forms, brute-force scalar loops, PyTorch's fp64 CPU
``scaled_dot_product_attention`` and autograd (a library routine for the same
definition), central finite differences and gradient invariants.
"""
from .attn_ref import attention_forward, attention_backward, attention_varlen, backward_head, forward_head  # noqa: F401
from .tiled_ref import tiled_forward_head  # noqa: F401
