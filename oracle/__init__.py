"""CPU oracle (fp64) for the MXFP8 SwiGLU MLP.

TEST INFRASTRUCTURE: only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg may import this package.  It shares no code with
the CUDA library (``mxfp8_swiglu_mlp_gb300``) and never imports it.

Parity pins: every function here is pinned by ``tests/test_oracle_*.py``
against library routines, closed forms, hand-worked examples under
``tests/golden/`` and brute force on tiny inputs.
"""
from .mx_oracle import *  # noqa: F401,F403
from . import mx_oracle  # noqa: F401
