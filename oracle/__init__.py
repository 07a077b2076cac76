"""fp64 CPU oracle for exact attention — test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline /
reference leg may import this package. The CUDA path never imports it and it
imports nothing from the CUDA path. Parity of every function here is pinned by
the ``-m "not gpu"`` tests (closed forms, invariants, brute force, finite
differences, a library special case and hand-derived golden values).
"""
from .attention_fp64 import (attend_head, attend_head_backward, backward, forward)  # noqa: F401
from .online_softmax import online_attend_head  # noqa: F401
from .exp2_method import exp2_exact, exp2_range_reduced, fit_exp2_poly  # noqa: F401
from . import fp8_e4m3  # noqa: F401
