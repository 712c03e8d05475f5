"""CPU oracle for MoE dispatch / combine -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline leg of
``bench.py`` may import this package.  The product path (the C-ABI library
and its Python binding in ``combine_topk_idx_gb300``) never imports, links or
calls anything here, and this package imports nothing from it.
"""
from .ep_oracle import *  # noqa: F401,F403
