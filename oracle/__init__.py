"""fp64 CPU oracle for the KVCMAS online low-rank KV-cache correction.

TEST INFRASTRUCTURE.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline / reference leg of ``bench.py`` may import this package.  The
product (the CUDA library under ``agent_shared_context_gb300/csrc`` and its
Python binding) never imports it, and it imports nothing from the product; the
two share only the seeded input generator ``agent_shared_context_gb300.synth``,
which holds none of the method's arithmetic.
"""
from .kvc_oracle import *  # noqa: F401,F403
from .kvc_oracle import __all__  # noqa: F401
