"""GB300-native online low-rank KV-cache correction (KVCMAS hot path).

``agent_shared_context_gb300.kvc`` is the ctypes binding of the C-ABI library
``libkvc.so`` (built in-tree by ``__graft_entry__.build()``);
``agent_shared_context_gb300.synth`` builds seeded synthetic workloads.
"""
__version__ = "0.1.0"
