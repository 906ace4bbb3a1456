"""CPU oracle for the MoE FFN layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import this package. The
product path (``sparse_expert_mlp_router_b300``) never imports, calls or
links it, and it shares no code with the CUDA kernels.
"""
from .moe_oracle import *  # noqa: F401,F403
