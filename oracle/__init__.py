"""fp64 CPU oracle of the Mixtral sparse-MoE layer (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline legs use it;
the CUDA library never imports it.
"""
from .moe_oracle import *  # noqa: F401,F403
