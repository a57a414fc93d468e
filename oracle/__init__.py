"""CPU fp64 oracle of the MoE layer (test infrastructure only).

Only tests/, __graft_entry__.smoke() and bench.py's CPU-baseline / reference legs may
import this package. The CUDA library and its binding never use it.
"""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import AUX_LOSS_WEIGHT  # noqa: F401
