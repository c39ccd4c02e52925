"""CPU oracle of the MoE expert layer (test infrastructure; see moe_oracle)."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import Permutation  # noqa: F401
