"""CPU oracle of the routed-MoE hot path (test infrastructure only; see rlmoe_oracle)."""
from .rlmoe_oracle import *  # noqa: F401,F403
from .rlmoe_oracle import NO_EARLY_OUT, BLOCK_BYTES, BLOCK_VALUES  # noqa: F401
