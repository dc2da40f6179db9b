"""CPU oracle (fp64, numpy) for the MoE layer forward. Test infrastructure only: the
product path never imports it."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import GATE_MODES  # noqa: F401
