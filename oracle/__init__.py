"""CPU oracle (fp64, numpy) for the MoE layer: forward (moe_oracle) and backward
(moe_backward). Test infrastructure only: the product path never imports it."""
from .moe_oracle import *  # noqa: F401,F403
from .moe_oracle import GATE_MODES  # noqa: F401
from .moe_backward import (aux_loss_backward, backward, expert_choice_backward,  # noqa: F401
                           gate_backward, silu_grad, swiglu_ffn_backward, z_loss_backward)
