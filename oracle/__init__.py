"""fp64 CPU oracle of the MoE expert layer.  Test infrastructure only: the
product path never imports this package."""
from .moe_oracle import (ACT_SWIGLU, ACT_CLAMPED_GLU, CLAMP_LIMIT, CLAMP_ALPHA,
                         sigmoid, activation, activation_grad, dispatch_plan, route,
                         gate_up_concatenated, gate_up_in_layout,
                         moe_forward, moe_backward, forward_rows)
