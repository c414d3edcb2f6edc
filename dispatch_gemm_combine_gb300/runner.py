"""Buffer management around the C ABI for one problem shape.

`LayerRunner` allocates (through PyTorch) the plan arrays, workspaces, the
saved context and the outputs for a fixed shape once, then runs
moe_plan / moe_ffn_fwd / moe_ffn_bwd on them.  All arithmetic happens in the
library's kernels.
"""

import torch

from . import (MOE_BF16, MOE_FP32, Shape, alloc_plan, bias_struct, check_device_error, ffn_bwd,
               ffn_fwd, moe_saved_size, plan, route, workspace)

_TORCH_DTYPE = {MOE_BF16: torch.bfloat16, MOE_FP32: torch.float32}


class LayerRunner:
    def __init__(self, T, H, I, E, k, act, dtype=MOE_BF16, clamp_limit=7.0, alpha=1.702,
                 device="cuda", training=True, backward=True, gate_up_layout=0, out_fp32=False):
        """out_fp32: y and dx in fp32 instead of the storage dtype."""
        self.shape = Shape(T, H, I, E, k, act, dtype, clamp_limit, alpha, gate_up_layout, out_fp32)
        self.device = device
        self.tdtype = _TORCH_DTYPE[dtype]
        odt = torch.float32 if out_fp32 else self.tdtype
        self.plan_t, self.plan_s = alloc_plan(self.shape, device)
        self.ws_plan = workspace(self.shape, 0, device)
        self.ws_fwd = workspace(self.shape, 1, device)
        self.ws_bwd = workspace(self.shape, 2, device) if backward else None
        self.saved = (torch.empty(moe_saved_size(self.shape), dtype=torch.uint8, device=device)
                      if training else None)
        self.y = torch.empty((T, H), dtype=odt, device=device)
        if backward:
            self.dx = torch.empty((T, H), dtype=odt, device=device)
            self.d_topk_w = torch.empty((T, k), dtype=torch.float32, device=device)
            self.dw_gate_up = torch.empty((E, H, 2 * I), dtype=torch.float32, device=device)
            self.dw_down = torch.empty((E, I, H), dtype=torch.float32, device=device)

    def plan(self, topk_idx, stream=None):
        plan(self.shape, topk_idx, self.plan_s, self.ws_plan, stream)

    def route(self, logits, topk_idx, topk_w, stream=None):
        """Fill topk_idx [T,k] int32 and topk_w [T,k] fp32 from fp32 logits
        [T,E] and build the plan of the chosen ids."""
        route(self.shape, logits, topk_idx, topk_w, self.plan_s, self.ws_plan, stream)

    def forward(self, x, topk_idx, topk_w, w_gate_up, w_down, use_plan=True, stream=None,
                b_gate_up=None, b_down=None, inference=False):
        """y = layer(x).  With use_plan the plan must have been built by plan();
        otherwise the forward builds its own inside the workspace.  b_gate_up
        [E,2I] / b_down [E,H] (storage dtype) are the optional per-expert biases.
        inference=True saves no context for the backward (as a runner built
        with training=False)."""
        ffn_fwd(self.shape, x, topk_idx, topk_w, w_gate_up, w_down, self.y, self.ws_fwd,
                self.plan_s if use_plan else None, None if inference else self.saved, stream,
                bias_struct(b_gate_up, b_down))
        return self.y

    def backward(self, dy, x, topk_idx, topk_w, w_gate_up, w_down, stream=None, recompute=False,
                 b_gate_up=None, b_down=None):
        """Gradients of <dy, y>: (dx, d_topk_w, dw_gate_up, dw_down), and with
        biases also (db_gate_up, db_down).  The biases must be those given to
        the forward.  With recompute the saved context is not used: the
        backward recomputes it in a larger workspace (allocated on first use)."""
        with_bias = b_gate_up is not None or b_down is not None
        bias = None
        if with_bias:
            if getattr(self, "db_gate_up", None) is None:
                E, H, I = self.shape.E, self.shape.H, self.shape.I
                self.db_gate_up = torch.empty((E, 2 * I), dtype=torch.float32, device=self.device)
                self.db_down = torch.empty((E, H), dtype=torch.float32, device=self.device)
            bias = bias_struct(b_gate_up, b_down, self.db_gate_up, self.db_down)
        if recompute:
            if getattr(self, "ws_bwd_recompute", None) is None:
                self.ws_bwd_recompute = workspace(self.shape, 3, self.device)
            ws, saved = self.ws_bwd_recompute, None
        else:
            ws, saved = self.ws_bwd, self.saved
        ffn_bwd(self.shape, dy, x, topk_idx, topk_w, w_gate_up, w_down, self.plan_s, saved,
                self.dx, self.d_topk_w, self.dw_gate_up, self.dw_down, ws, stream, bias)
        out = (self.dx, self.d_topk_w, self.dw_gate_up, self.dw_down)
        return out + (self.db_gate_up, self.db_down) if with_bias else out

    def check(self, stream=None):
        for ws in (self.ws_plan, self.ws_fwd, self.ws_bwd, getattr(self, "ws_bwd_recompute", None)):
            if ws is not None:
                check_device_error(ws, stream)
