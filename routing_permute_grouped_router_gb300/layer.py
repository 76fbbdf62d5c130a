"""A mixture-of-experts layer held on one GPU, driven through the C ABI.

``MoELayer`` owns the device copies of the weights, the saved routing state,
the float32 gradient buffers and the workspace (allocated with torch), and
calls ``moe_layer_fwd`` / ``moe_layer_bwd``.  It does no arithmetic itself.
"""
from __future__ import annotations

from typing import Optional

import torch

from . import (MOE_BF16, MoeConfig, allocate_grads, allocate_saved, moe_layer_bwd, moe_layer_fwd, moe_max_rows,
               workspace)


class MoELayer:
    def __init__(self, cfg: MoeConfig, W_r: torch.Tensor, bias: Optional[torch.Tensor], W1: torch.Tensor,
                 W3: torch.Tensor, W2: torch.Tensor, training: bool = True, recompute: bool = False):
        self.cfg = cfg
        self.device = W1.device
        self.act_dtype = torch.bfloat16 if cfg.dtype == MOE_BF16 else torch.float32
        self.weights = dict(W_r=W_r.contiguous(), bias=None if bias is None else bias.contiguous(),
                            W1=W1.contiguous(), W3=W3.contiguous(), W2=W2.contiguous())
        self.training = training
        self.max_rows = moe_max_rows(cfg)
        self.recompute = training and recompute  # keep no a, b, h: the backward recomputes them
        self.saved = allocate_saved(cfg, self.device, self.recompute) if training else None
        self.grads = allocate_grads(cfg, self.device) if training else None
        self.ws = workspace(cfg, (2 if self.recompute else 1) if training else 0, self.device)
        T, d = max(cfg.T, 1), cfg.d_model
        self.y = torch.empty(T, d, dtype=self.act_dtype, device=self.device)
        self.dx = torch.empty(T, d, dtype=self.act_dtype, device=self.device) if training else None

    def forward(self, x: torch.Tensor, stream=None) -> torch.Tensor:
        moe_layer_fwd(self.cfg, self.weights, x, self.y, self.saved, self.ws, stream)
        return self.y

    def backward(self, x: torch.Tensor, dy: torch.Tensor, accumulate: bool, stream=None) -> torch.Tensor:
        if not self.training:
            raise RuntimeError("layer was built without training buffers")
        moe_layer_bwd(self.cfg, self.weights, x, dy, self.saved, self.dx, self.grads, int(accumulate), self.ws,
                      stream)
        return self.dx


def from_workload(wl, device="cuda", training: bool = True, T: Optional[int] = None,
                  aux_loss_coeff: float = 0.0, recompute: bool = False) -> MoELayer:
    """Upload a ``workload.Workload``'s weights and build the layer."""
    from . import config_of

    cfg = config_of(wl.shape, T, aux_loss_coeff)
    bias = None if wl.bias is None else torch.from_numpy(wl.bias).to(device)
    return MoELayer(cfg, torch.from_numpy(wl.W_r).to(device), bias, wl.W1.torch(device), wl.W3.torch(device),
                    wl.W2.torch(device), training=training, recompute=recompute)
