"""MXFP4 linear layer for PyTorch autograd.

"Pretraining Large Language Models with MXFP4 on Native FP4 Hardware" (C.1-C.3) runs
the three GEMMs of a linear layer in MXFP4 behind the framework's ordinary linear
module.  This module does the same for PyTorch: the forward pass is
``mxfp4_linear_fprop`` (Y = X W^T, bf16 out), which also saves X^T and W^T quantised
along the tokens and the output features; the backward pass is ``mxfp4_linear_backward``
(dY quantised once; dX = dY W, bf16 out, and dW = dY^T X, fp32 out, in one grouped
GEMM launch).  Every step runs in the CUDA library; this file only wires the
calls into autograd.  The quantised copies live on the autograd context between the
two passes: about 0.53 bytes per element of X and W.
"""
from __future__ import annotations

import torch

from . import binding as mx


class MXFP4LinearFunction(torch.autograd.Function):
    """y = x @ w.T with x [..., K] and w [N, K] bf16 CUDA tensors (unit inner stride)."""

    @staticmethod
    def forward(ctx, x: torch.Tensor, w: torch.Tensor, had: int, mode: int) -> torch.Tensor:
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1]).contiguous()
        cfg = mx.Config(had=had, mode=mode, out_dtype=mx.OUT_BF16)
        y, xT, wT = mx.linear_fprop(x2, w.contiguous(), cfg)
        ctx.xT, ctx.wT, ctx.had, ctx.mode, ctx.lead = xT, wT, had, mode, lead
        return y.reshape(*lead, w.shape[0])

    @staticmethod
    def backward(ctx, dy: torch.Tensor):
        dy2 = dy.reshape(-1, dy.shape[-1]).to(torch.bfloat16).contiguous()
        # one dY quantisation, then Dgrad (bf16 dX) and Wgrad (fp32 dW; autograd casts it
        # to the weight's dtype) in one grouped launch
        dx, dw = mx.linear_backward(dy2, ctx.wT, ctx.xT, mx.Config(had=ctx.had, mode=ctx.mode, out_dtype=mx.OUT_BF16))
        ctx.xT = ctx.wT = None
        return dx.reshape(*ctx.lead, dx.shape[-1]), dw, None, None


def mxfp4_linear(x: torch.Tensor, w: torch.Tensor, had: int = mx.HAD_16, mode: int = mx.SCALE_FLOOR) -> torch.Tensor:
    """MXFP4 linear layer (no bias): Fprop, Dgrad and Wgrad each rotate their operands
    along the contraction (H16 by default) and quantise them to MXFP4.  The number of
    tokens (the product of x's leading dimensions) must be a multiple of 32, and so must
    K and N."""
    return MXFP4LinearFunction.apply(x, w, had, mode)
