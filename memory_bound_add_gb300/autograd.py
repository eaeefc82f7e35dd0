"""Training use of the fused residual-Add + LayerNorm.

``AddLayerNormFunction`` is a ``torch.autograd.Function`` whose forward is
``add_layernorm_fwd`` and whose backward is ``add_layernorm_bwd``. The forward
keeps A = X + R (rounded to the dtype) and each row's mean and rstd. The
backward turns dY into dX = dR, dgamma and dbeta. Both directions run in the
library's kernels; this module only holds the tensors the backward needs
between the two calls.

X and R are ``[..., H]`` CUDA tensors of one dtype (fp32, fp16 or bf16). gamma
and beta are fp32 ``[H]``.
"""
from __future__ import annotations

import torch

from . import binding


class AddLayerNormFunction(torch.autograd.Function):
    """y = LayerNorm(x + r) * gamma + beta over the last dimension, with the
    textbook derivative: per row, xhat = (A - mean) rstd and g = dY gamma give
    dA = rstd (g - mean(g) - xhat mean(g xhat)), which is both dX and dR;
    dgamma = sum over rows of dY xhat, dbeta = sum over rows of dY."""

    @staticmethod
    def forward(ctx, x, r, gamma, beta, eps):
        x, r = x.contiguous(), r.contiguous()
        y, a, mean, rstd = binding.add_layernorm(x, r, gamma.contiguous(), beta.contiguous(),
                                                 eps=float(eps), want_resid=True, want_stats=True)
        ctx.save_for_backward(a, mean, rstd, gamma)
        return y

    @staticmethod
    def backward(ctx, dy):
        a, mean, rstd, gamma = ctx.saved_tensors
        need_x, need_r, need_g, need_b = ctx.needs_input_grad[:4]
        dy = dy.contiguous()
        if need_g or need_b:
            dx, dg, db = binding.add_layernorm_backward(dy, a, mean, rstd, gamma.contiguous())
        else:
            dx = torch.empty_like(dy)
            binding.add_layernorm_bwd(dy, a, mean, rstd, gamma.contiguous(), dx)
            dg = db = None
        # dX and dR are the same values: one tensor serves both inputs
        return (dx if need_x else None, dx if need_r else None, dg if need_g else None,
                db if need_b else None, None)


def add_layernorm_train(x, r, gamma, beta, eps: float = 1e-5):
    """The fused Add + LayerNorm with gradients for x, r, gamma and beta."""
    return AddLayerNormFunction.apply(x, r, gamma, beta, eps)


class FusedAddLayerNorm(torch.nn.Module):
    """LayerNorm(x + r) over the last dimension as one module: learnable fp32
    gamma (ones) and beta (zeros) of size H, forward and backward in the
    library's kernels."""

    def __init__(self, hidden: int, eps: float = 1e-5, device=None):
        super().__init__()
        self.eps = float(eps)
        self.weight = torch.nn.Parameter(torch.ones(hidden, dtype=torch.float32, device=device))
        self.bias = torch.nn.Parameter(torch.zeros(hidden, dtype=torch.float32, device=device))

    def forward(self, x, r):
        return AddLayerNormFunction.apply(x, r, self.weight, self.bias, self.eps)
