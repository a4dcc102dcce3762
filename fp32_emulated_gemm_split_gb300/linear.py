"""EmuLinear: a drop-in replacement for torch.nn.Linear whose matrix
products run through libemusgemm.

The blog post ("Unlocking Tensor Core Performance for Machine Learning
Interatomic Potentials", section on TF32x3 on Ampere GPUs) swaps a model's
nn.Linear layers for a custom layer that keeps the trained weights, bias and
input shapes, takes and returns FP32, and runs the products with the
emulated FP32 GEMM; because the model's forces are derivatives of its energy,
the gradient with respect to the layer input goes through the same GEMM.
This module does that for both emulations:

  forward          y  = x W^T + b      emu_sgemm(x, W, transB=1)
  input gradient   dx = dy W           emu_sgemm(dy, W)
  weight gradient  dW = dy^T x         emu_sgemm(dy, x, transA=1)
  bias gradient    db = sum of dy over the leading dimensions

Inputs of any leading shape (..., in_features) are flattened to 2-D.
"""
from __future__ import annotations

import torch

from . import emu_sgemm


class _EmuLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, mode):
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1])
        if x2.stride(-1) != 1:
            x2 = x2.contiguous()
        out = torch.empty((x2.shape[0], weight.shape[0]), dtype=torch.float32, device=x.device)
        if x2.shape[0] > 0:
            if bias is not None:
                out.copy_(bias.expand_as(out))
                emu_sgemm(x2, weight, out, transB=True, beta=1.0, mode=mode)
            else:
                emu_sgemm(x2, weight, out, transB=True, mode=mode)
        ctx.save_for_backward(x2, weight)
        ctx.mode = mode
        ctx.has_bias = bias is not None
        ctx.lead = lead
        return out.reshape(*lead, weight.shape[0])

    @staticmethod
    def backward(ctx, grad_out):
        x2, weight = ctx.saved_tensors
        g2 = grad_out.reshape(-1, weight.shape[0])
        if g2.stride(-1) != 1:
            g2 = g2.contiguous()
        gx = gw = gb = None
        if ctx.needs_input_grad[0]:
            gx = torch.empty_like(x2)
            if g2.shape[0] > 0:
                emu_sgemm(g2, weight, gx, mode=ctx.mode)
            else:
                gx.zero_()
            gx = gx.reshape(*ctx.lead, weight.shape[1])
        if ctx.needs_input_grad[1]:
            gw = torch.empty_like(weight)
            if g2.shape[0] > 0:
                emu_sgemm(g2, x2, gw, transA=True, mode=ctx.mode)
            else:
                gw.zero_()
        if ctx.has_bias and ctx.needs_input_grad[2]:
            gb = g2.sum(dim=0)
        return gx, gw, gb, None


class EmuLinear(torch.nn.Module):
    """nn.Linear with its products computed by the emulated FP32 GEMM.

    ``mode`` is "bf16x9" (default), "tf32x3" or "fp32_simt".  Parameters are
    FP32 CUDA tensors; ``EmuLinear.from_linear(layer)`` reuses a trained
    layer's weight and bias (shared, not copied)."""

    def __init__(self, in_features, out_features, bias=True, device=None, mode="bf16x9"):
        super().__init__()
        ref = torch.nn.Linear(in_features, out_features, bias=bias, device=device,
                              dtype=torch.float32)
        self.weight = ref.weight
        self.bias = ref.bias
        self.in_features = in_features
        self.out_features = out_features
        self.mode = mode

    @classmethod
    def from_linear(cls, layer: torch.nn.Linear, mode="bf16x9") -> "EmuLinear":
        m = cls.__new__(cls)
        torch.nn.Module.__init__(m)
        m.weight = layer.weight
        m.bias = layer.bias
        m.in_features = layer.in_features
        m.out_features = layer.out_features
        m.mode = mode
        return m

    def forward(self, x):
        if x.dtype != torch.float32:
            raise TypeError("EmuLinear computes FP32 in and out")
        return _EmuLinearFn.apply(x, self.weight, self.bias, self.mode)

    def extra_repr(self):
        return (f"in_features={self.in_features}, out_features={self.out_features}, "
                f"bias={self.bias is not None}, mode={self.mode}")


def swap_linear_layers(module: torch.nn.Module, mode="bf16x9") -> torch.nn.Module:
    """Replace every torch.nn.Linear inside `module` (in place) by an
    EmuLinear that shares its parameters; returns the module."""
    for name, child in list(module.named_children()):
        if isinstance(child, torch.nn.Linear):
            setattr(module, name, EmuLinear.from_linear(child, mode))
        else:
            swap_linear_layers(child, mode)
    return module
