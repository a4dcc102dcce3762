"""EmuLinear: a drop-in replacement for torch.nn.Linear whose matrix
products run through libemusgemm.

The blog post ("Unlocking Tensor Core Performance for Machine Learning
Interatomic Potentials", section on TF32x3 on Ampere GPUs) swaps a model's
nn.Linear layers for a custom layer that keeps the trained weights, bias and
input shapes, takes and returns FP32, and runs the products with the
emulated FP32 GEMM; because the model's forces are derivatives of its energy,
the gradient with respect to the layer input goes through the same GEMM.
This module does that for both emulations:

  forward          y  = x W^T + b      emu_sgemm_bsplit(x, pieces of W)
  input gradient   dx = dy W           emu_sgemm_bsplit(dy, pieces of W^T)
  weight gradient  dW = dy^T x         emu_sgemm(dy, x, transA=1)
  bias gradient    db = sum of dy over the leading dimensions

Inputs of any leading shape (..., in_features) are flattened to 2-D.

The weight is the same for every batch until an optimiser changes it, so
the layer splits it once per version of the weight (two piece sets: W for
the forward product, W^T for the input gradient) and the forward and
input-gradient products run emu_sgemm_bsplit on those pieces: no split of
the weight per call, and in BF16x9 with 4096 rows or more and at most 256
output columns a single kernel launch per product.  The pieces are dropped
and made again whenever the weight's storage or version changes (an
in-place update bumps the version).
"""
from __future__ import annotations

import torch

from . import emu_sgemm, emu_sgemm_bsplit, emu_split_b


class _WeightPieces:
    """The split pieces of one weight, for the forward product (op(B) = W^T)
    and the input gradient (op(B) = W), made on first use and remade when
    the weight changes."""

    def __init__(self):
        self._cache = {}

    def get(self, weight, transB, mode):
        key = (bool(transB), mode)
        stamp = (weight.data_ptr(), weight._version, tuple(weight.shape), weight.device)
        hit = self._cache.get(key)
        if hit is None or hit[0] != stamp:
            hit = (stamp, emu_split_b(weight.detach(), transB=transB, mode=mode))
            self._cache[key] = hit
        return hit[1]

    def clear(self):
        self._cache.clear()


def _product(a, weight, out, transB, beta, mode, pieces):
    """out = a op(W) + beta out, with W's pieces from the cache when the mode
    runs on the tensor cores."""
    if pieces is not None and mode != "fp32_simt":
        emu_sgemm_bsplit(a, pieces.get(weight, transB, mode), out, beta=beta, mode=mode)
    else:
        emu_sgemm(a, weight, out, transB=transB, beta=beta, mode=mode)


class _EmuLinearFn(torch.autograd.Function):
    @staticmethod
    def forward(ctx, x, weight, bias, mode, pieces):
        lead = x.shape[:-1]
        x2 = x.reshape(-1, x.shape[-1])
        if x2.stride(-1) != 1:
            x2 = x2.contiguous()
        out = torch.empty((x2.shape[0], weight.shape[0]), dtype=torch.float32, device=x.device)
        if x2.shape[0] > 0:
            if bias is not None:
                out.copy_(bias.expand_as(out))
                _product(x2, weight, out, True, 1.0, mode, pieces)
            else:
                _product(x2, weight, out, True, 0.0, mode, pieces)
        ctx.save_for_backward(x2, weight)
        ctx.mode = mode
        ctx.pieces = pieces
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
                _product(g2, weight, gx, False, 0.0, ctx.mode, ctx.pieces)
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
        return gx, gw, gb, None, None


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
        self._pieces = _WeightPieces()

    @classmethod
    def from_linear(cls, layer: torch.nn.Linear, mode="bf16x9") -> "EmuLinear":
        m = cls.__new__(cls)
        torch.nn.Module.__init__(m)
        m.weight = layer.weight
        m.bias = layer.bias
        m.in_features = layer.in_features
        m.out_features = layer.out_features
        m.mode = mode
        m._pieces = _WeightPieces()
        return m

    def forward(self, x):
        if x.dtype != torch.float32:
            raise TypeError("EmuLinear computes FP32 in and out")
        return _EmuLinearFn.apply(x, self.weight, self.bias, self.mode, self._pieces)

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
