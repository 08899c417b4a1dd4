"""Autograd forms of the two operations, for code that builds a loss and calls ``loss.backward()``.

* ``linear_cross_entropy(hidden, W, target, bias=None, ...)``: the fused LM-head loss of "Fused Linear
  Cross-Entropy: The Math, the Memory Wall, and Two Ways Around It" ("The setting"; the gradients of "From
  dlogits to grad_input and grad_W").  For the mean and sum reductions the forward call already computes
  every gradient (the fused forward + backward that the page is about) with an upstream gradient of 1;
  backward multiplies them in place by the incoming gradient, on the device (``flce_scale_gradient``),
  and hands them to autograd.  For reduction "none" the gradient depends on the per-token upstream
  gradients, so forward computes the per-token losses only and backward runs the fused call with them.
* ``cross_entropy(logits, labels, ...)``: the standalone row-wise CE of "Greyhound -- Cross-Entropy"
  ("Usage": the non-mutating functional form with normal autograd semantics).  Forward writes dlogits into
  a new tensor (the logits are left unchanged) and forms the reduced loss on the device
  (``ce_reduce_loss``); backward scales dlogits by the incoming gradient (and 1/max(n_valid, 1) for the
  mean) in place.

All arithmetic runs in libflce.so; these classes only move tensors between autograd and the C ABI.  The
saved gradients are scaled in place, so a graph built by these functions can be backpropagated once.
"""
from __future__ import annotations

import torch

from . import _lib


class _LinearCrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, hidden, W, target, bias, ignore_index, reduction, z_loss):
        need_gi = bool(ctx.needs_input_grad[0])
        need_gw = bool(ctx.needs_input_grad[1]) or (bias is not None and bool(ctx.needs_input_grad[3]))
        ctx.reduction = reduction
        if reduction == "none":
            out = _lib.flce_fwd_bwd(hidden, W, target, bias=bias, ignore_index=ignore_index, reduction="none",
                                    z_loss=z_loss, need_grad_input=False, need_grad_W=False)
            ctx.save_for_backward(hidden, W, target, bias)
            ctx.args = (ignore_index, z_loss, need_gi, need_gw)
            return out["loss_per_token"]
        out = _lib.flce_fwd_bwd(hidden, W, target, bias=bias, ignore_index=ignore_index, reduction=reduction,
                                z_loss=z_loss, need_grad_input=need_gi, need_grad_W=need_gw)
        ctx.grads = (out["grad_input"], out["grad_W"], out["grad_bias"])
        return out["loss"].reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        needs = ctx.needs_input_grad
        if ctx.reduction == "none":
            hidden, W, target, bias = ctx.saved_tensors
            ignore_index, z_loss, need_gi, need_gw = ctx.args
            out = _lib.flce_fwd_bwd(hidden, W, target, bias=bias, ignore_index=ignore_index, reduction="none",
                                    z_loss=z_loss, need_grad_input=need_gi, need_grad_W=need_gw,
                                    grad_loss_per_token=grad_out.float().contiguous())
            gi, gw, gb = out["grad_input"], out["grad_W"], out["grad_bias"]
        else:
            gi, gw, gb = ctx.grads
            ctx.grads = None
            upstream = grad_out.float().reshape(1).contiguous()
            for g in (gi, gw, gb):
                if g is not None:
                    _lib.scale_gradient_(g, upstream)
        return (gi if needs[0] else None, gw if needs[1] else None, None, gb if needs[3] else None, None, None,
                None)


def linear_cross_entropy(hidden, W, target, bias=None, ignore_index: int = -100, reduction: str = "mean",
                         z_loss: float = 0.0):
    """Cross-entropy of the logits hidden . W^T (+ bias) against ``target``, without the logits in memory.

    hidden [BT, H] bf16, W [V, H] bf16, target [BT] int64, bias [V] fp32 or None, all on the GPU.  Returns
    the reduced loss (a 0-dim fp32 tensor) for "mean" / "sum", the per-token losses [BT] for "none".
    Gradients (bf16 for hidden, fp32 for W and bias) reach autograd through ``backward``.
    """
    if reduction not in ("mean", "sum", "none"):
        raise ValueError("reduction must be 'mean', 'sum' or 'none'")
    return _LinearCrossEntropy.apply(hidden, W, target, bias, int(ignore_index), reduction, float(z_loss))


class _CrossEntropy(torch.autograd.Function):
    @staticmethod
    def forward(ctx, logits, labels, ignore_index, z_loss, reduction):
        r = _lib.cross_entropy(logits, labels, ignore_index=ignore_index, z_loss=z_loss,
                               want_grad=bool(ctx.needs_input_grad[0]))
        loss = _lib.ce_reduce_loss(r["ce_sum"], r["z_sum"], r["n_valid"], z_loss=z_loss, reduction=reduction)
        ctx.dlogits = r["dlogits"]
        ctx.n_valid = r["n_valid"] if reduction == "mean" else None
        return loss.reshape(())

    @staticmethod
    def backward(ctx, grad_out):
        dl = ctx.dlogits
        ctx.dlogits = None
        if dl is not None:
            _lib.scale_gradient_(dl, grad_out.float().reshape(1).contiguous(), ctx.n_valid)
        return dl, None, None, None, None


def cross_entropy(logits, labels, ignore_index: int = -100, z_loss: float = 0.0, reduction: str = "mean"):
    """Row-wise cross-entropy of ``logits`` [B, V] (bf16, fp16 or fp32, on the GPU) against ``labels`` [B]
    int64: (ce_sum + z_loss z_sum) / max(n_valid, 1) for "mean", the plain sum for "sum", as a 0-dim fp32
    tensor.  The logits are not modified; their gradient (same dtype) reaches autograd through backward."""
    if reduction not in ("mean", "sum"):
        raise ValueError("reduction must be 'mean' or 'sum'")
    return _CrossEntropy.apply(logits, labels, int(ignore_index), float(z_loss), reduction)
