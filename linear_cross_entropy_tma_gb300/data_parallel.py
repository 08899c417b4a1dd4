"""Data parallelism over tokens for fused linear cross-entropy.

The loss and every gradient of the method are sums over tokens ("Fused Linear Cross-Entropy", "The
setting" and "From dlogits to grad_input and grad_W"): with s = 1/max(n_valid, 1) for the mean,

    loss        = s * sum_t l_t
    grad_input  = s * dS_sum . W          (row t depends on token t only)
    grad_W      = s * dS_sum^T . hidden   (a sum over tokens)
    grad_bias   = s * column sums of dS_sum

where dS_sum is dlogits of the sum reduction.  So each rank runs the single-GPU path with
reduction="sum" on its own shard of tokens; the ranks then all-reduce the loss sum, the valid count
and grad_W / grad_bias, and each rank scales its results by 1/max(n_valid, 1) with the GLOBAL count.
grad_input stays on the rank that owns the tokens.  This reproduces the single-GPU mean exactly up to
rounding; for a bf16 grad_input the scaling is one extra rounding of the stored value (relative error
at most 2^-8 per element on top of the kernel's own rounding).

The exchange is the only collective of the path; it runs through torch.distributed (NCCL on GPUs,
gloo on CPU).
"""
from __future__ import annotations


def compose_token_shards(loss, n_valid, grad_input=None, grad_W=None, grad_bias=None, reduction: str = "mean",
                         group=None) -> None:
    """Turns one rank's sum-reduced shard results into the global result, in place.

    loss: 1-element tensor holding this shard's loss sum; n_valid: 1-element int64 tensor with this
    shard's valid count; grad_input / grad_W / grad_bias: this shard's sum-reduced gradients (any of
    them None when not computed).  After the call every rank holds the global loss, the global
    n_valid, the global grad_W / grad_bias, and its own rows of the global grad_input.  No host
    synchronisation: the mean scale stays on the device.
    """
    import torch
    import torch.distributed as dist

    if reduction not in ("mean", "sum"):
        raise ValueError("reduction must be 'mean' or 'sum'")
    dist.all_reduce(n_valid, op=dist.ReduceOp.SUM, group=group)
    dist.all_reduce(loss, op=dist.ReduceOp.SUM, group=group)
    if grad_W is not None:
        dist.all_reduce(grad_W, op=dist.ReduceOp.SUM, group=group)
    if grad_bias is not None:
        dist.all_reduce(grad_bias, op=dist.ReduceOp.SUM, group=group)
    if reduction == "sum":
        return
    scale = 1.0 / n_valid.clamp(min=1).to(torch.float64)
    for t in (loss, grad_input, grad_W, grad_bias):
        if t is None:
            continue
        if t.dtype in (torch.float32, torch.float64):
            t.mul_(scale.to(t.dtype))
        else:
            # one rounding of the product, computed in fp32
            t.copy_(t.to(torch.float32) * scale.to(torch.float32))


def flce_fwd_bwd_data_parallel(hidden, W, target, bias=None, ignore_index: int = -100, reduction: str = "mean",
                               z_loss: float = 0.0, group=None, **kwargs) -> dict:
    """flce_fwd_bwd on this rank's token shard, composed across the ranks of `group`.

    hidden / target are this rank's tokens; W and bias are replicated.  Returns the dict of
    flce_fwd_bwd with the global loss, n_valid, grad_W and grad_bias and this rank's grad_input rows.
    """
    from ._lib import flce_fwd_bwd

    out = flce_fwd_bwd(hidden, W, target, bias=bias, ignore_index=ignore_index, reduction="sum", z_loss=z_loss,
                       **kwargs)
    compose_token_shards(out["loss"], out["n_valid"], out.get("grad_input"), out.get("grad_W"),
                         out.get("grad_bias"), reduction=reduction, group=group)
    return out
