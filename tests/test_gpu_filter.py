"""Gradient filtering (filter_eps, the skip variant of "Cut Cross Entropy visualized", "Gradient
filtering") against the fp64 oracle on the GPU, through the C ABI.

Stated tolerance: every element of grad_input (grad_W) may differ from the exact gradient by the sum
of |dS| |W| (|dS| |hidden|) over the dS entries whose unscaled value p f - onehot (dS divided by the
row's gradient weight) is at most filter_eps, on top of the usual bars; the loss, n_valid and
grad_bias keep the exact bars.  The bound is evaluated from the oracle's fp64 dS, with a 1/64 margin
on the threshold for the kernel deciding on its fp32 values.  Workloads: logits with a
standard deviation near 5 (a few large probabilities per row, most blocks skippable) and the
near-uniform synthetic case (p ~ 1/V: everything but the target blocks is skippable).
"""
import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import GRAD_MAXABS, assert_scalar_close, assert_within_bound, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def flce():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as m
    m.load()
    return m


def _inputs(BT, H, V, hidden_std, bias, z_loss, reduction, seed, ignore=()):
    w = wl.FusedWorkload("filter", BT=BT, H=H, V=V, hidden_std=hidden_std, w_std=0.02,
                         bias_std=0.1 if bias else None, ignore_frac=0.0, z_loss=z_loss, reduction=reduction,
                         seed=seed)
    d = wl.make_fused_inputs(w)
    for r in ignore:
        d["target"][r] = -100
    return d


def _upload(d):
    import torch
    return (bf16_tensor(d["hidden"]), bf16_tensor(d["W"]), torch.from_numpy(d["target"]).cuda(),
            torch.from_numpy(d["bias"]).cuda() if d["bias"] is not None else None)


CASES = {
    # name: (BT, H, V, hidden std, bias, z_loss, reduction, eps, ignored rows)
    "peaked-two-pairs": (520, 512, 3000, 25.0, True, 1e-4, "mean", 2.0 ** -12, (3, 400)),
    "peaked-one-pair": (300, 128, 2000, 50.0, False, 0.0, "sum", 1e-3, (0,)),
    "uniform-two-pairs": (260, 512, 4000, 1.0, True, 0.0, "mean", 2.0 ** -12, (7,)),
}


def _check_filtered(flce, d, red, zl, eps, **kw):
    """One filtered call against the oracle within the stated bound; returns the workspace."""
    import torch
    V = d["W"].shape[0]
    hidden, W, target, b = _upload(d)
    out = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction=red, z_loss=zl, filter_eps=eps, **kw)
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0
    skips = flce.read_filter_skips(out["workspace"])
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction=red, z_loss=zl)
    dS = oracle.flce_dlogits(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction=red, z_loss=zl)
    # the unscaled gradient: dS over the row's weight s [valid] (rows of zero weight are zero)
    valid = (d["target"] >= 0) & (d["target"] < V)
    s_w = (1.0 / max(int(valid.sum()), 1) if red == "mean" else 1.0) * valid
    unscaled = np.divide(np.abs(dS), s_w[:, None], out=np.zeros_like(dS), where=s_w[:, None] > 0)
    small = np.where(unscaled <= eps * (1.0 + 1.0 / 64), np.abs(dS), 0.0)
    Wf = np.abs(oracle.widen(d["W"]))
    hf = np.abs(oracle.widen(d["hidden"]))
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(out["loss"].item(), ref["loss"], "loss")
    assert_within_bound(bf16_to_numpy_f32(out["grad_input"]), ref["grad_input"], small @ Wf, "grad_input")
    assert_within_bound(out["grad_W"].cpu().numpy(), ref["grad_W"], small.T @ hf, "grad_W")
    if d["bias"] is not None:
        gb = out["grad_bias"].cpu().numpy()
        assert np.max(np.abs(gb - ref["grad_bias"])) <= GRAD_MAXABS * np.max(np.abs(ref["grad_bias"]))
    # the filter must actually have skipped blocks here (both passes counted)
    assert skips > 0, "no dS block was skipped"
    return out["workspace"]


@pytest.mark.parametrize("separate_lse", [False, True], ids=["lse-in-grad-input-pass", "separate-lse-pass"])
@pytest.mark.parametrize("name", sorted(CASES))
def test_filter_within_stated_bound(flce, name, separate_lse):
    # (by default the grad_input pass finds the LSE itself and is exact; only the grad_W pass filters)
    BT, H, V, hs, bias, zl, red, eps, ign = CASES[name]
    d = _inputs(BT, H, V, hs, bias, zl, red, seed=BT + V, ignore=ign)
    _check_filtered(flce, d, red, zl, eps, separate_lse_pass=separate_lse)


def test_filter_with_split_tails(flce):
    # the filtering grad_W pass with token-split clusters (its partial rows merged in order) within the
    # same bound; BT large enough for the split scratch, 8 vocabulary blocks so that blocks are skippable
    d = _inputs(20000, 256, 2000, 25.0, True, 1e-4, "mean", seed=41, ignore=(5, 19999))
    ws = _check_filtered(flce, d, "mean", 1e-4, 2.0 ** -12, token_splits=2)
    assert flce.read_token_split_units(ws) > 0


def test_filter_threshold_below_every_entry_is_exact(flce):
    # a threshold below every nonzero |dS| skips only all-zero blocks (the token padding of the last
    # block of the grad_W pass: 24 halves here): the result must equal the unfiltered call bit for bit
    # (the filtered path starts O from zeros and always accumulates; both compute the LSE in its own pass)
    import torch
    d = _inputs(260, 512, 3000, 1.0, True, 1e-4, "mean", seed=33)
    hidden, W, target, b = _upload(d)
    a = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction="mean", z_loss=1e-4, separate_lse_pass=True)
    c = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction="mean", z_loss=1e-4, filter_eps=1e-30,
                          separate_lse_pass=True)
    torch.cuda.synchronize()
    assert flce.read_filter_skips(c["workspace"]) == 24
    assert torch.equal(a["grad_input"].view(torch.int16), c["grad_input"].view(torch.int16))
    assert torch.equal(a["grad_W"], c["grad_W"])
    assert torch.equal(a["grad_bias"], c["grad_bias"])
    assert torch.equal(a["loss"], c["loss"])
