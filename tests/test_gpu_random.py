"""Seeded randomised shapes and option combinations against the fp64 oracle, through the C ABI.

flce_fwd_bwd: ragged BT / V / H (H a multiple of 8), bias, z-loss, the three reductions with per-token
upstream gradients, ignored rows, both flows, forced vocabulary / token splits, accumulation and the
vocabulary sort.  The standalone CE kernel:
aligned and ragged rows, the three logits types, in place / separate / loss only, ignored and
out-of-range labels.  Element-wise bars as in the other parity tests."""
import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu
N_CASES = 24


@pytest.fixture(scope="module")
def flce():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as m
    m.load()
    return m


def _case(i):
    rng = np.random.Generator(np.random.PCG64(1000 + i))
    BT = int(rng.integers(1, 700))
    H = 8 * int(rng.integers(1, 145))          # 8 .. 1152
    V = int(rng.integers(1, 5000))
    opts = dict(
        bias=bool(rng.integers(0, 2)),
        z_loss=float(rng.choice([0.0, 1e-4, 1e-2])),
        reduction=str(rng.choice(["mean", "sum", "none"])),
        separate_lse_pass=bool(rng.integers(0, 4) == 0),
        vocab_splits=int(rng.choice([0, 1, 2, 3])),
        ignore=int(rng.integers(0, 3)),
        hidden_std=float(rng.choice([1.0, 4.0])),
    )
    # drawn after the above, so that adding them left the earlier draws of each case unchanged
    opts["accumulate"] = bool(rng.integers(0, 4) == 0)
    opts["sort_vocab"] = bool(rng.integers(0, 4) == 0)
    opts["token_splits"] = int(rng.choice([0, 0, 1, 2]))
    return BT, H, V, opts, rng


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_case(flce, i):
    import torch
    BT, H, V, o, rng = _case(i)
    w = wl.FusedWorkload("random", BT=BT, H=H, V=V, hidden_std=o["hidden_std"], w_std=0.02,
                         bias_std=0.1 if o["bias"] else None, ignore_frac=0.0, z_loss=o["z_loss"],
                         reduction=o["reduction"], seed=2000 + i)
    d = wl.make_fused_inputs(w)
    for r in rng.choice(BT, size=min(o["ignore"], BT), replace=False):
        d["target"][r] = -100
    gtok = (rng.standard_normal(BT).astype(np.float32) if o["reduction"] == "none" else None)
    hidden, W = bf16_tensor(d["hidden"]), bf16_tensor(d["W"])
    target = torch.from_numpy(d["target"]).cuda()
    bias = torch.from_numpy(d["bias"]).cuda() if d["bias"] is not None else None
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction=o["reduction"],
                                z_loss=o["z_loss"], grad_loss_per_token=gtok)
    acc, gi0, gw0, gb0 = None, 0.0, 0.0, 0.0
    if o["accumulate"]:
        # existing gradients of the same magnitude to add to
        gi0b = wl.f32_to_bf16_bits((rng.standard_normal((BT, H)) * (np.std(ref["grad_input"]) + 1e-6)).astype(np.float32))
        gi0 = (gi0b.astype(np.uint32) << 16).view(np.float32)
        gw0 = (rng.standard_normal((V, H)) * (np.std(ref["grad_W"]) + 1e-6)).astype(np.float32)
        acc = {"grad_input": bf16_tensor(gi0b), "grad_W": torch.from_numpy(gw0.copy()).cuda()}
        if d["bias"] is not None:
            gb0 = (rng.standard_normal(V) * (np.std(ref["grad_bias"]) + 1e-6)).astype(np.float32)
            acc["grad_bias"] = torch.from_numpy(gb0.copy()).cuda()
    out = flce.flce_fwd_bwd(hidden, W, target, bias=bias, reduction=o["reduction"], z_loss=o["z_loss"],
                            grad_loss_per_token=torch.from_numpy(gtok).cuda() if gtok is not None else None,
                            separate_lse_pass=o["separate_lse_pass"], vocab_splits=o["vocab_splits"],
                            token_splits=o["token_splits"], sort_vocab=o["sort_vocab"],
                            accumulate=o["accumulate"], out=acc)
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0, f"case {i}: {BT}x{H}x{V} {o}"
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(out["loss"].item(), ref["loss"], f"loss (case {i})")
    if o["reduction"] == "none":
        assert_grad_close(out["loss_per_token"].cpu().numpy(), ref["loss_per_token"], f"loss_per_token (case {i})")
    assert_grad_close(bf16_to_numpy_f32(out["grad_input"]), ref["grad_input"] + gi0, f"grad_input (case {i})")
    assert_grad_close(out["grad_W"].cpu().numpy(), ref["grad_W"] + gw0, f"grad_W (case {i})")
    if d["bias"] is not None:
        assert_grad_close(out["grad_bias"].cpu().numpy(), ref["grad_bias"] + gb0, f"grad_bias (case {i})")


@pytest.mark.parametrize("i", range(N_CASES))
def test_random_ce_case(flce, i):
    # the standalone CE kernel: random rows / vocabulary (aligned or not), dtype, in place / separate /
    # loss only, ignored and out-of-range labels
    import torch
    rng = np.random.Generator(np.random.PCG64(3000 + i))
    B = int(rng.integers(1, 400))
    V = int(rng.integers(1, 60000)) if rng.integers(0, 2) else 8 * int(rng.integers(1, 8000))
    dtype = str(rng.choice(["bfloat16", "float16", "float32"]))
    mode = str(rng.choice(["inplace", "separate", "nograd"]))
    z_loss = float(rng.choice([0.0, 1e-4, 1e-2]))
    x32 = (rng.standard_normal((B, V)) * float(rng.choice([1.0, 3.0]))).astype(np.float32)
    lab = rng.integers(0, V, B).astype(np.int64)
    n_ign = int(rng.integers(0, 3))
    for r in rng.choice(B, size=min(n_ign, B), replace=False):
        lab[r] = -100
    bad = bool(rng.integers(0, 4) == 0) and B > 1
    if bad:
        lab[B - 1] = V + 7
    logits = torch.from_numpy(x32).to(getattr(torch, dtype)).cuda()
    xin = logits.float().cpu().numpy().astype(np.float64)
    labels = torch.from_numpy(lab).cuda()
    if mode == "inplace":
        r = flce.ce_with_grad(logits, labels, z_loss=z_loss)
        dl = logits
    else:
        r = flce.cross_entropy(logits, labels, z_loss=z_loss, want_grad=(mode == "separate"))
        dl = r["dlogits"]
    torch.cuda.synchronize()
    status = flce.read_device_status(r["workspace"])
    assert status == (flce.STATUS_BAD_TARGET if bad else 0), f"case {i}: B={B} V={V} {dtype} {mode}"
    ref = oracle.ce_reference(xin, lab, z_loss=z_loss)
    assert int(r["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(r["ce_sum"].item(), ref["ce_sum"], f"ce_sum (case {i})")
    assert_scalar_close(r["z_sum"].item(), ref["z_sum"], f"z_sum (case {i})")
    if mode != "nograd":
        assert_grad_close(dl.float().cpu().numpy(), ref["dlogits"], f"dlogits (case {i})")
