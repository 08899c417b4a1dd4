"""flce_fwd_bwd_ex options against the fp64 oracle on the GPU, through the C ABI: reduction "none" with
per-token upstream gradients (positive, negative and zero), a scalar gradient scale (including a
negative one, which takes the general form of the dS arithmetic), per-token losses, and accumulation
into existing gradient buffers, and the per-row entropy output.  Sizes span several tiles, ragged tails, and both the one-pair (H <=
256) and the cluster (H = 512, two pairs sharing each logits tile) variants of the gradient passes.
"""
import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def flce():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as m
    m.load()
    return m


def _inputs(BT, H, V, bias, z_loss, seed, ignore=()):
    w = wl.FusedWorkload("opt", BT=BT, H=H, V=V, hidden_std=1.0, w_std=0.02, bias_std=0.1 if bias else None,
                         ignore_frac=0.0, z_loss=z_loss, reduction="mean", seed=seed)
    d = wl.make_fused_inputs(w)
    for r in ignore:
        d["target"][r] = -100
    return d


def _upload(d):
    import torch
    return (bf16_tensor(d["hidden"]), bf16_tensor(d["W"]), torch.from_numpy(d["target"]).cuda(),
            torch.from_numpy(d["bias"]).cuda() if d["bias"] is not None else None)


def _compare(out, ref, with_grads=True, base=None):
    base = base or {}
    assert int(out["n_valid"].item()) == ref["n_valid"]
    if with_grads:
        for k in ("grad_input", "grad_W", "grad_bias"):
            if out.get(k) is None:
                continue
            got = bf16_to_numpy_f32(out[k]) if k == "grad_input" else out[k].cpu().numpy()
            want = ref[k] + base.get(k, 0.0)
            assert_grad_close(got, want, k)


SHAPES = {
    # name: (BT, H, V, bias, z_loss, ignored rows)
    "one-pair": (300, 128, 1000, True, 1e-3, (0, 150, 299)),
    "two-pairs": (260, 512, 3000, True, 1e-4, (7,)),
}


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("signs", ["positive", "mixed"])
def test_unreduced_with_upstream_gradient(flce, shape, signs):
    import torch
    BT, H, V, bias, zl, ign = SHAPES[shape]
    d = _inputs(BT, H, V, bias, zl, seed=BT + H, ignore=ign)
    rng = np.random.Generator(np.random.PCG64(5))
    g = rng.uniform(0.2, 2.0, BT).astype(np.float32)
    if signs == "mixed":
        g[::3] *= -1.0
        g[1::7] = 0.0
    gs = 0.5
    hidden, W, target, b = _upload(d)
    out = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction="none", z_loss=zl, grad_scale=gs,
                            grad_loss_per_token=torch.from_numpy(g).cuda())
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="none", z_loss=zl,
                                grad_scale=gs, grad_loss_per_token=g.astype(np.float64))
    lt = out["loss_per_token"].cpu().numpy()
    assert_grad_close(lt, ref["loss_per_token"], "loss_per_token")
    assert np.all(lt[list(ign)] == 0.0)
    assert_scalar_close(out["loss"].item(), ref["loss"], "loss (sum of per-token losses)")
    _compare(out, ref)


@pytest.mark.parametrize("shape", sorted(SHAPES))
@pytest.mark.parametrize("reduction,gs", [("mean", -1.5), ("sum", 0.25), ("mean", 0.0)])
def test_grad_scale(flce, shape, reduction, gs):
    import torch
    BT, H, V, bias, zl, ign = SHAPES[shape]
    d = _inputs(BT, H, V, bias, zl, seed=3 * BT + H, ignore=ign)
    hidden, W, target, b = _upload(d)
    out = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction=reduction, z_loss=zl, grad_scale=gs,
                            want_loss_per_token=True)
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction=reduction, z_loss=zl,
                                grad_scale=gs)
    assert_scalar_close(out["loss"].item(), ref["loss"], "loss")
    assert_grad_close(out["loss_per_token"].cpu().numpy(), ref["loss_per_token"], "loss_per_token")
    _compare(out, ref)


@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_accumulate(flce, shape):
    import torch
    BT, H, V, bias, zl, ign = SHAPES[shape]
    d = _inputs(BT, H, V, bias, zl, seed=5 * BT + H, ignore=ign)
    hidden, W, target, b = _upload(d)
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="sum", z_loss=zl)
    rng = np.random.Generator(np.random.PCG64(9))
    gi0 = wl.f32_to_bf16_bits((rng.standard_normal((BT, H)) * np.std(ref["grad_input"])).astype(np.float32))
    gw0 = (rng.standard_normal((V, H)) * np.std(ref["grad_W"])).astype(np.float32)
    gb0 = (rng.standard_normal(V) * np.std(ref["grad_bias"])).astype(np.float32)
    out = {"grad_input": bf16_tensor(gi0), "grad_W": torch.from_numpy(gw0.copy()).cuda(),
           "grad_bias": torch.from_numpy(gb0.copy()).cuda()}
    res = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction="sum", z_loss=zl, accumulate=True, out=out)
    torch.cuda.synchronize()
    assert flce.read_device_status(res["workspace"]) == 0
    assert_scalar_close(res["loss"].item(), ref["loss"], "loss")
    base = {"grad_input": (gi0.astype(np.uint32) << 16).view(np.float32).astype(np.float64),
            "grad_W": gw0.astype(np.float64), "grad_bias": gb0.astype(np.float64)}
    _compare(res, ref, base=base)


def test_unreduced_empty_batch_leaves_accumulators(flce):
    import torch
    d = _inputs(1, 64, 100, True, 0.0, seed=1)
    hidden, W, _, b = _upload(d)
    target = torch.empty(0, dtype=torch.int64, device="cuda")
    gw0 = torch.full((100, 64), 0.5, device="cuda")
    gb0 = torch.full((100,), -0.25, device="cuda")
    res = flce.flce_fwd_bwd(hidden[:0], W, target, bias=b, reduction="none", need_grad_input=False,
                            accumulate=True, out={"grad_W": gw0, "grad_bias": gb0})
    torch.cuda.synchronize()
    assert int(res["n_valid"].item()) == 0
    assert torch.all(gw0 == 0.5) and torch.all(gb0 == -0.25)
    assert res["loss"].item() == 0.0


@pytest.mark.parametrize("separate_lse", [False, True], ids=["lse-in-grad-input-pass", "separate-lse-pass"])
@pytest.mark.parametrize("shape", sorted(SHAPES))
def test_entropy(flce, shape, separate_lse):
    # per-row entropy of softmax(z); tolerance: H = LSE - sum p z is a difference of two fp32 quantities of
    # size about LSE, so each row is held to the loss bar relative to max(1, LSE)
    import torch
    BT, H, V, bias, zl, ign = SHAPES[shape]
    d = _inputs(BT, H, V, bias, zl, seed=7 * BT + H, ignore=ign)
    hidden, W, target, b = _upload(d)
    out = flce.flce_fwd_bwd(hidden, W, target, bias=b, reduction="mean", z_loss=zl, want_entropy=True,
                            separate_lse_pass=separate_lse)
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="mean", z_loss=zl)
    got = out["entropy"].cpu().numpy().astype(np.float64)
    err = np.abs(got - ref["entropy"])
    assert np.all(err <= 2e-4 * np.maximum(1.0, ref["lse"])), float(np.max(err))
    # the other outputs are unchanged by the extra accumulation
    assert_scalar_close(out["loss"].item(), ref["loss"], "loss")
    _compare(out, ref)


@pytest.mark.parametrize("separate_lse", [False, True], ids=["lse-in-grad-input-pass", "separate-lse-pass"])
def test_entropy_peaked(flce, separate_lse):
    # logits with a standard deviation near 5 (hidden scaled): low-entropy rows
    import torch
    w = wl.FusedWorkload("peaked", BT=130, H=64, V=700, hidden_std=31.0, w_std=0.02, bias_std=None,
                         ignore_frac=0.0, z_loss=0.0, reduction="sum", seed=21)
    d = wl.make_fused_inputs(w)
    hidden, W, target, b = _upload(d)
    out = flce.flce_fwd_bwd(hidden, W, target, reduction="sum", want_entropy=True, need_grad_W=False,
                            separate_lse_pass=separate_lse)
    torch.cuda.synchronize()
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], reduction="sum", want_grads=False)
    got = out["entropy"].cpu().numpy().astype(np.float64)
    assert float(np.min(ref["entropy"])) < 1.0
    assert np.all(np.abs(got - ref["entropy"]) <= 2e-4 * np.maximum(1.0, np.abs(ref["lse"])))
