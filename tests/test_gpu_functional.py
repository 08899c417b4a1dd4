"""The autograd forms (linear_cross_entropy_tma_gb300.functional) against the fp64 oracle on the GPU:
``loss.backward()`` with an upstream gradient other than 1 gives the oracle's gradients times that
gradient, for the mean, sum and unreduced losses of the fused call and the mean and sum of the standalone
CE ("Greyhound -- Cross-Entropy", "Usage": normal autograd semantics, logits left unchanged).  Also the
gradient-scaling kernel itself on every dtype, ragged lengths and the factor 1."""
import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def F():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as m
    m.load()
    from linear_cross_entropy_tma_gb300 import functional
    return functional


def _fused_case(BT=300, H=128, V=1000, seed=21):
    w = wl.FusedWorkload("autograd", BT=BT, H=H, V=V, bias_std=0.1, ignore_frac=0.05, z_loss=1e-3, seed=seed)
    return wl.make_fused_inputs(w)


@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_linear_cross_entropy_backward(F, reduction):
    import torch
    d = _fused_case()
    hidden = bf16_tensor(d["hidden"]).requires_grad_(True)
    W = bf16_tensor(d["W"]).requires_grad_(True)
    bias = torch.from_numpy(d["bias"]).cuda().requires_grad_(True)
    target = torch.from_numpy(d["target"]).cuda()
    loss = F.linear_cross_entropy(hidden, W, target, bias=bias, reduction=reduction, z_loss=d["z_loss"])
    assert loss.dim() == 0 and loss.requires_grad
    (0.75 * loss).backward()
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction=reduction,
                                z_loss=d["z_loss"], grad_scale=0.75)
    assert_scalar_close(loss.item(), ref["loss"], "loss")
    assert hidden.grad.dtype == torch.bfloat16 and bias.grad.dtype == torch.float32
    assert_grad_close(bf16_to_numpy_f32(hidden.grad), ref["grad_input"], "hidden.grad")
    # (autograd hands W's gradient over in W's dtype, bf16)
    assert_grad_close(W.grad.float().cpu().numpy(), ref["grad_W"], "W.grad")
    assert_grad_close(bias.grad.cpu().numpy(), ref["grad_bias"], "bias.grad")


def test_linear_cross_entropy_none_and_partial_requires_grad(F):
    import torch
    d = _fused_case(BT=260, H=64, V=700, seed=22)
    hidden = bf16_tensor(d["hidden"]).requires_grad_(True)
    W = bf16_tensor(d["W"])            # no gradient for W: only the grad_input pass runs
    target = torch.from_numpy(d["target"]).cuda()
    per_tok = F.linear_cross_entropy(hidden, W, target, reduction="none", z_loss=d["z_loss"])
    assert per_tok.shape == (260,)
    u = torch.from_numpy(np.random.default_rng(5).standard_normal(260).astype(np.float32)).cuda()
    (per_tok * u).sum().backward()
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], reduction="none", z_loss=d["z_loss"],
                                grad_loss_per_token=u.cpu().numpy())
    assert_grad_close(per_tok.detach().cpu().numpy(), ref["loss_per_token"], "per-token loss")
    assert_grad_close(bf16_to_numpy_f32(hidden.grad), ref["grad_input"], "hidden.grad")
    assert W.grad is None


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("reduction", ["mean", "sum"])
def test_cross_entropy_backward(F, dtype, reduction):
    import torch
    c = wl.make_ce_inputs(wl.CEWorkload("autograd ce", B=97, V=3001, seed=3))
    if dtype == "bf16":
        x = bf16_tensor(c["logits"])
    else:
        x = torch.from_numpy(bf16_to_numpy_f32_np(c["logits"])).cuda()
    before = x.clone()
    x.requires_grad_(True)
    labels = torch.from_numpy(c["labels"]).cuda()
    loss = F.cross_entropy(x, labels, z_loss=c["z_loss"], reduction=reduction)
    (2.0 * loss).backward()
    ref = oracle.ce_reference(c["logits"], c["labels"], z_loss=c["z_loss"])
    s = 1.0 / max(ref["n_valid"], 1) if reduction == "mean" else 1.0
    assert_scalar_close(loss.item(), s * (ref["ce_sum"] + c["z_loss"] * ref["z_sum"]), "loss")
    assert torch.equal(x.detach(), before), "the logits were modified"
    assert x.grad.dtype == x.dtype
    g = bf16_to_numpy_f32(x.grad) if dtype == "bf16" else x.grad.cpu().numpy()
    assert_grad_close(g, 2.0 * s * ref["dlogits"], "logits.grad")


def bf16_to_numpy_f32_np(bits):
    return (np.asarray(bits).astype(np.uint32) << 16).view(np.float32)


@pytest.mark.parametrize("dtype", ["bf16", "f16", "f32"])
@pytest.mark.parametrize("n", [1, 7, 8, 4099, 1 << 20])
def test_scale_gradient_kernel(F, dtype, n):
    import torch
    from linear_cross_entropy_tma_gb300 import _lib
    tdt = {"bf16": torch.bfloat16, "f16": torch.float16, "f32": torch.float32}[dtype]
    rng = np.random.default_rng(n)
    x64 = rng.standard_normal(n)
    x = torch.from_numpy(x64.astype(np.float32)).cuda().to(tdt)
    ref = x.double().cpu().numpy()
    up = torch.tensor([-1.7], dtype=torch.float32, device="cuda")
    div = torch.tensor([5], dtype=torch.int64, device="cuda")
    y = x.clone()
    _lib.scale_gradient_(y, up, div)
    want = ref * (np.float32(-1.7) / np.float32(5.0))
    got = y.double().cpu().numpy()
    # one rounding to nearest: half an ulp relative, or half the smallest subnormal step absolute (fp16)
    ulp = {"bf16": 2.0 ** -8, "f16": 2.0 ** -11, "f32": 2.0 ** -23}[dtype]
    tiny = {"bf16": 2.0 ** -134, "f16": 2.0 ** -25, "f32": 2.0 ** -150}[dtype]
    assert np.all(np.abs(got - want) <= ulp * np.abs(want) + tiny), dtype
    # the factor 1 leaves the buffer untouched; a divisor of 0 counts as 1
    z = x.clone()
    _lib.scale_gradient_(z, torch.ones(1, device="cuda"), torch.zeros(1, dtype=torch.int64, device="cuda"))
    assert torch.equal(z, x)
    torch.cuda.synchronize()


def test_ce_reduce_loss_kernel(F):
    import torch
    from linear_cross_entropy_tma_gb300 import _lib
    cs = torch.tensor([10.5], device="cuda")
    zs = torch.tensor([300.0], device="cuda")
    for n, red, want in ((4, "mean", (10.5 + 0.01 * 300.0) / 4), (0, "mean", 10.5 + 3.0), (4, "sum", 13.5)):
        nv = torch.tensor([n], dtype=torch.int64, device="cuda")
        got = _lib.ce_reduce_loss(cs, zs, nv, z_loss=0.01, reduction=red).item()
        assert abs(got - want) <= 1e-6 * abs(want), (n, red, got, want)
