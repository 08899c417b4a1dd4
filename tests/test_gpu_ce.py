"""Standalone CE kernel (ce_with_grad) against the fp64 oracle on the GPU, through the C ABI."""
import os

import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu
GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def flce():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as m
    m.load()
    return m


def _case(B, V, std=2.0, ignore=(), bad=(), seed=0):
    rng = np.random.default_rng(seed)
    x = wl.f32_to_bf16_bits((rng.standard_normal((B, V)) * std).astype(np.float32))
    lab = rng.integers(0, V, B).astype(np.int64)
    for r in ignore:
        lab[r] = -100
    for r in bad:
        lab[r] = V + 3
    return x, lab


def _run(flce, x, lab, z_loss):
    import torch
    logits = bf16_tensor(x)
    labels = torch.from_numpy(lab).cuda()
    out = flce.ce_with_grad(logits, labels, ignore_index=-100, z_loss=z_loss)
    torch.cuda.synchronize()
    status = flce.read_device_status(out["workspace"])
    return out, logits, status


@pytest.mark.parametrize("B,V,z_loss,ignore", [
    (64, 1000, 1e-4, (3, 10)),       # several 16-byte vectors per thread, ignored rows
    (37, 1003, 0.0, (0,)),           # V % 8 != 0: rows are not 16-byte aligned (scalar head/tail)
    (16, 8, 1e-2, ()),               # one vector per row
    (5, 1, 1e-2, (2,)),              # V = 1: the CE part vanishes
    (300, 4101, 1e-4, (7, 299)),     # more rows than a few CTAs, ragged
    (3, 200003, 1e-4, ()),           # long rows: many iterations per thread
    # aligned rows longer than the shared-memory head (the rest of each row re-read in pass 2)
    (40, 65536, 0.0, ()),
    (300, 50000, 1e-4, (5, 299)),    # many rows per CTA
    (7, 131064, 1e-3, (2,)),
])
def test_ce_matches_oracle(flce, B, V, z_loss, ignore):
    x, lab = _case(B, V, ignore=ignore, seed=B + V)
    out, logits, status = _run(flce, x, lab, z_loss)
    ref = oracle.ce_reference(x, lab, z_loss=z_loss)
    assert status == 0
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(out["ce_sum"].item(), ref["ce_sum"], "ce_sum")
    assert_scalar_close(out["z_sum"].item(), ref["z_sum"], "z_sum")
    assert_grad_close(bf16_to_numpy_f32(logits), ref["dlogits"], "dlogits")


def test_ce_all_ignored_and_bad_labels(flce):
    x, lab = _case(20, 300, ignore=range(20))
    out, logits, status = _run(flce, x, lab, 1e-4)
    assert status == 0
    assert int(out["n_valid"].item()) == 0 and out["ce_sum"].item() == 0.0 and out["z_sum"].item() == 0.0
    assert np.all(bf16_to_numpy_f32(logits) == 0.0)
    # a label outside [0, V) that is not ignore_index: the row is treated as ignored and flagged
    for V in (500, 48000):   # (the second with rows longer than the shared-memory head)
        x, lab = _case(12, V, ignore=(1,), bad=(4, 9))
        out, logits, status = _run(flce, x, lab, 1e-4)
        assert status & flce.STATUS_BAD_TARGET
        ref = oracle.ce_reference(x, lab, z_loss=1e-4)
        assert int(out["n_valid"].item()) == ref["n_valid"] == 9
        assert_scalar_close(out["ce_sum"].item(), ref["ce_sum"], "ce_sum")
        assert_grad_close(bf16_to_numpy_f32(logits), ref["dlogits"], "dlogits")


def test_ce_empty(flce):
    import torch
    logits = torch.empty((0, 128), dtype=torch.bfloat16, device="cuda")
    labels = torch.empty((0,), dtype=torch.int64, device="cuda")
    out = flce.ce_with_grad(logits, labels)
    assert out["ce_sum"].item() == 0.0 and out["z_sum"].item() == 0.0 and out["n_valid"].item() == 0


def test_ce_full_size(flce):
    """[8192, 128256] bf16 logits, sum, z-loss 1e-4: sums against the stored oracle values, sampled
    dlogits rows against the oracle computed here, and bitwise-equal results on a second call."""
    import torch
    w = wl.CE_LOGITS
    exp = np.load(os.path.join(GOLDEN, "expected_ce.npz"))
    d = wl.make_ce_inputs(w)
    assert wl.digest(d["logits"], d["labels"]) == str(exp["digest"]), "input generator drifted from the stored digest"
    out, logits, status = _run(flce, d["logits"], d["labels"], w.z_loss)
    assert status == 0
    assert int(out["n_valid"].item()) == int(exp["n_valid"])
    assert_scalar_close(out["ce_sum"].item(), float(exp["ce_sum"]), "ce_sum")
    assert_scalar_close(out["z_sum"].item(), float(exp["z_sum"]), "z_sum")
    rows = exp["rows"]
    ref = oracle.ce_reference(d["logits"][rows], d["labels"][rows], z_loss=w.z_loss)
    got = bf16_to_numpy_f32(logits[torch.from_numpy(rows).cuda()])
    assert_grad_close(got, ref["dlogits"], "dlogits rows")
    first = (out["ce_sum"].item(), out["z_sum"].item())
    del logits
    out2, logits2, _ = _run(flce, d["logits"], d["labels"], w.z_loss)
    assert (out2["ce_sum"].item(), out2["z_sum"].item()) == first, "reduction is not deterministic"


@pytest.mark.parametrize("dtype", ["float16", "float32", "bfloat16"])
@pytest.mark.parametrize("mode", ["inplace", "separate", "nograd"])
@pytest.mark.parametrize("B,V,z_loss,ignore", [(300, 4101, 1e-4, (7, 299)), (37, 1003, 0.0, (0,)), (4, 130001, 1e-3, (1,)),
                                                (6, 65536, 1e-3, (1,))])
def test_ce_dtypes_and_modes(flce, dtype, mode, B, V, z_loss, ignore):
    import torch
    tdt = getattr(torch, dtype)
    rng = np.random.default_rng(B * 7 + V)
    x32 = (rng.standard_normal((B, V)) * 2.0).astype(np.float32)
    lab = rng.integers(0, V, B).astype(np.int64)
    for r in ignore:
        lab[r] = -100
    logits = torch.from_numpy(x32).to(tdt).cuda()
    xin = logits.float().cpu().numpy().astype(np.float64)    # the exact values the kernel reads
    orig = logits.clone()
    labels = torch.from_numpy(lab).cuda()
    if mode == "inplace":
        r = flce.ce_with_grad(logits, labels, z_loss=z_loss)
        dl = logits
    else:
        r = flce.cross_entropy(logits, labels, z_loss=z_loss, want_grad=(mode == "separate"))
        dl = r["dlogits"]
    torch.cuda.synchronize()
    assert flce.read_device_status(r["workspace"]) == 0
    ref = oracle.ce_reference(xin, lab, z_loss=z_loss)
    assert int(r["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(r["ce_sum"].item(), ref["ce_sum"], "ce_sum")
    assert_scalar_close(r["z_sum"].item(), ref["z_sum"], "z_sum")
    if mode != "inplace":
        assert torch.equal(logits, orig), "the logits must be left unchanged"
    if mode == "nograd":
        assert dl is None
        return
    assert dl.dtype == tdt
    assert_grad_close(dl.float().cpu().numpy(), ref["dlogits"], "dlogits")


def test_ce_separate_equals_inplace_bitwise(flce):
    # the non-mutating form runs the same arithmetic: its dlogits must equal the in-place result bit for bit
    import torch
    for B, V in ((96, 5003), (33, 60000)):   # (the second with rows longer than the shared-memory head)
        x, lab = _case(B, V, ignore=(3,), seed=11)
        a = bf16_tensor(x)
        labels = torch.from_numpy(lab).cuda()
        r = flce.cross_entropy(a, labels, z_loss=1e-4)
        b = bf16_tensor(x)
        flce.ce_with_grad(b, labels, z_loss=1e-4)
        torch.cuda.synchronize()
        assert torch.equal(r["dlogits"].view(torch.int16), b.view(torch.int16))
        assert torch.equal(a.view(torch.int16), bf16_tensor(x).view(torch.int16))
