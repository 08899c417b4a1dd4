"""The bounded waits of the gradient kernels, made to give up on purpose on the GPU.

Every wait inside the tensor-core kernels is bounded; one that gives up raises the CTA's abort flag, the
other roles of the cluster wind down, TMEM is freed and the kernel returns with FLCE_STATUS_TIMEOUT set in
the workspace status word (the bounded replacement of the spin lock of "Cut Cross Entropy visualized",
"Forward kernel").  The test-only option debug_stall_us makes every TMA producer of the gradient passes
first wait for an mbarrier phase that nothing completes, with that short limit, before it issues any copy:
nothing is in flight when the wait gives up, so no GPU can fault or hang.  The call must return the
timeout bit within a fraction of a second, and the next call on the same stream and workspace must be
correct."""
import time

import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("separate", [False, True])
def test_wait_that_gives_up_reports_timeout_and_next_call_is_correct(separate):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as flce
    flce.load()
    w = wl.FusedWorkload("timeout", BT=512, H=256, V=4000, bias_std=0.1, ignore_frac=0.05, z_loss=1e-4, seed=31)
    d = wl.make_fused_inputs(w)
    hidden, W = bf16_tensor(d["hidden"]), bf16_tensor(d["W"])
    target = torch.from_numpy(d["target"]).cuda()
    bias = torch.from_numpy(d["bias"]).cuda()
    kw = dict(bias=bias, z_loss=w.z_loss, separate_lse_pass=separate, vocab_splits=1, token_splits=1)
    out = flce.flce_fwd_bwd(hidden, W, target, **kw)   # warm-up: module load, occupancy queries
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0
    ws = out["workspace"]
    res = {k: v for k, v in out.items() if k in ("loss", "n_valid", "grad_input", "grad_W", "grad_bias")}
    t0 = time.perf_counter()
    flce.flce_fwd_bwd(hidden, W, target, workspace=ws, out=res, debug_stall_us=2000, **kw)
    st = flce.read_device_status(ws)
    dt = time.perf_counter() - t0
    assert st & flce.STATUS_TIMEOUT, f"status {st:#x}: the stalled wait did not report a timeout"
    assert dt < 1.0, f"the stalled call took {dt:.3f} s (the 2 ms limit, not the 4 s default, should end it)"
    # the context and the workspace stay usable: the next call is correct and reports no error
    flce.flce_fwd_bwd(hidden, W, target, workspace=ws, out=res, **kw)
    assert flce.read_device_status(ws) == 0
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], z_loss=w.z_loss)
    assert int(res["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(res["loss"].item(), ref["loss"], "loss")
    assert_grad_close(bf16_to_numpy_f32(res["grad_input"]), ref["grad_input"], "grad_input")
    assert_grad_close(res["grad_W"].cpu().numpy(), ref["grad_W"], "grad_W")
    assert_grad_close(res["grad_bias"].cpu().numpy(), ref["grad_bias"], "grad_bias")


def test_wait_that_gives_up_in_persistent_clusters():
    """The same in a pass run by persistent clusters: the grad_W pass of this shape (118 vocabulary row
    pairs of 17 token blocks) runs four-pair clusters with side and single-pair clusters beside them.
    Every unit's producer stalls, so every cluster gives up in its first unit; the claim of a next unit
    then sees the abort and the cluster stops.  The call reports the timeout within a fraction of a second,
    and the next call gives the results of a call before it bit for bit."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as flce
    flce.load()
    w = wl.FusedWorkload("timeout-persistent", BT=4100, H=1024, V=30000, bias_std=0.1, ignore_frac=0.05,
                         z_loss=1e-4, seed=37)
    d = wl.make_fused_inputs(w)
    hidden, W = bf16_tensor(d["hidden"]), bf16_tensor(d["W"])
    target = torch.from_numpy(d["target"]).cuda()
    bias = torch.from_numpy(d["bias"]).cuda()
    kw = dict(bias=bias, z_loss=w.z_loss)
    first = flce.flce_fwd_bwd(hidden, W, target, **kw)
    torch.cuda.synchronize()
    ws = first["workspace"]
    assert flce.read_device_status(ws) == 0
    assert flce.read_side_launches(ws) == 1 and flce.read_single_launches(ws) == 1
    res = {k: v for k, v in first.items() if k in ("loss", "n_valid", "grad_input", "grad_W", "grad_bias")}
    before = {k: v.clone() for k, v in res.items()}
    t0 = time.perf_counter()
    flce.flce_fwd_bwd(hidden, W, target, workspace=ws, out=res, debug_stall_us=2000, **kw)
    st = flce.read_device_status(ws)
    dt = time.perf_counter() - t0
    assert st & flce.STATUS_TIMEOUT, f"status {st:#x}: the stalled wait did not report a timeout"
    assert dt < 1.0, f"the stalled call took {dt:.3f} s"
    flce.flce_fwd_bwd(hidden, W, target, workspace=ws, out=res, **kw)
    assert flce.read_device_status(ws) == 0
    assert flce.read_side_launches(ws) == 1
    for k, v in before.items():
        assert torch.equal(res[k], v), f"{k} differs after the stalled call"
