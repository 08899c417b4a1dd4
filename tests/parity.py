"""Tolerances of the parity tests and helpers to move data between numpy and torch.

Floating-point bars (from the stated targets of this library):
  * loss, ce_sum, z_sum: relative error <= 2e-4;
  * every gradient (grad_input, grad_W, grad_bias, dlogits): max-abs error <= 1e-2 * max|ref| and
    relative Frobenius error <= 5e-3;
  * n_valid: exact.
The gradients pass through one bf16 rounding of dlogits (relative 2^-9 per element) before the
tensor-core GEMMs, which puts the expected Frobenius error near 1e-3.
"""
from __future__ import annotations

import numpy as np

LOSS_RTOL = 2e-4
GRAD_MAXABS = 1e-2
GRAD_FROB = 5e-3


def assert_scalar_close(got: float, ref: float, name: str, rtol: float = LOSS_RTOL, atol: float = 1e-6) -> None:
    err = abs(float(got) - float(ref))
    assert err <= max(rtol * abs(float(ref)), atol), f"{name}: got {got!r}, oracle {ref!r}, |err| {err:.3e}"


def assert_grad_close(got, ref, name: str) -> None:
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    assert g.shape == r.shape, f"{name}: shape {g.shape} vs {r.shape}"
    assert np.all(np.isfinite(g)), f"{name}: non-finite values"
    maxref = float(np.max(np.abs(r))) if r.size else 0.0
    diff = g - r
    maxerr = float(np.max(np.abs(diff))) if r.size else 0.0
    if maxref == 0.0:
        assert maxerr == 0.0, f"{name}: oracle is all zero, kernel max |value| {maxerr:.3e}"
        return
    assert maxerr <= GRAD_MAXABS * maxref, f"{name}: max-abs error {maxerr:.3e} > {GRAD_MAXABS} * {maxref:.3e}"
    frob = float(np.linalg.norm(diff)) / float(np.linalg.norm(r))
    assert frob <= GRAD_FROB, f"{name}: relative Frobenius error {frob:.3e} > {GRAD_FROB}"


def assert_within_bound(got, ref, bound, name: str) -> None:
    """The gradient bars applied to the error left after subtracting a per-element allowance (the
    gradient filter's bound): max(|got - ref| - bound, 0)."""
    g = np.asarray(got, dtype=np.float64)
    r = np.asarray(ref, dtype=np.float64)
    excess = np.maximum(np.abs(g - r) - bound, 0.0)
    maxref = float(np.max(np.abs(r)))
    assert float(np.max(excess)) <= GRAD_MAXABS * maxref, f"{name}: error beyond the filter bound"
    assert float(np.linalg.norm(excess)) <= GRAD_FROB * float(np.linalg.norm(r)), f"{name}: Frobenius"


def bf16_tensor(bits: np.ndarray, device="cuda"):
    """uint16 bf16 bit patterns -> torch bfloat16 tensor on the device (bit-exact)."""
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


def bf16_to_numpy_f32(t) -> np.ndarray:
    import torch
    u = t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
    return (u.astype(np.uint32) << 16).view(np.float32)


def check_full_size_rows(exp, gi_rows, gw_rows, gb_rows=None) -> None:
    """Sampled rows of a full-size fused call against the stored oracle rows (tests/golden/expected_*.npz).

    Every sampled row is checked on its own (the gradient bars against that row's own max |ref| and
    norm), so that no row hides behind a larger one.  grad_W rows of vocabulary entries that no token
    targets are the softmax part of the gradient alone, so those rows check the logits recompute, the
    exponentials and the gradient GEMM of the grad_W pass without the onehot term around them; they are
    also checked jointly.  grad_bias: the joint bars over all sampled entries and over the untargeted ones.
    """
    gi_rows = np.asarray(gi_rows, dtype=np.float64)
    gw_rows = np.asarray(gw_rows, dtype=np.float64)
    for i, r in enumerate(exp["rows"]):
        assert_grad_close(gi_rows[i], exp["grad_input_rows"][i], f"grad_input row {int(r)}")
    for i, n in enumerate(exp["vocab_rows"]):
        assert_grad_close(gw_rows[i], exp["grad_W_rows"][i], f"grad_W row {int(n)}")
    free = np.asarray(exp["vocab_target_count"]) == 0
    assert free.sum() >= 8, "the sample needs untargeted vocabulary entries"
    assert np.array_equal(exp["grad_W_rows"][free], exp["grad_W_rows_softmax"][free])
    assert_grad_close(gw_rows[free], exp["grad_W_rows_softmax"][free], "grad_W rows of untargeted entries")
    if gb_rows is not None:
        gb_rows = np.asarray(gb_rows, dtype=np.float64)
        assert_grad_close(gb_rows, exp["grad_bias_rows"], "grad_bias rows")
        assert_grad_close(gb_rows[free], exp["grad_bias_rows_softmax"][free], "grad_bias rows of untargeted entries")
