"""The full-size sampled checks (parity.check_full_size_rows) against planted mistakes, on the CPU.

The GPU test compares a full-size call's sampled rows with the oracle's stored rows.  Here the stored
rows themselves stand in for a kernel's output: rounded to the output precision they must pass, and
with a plausible mistake planted in them they must fail.  The mistakes: the softmax part of dlogits
dropped from a gradient GEMM (what remains is the onehot term alone), the softmax part scaled by 1.01
(an LSE off by 0.01; grad_W only), and the onehot term dropped.
"""
import os

import numpy as np
import pytest

from parity import bf16_to_numpy_f32, check_full_size_rows  # noqa: F401

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")
KEYS = ["qwen3", "gemma2", "long"]


def _load(key):
    return dict(np.load(os.path.join(GOLDEN, f"expected_{key}.npz")))


def _bf16_round(x):
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16   # round to nearest even
    return (u.astype(np.uint32) << 16).view(np.float32)


def _parts(exp):
    gi, gw = exp["grad_input_rows"], exp["grad_W_rows"]
    gis, gws = exp["grad_input_rows_softmax"], exp["grad_W_rows_softmax"]
    gb, gbs = exp.get("grad_bias_rows"), exp.get("grad_bias_rows_softmax")
    return gi, gw, gb, gis, gws, gbs


@pytest.mark.parametrize("key", KEYS)
def test_stored_rows_pass_at_output_precision(key):
    exp = _load(key)
    gi, gw, gb, *_ = _parts(exp)
    check_full_size_rows(exp, _bf16_round(gi), gw.astype(np.float32), None if gb is None else gb.astype(np.float32))


@pytest.mark.parametrize("key", KEYS)
@pytest.mark.parametrize("which", ["grad_input", "grad_W"])
@pytest.mark.parametrize("mistake", ["softmax part dropped", "softmax part x 1.01", "onehot term dropped"])
def test_planted_mistake_fails(key, which, mistake):
    exp = _load(key)
    gi, gw, gb, gis, gws, gbs = _parts(exp)
    if mistake == "softmax part dropped":
        bad = {"grad_input": gi - gis, "grad_W": gw - gws}
    elif mistake == "softmax part x 1.01":
        bad = {"grad_input": gi + 0.01 * gis, "grad_W": gw + 0.01 * gws}
    else:
        bad = {"grad_input": gis, "grad_W": gws}
    if which == "grad_input" and mistake == "softmax part x 1.01":
        # the softmax part of a grad_input row is ~2% of the row (the row is dominated by -s W[y]), so 1% of
        # it is below the bf16 rounding of the stored gradient: this mistake shows in grad_W only
        pytest.skip("below the output resolution of grad_input")
    got_gi = bad["grad_input"] if which == "grad_input" else gi
    got_gw = bad["grad_W"] if which == "grad_W" else gw
    with pytest.raises(AssertionError):
        check_full_size_rows(exp, _bf16_round(got_gi), got_gw.astype(np.float32), gb)
