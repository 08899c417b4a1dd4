"""Host-side checks of the seeded input generators (no GPU)."""
import numpy as np
import torch

from linear_cross_entropy_tma_gb300 import workloads as wl


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * s for s in (1e-3, 0.02, 1, 300)])
    x = np.concatenate([x, np.array([0.0, -0.0, 1.0, 1.00390625, 1.005859375, 65504.0], np.float32)])
    ours = wl.f32_to_bf16_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)
    assert np.array_equal(wl.bf16_bits_to_f32(ours), torch.from_numpy(x).to(torch.bfloat16).float().numpy())


def test_ignore_counts():
    # exactly rint(p * BT) ignored rows (half to even)
    assert [w.n_valid for w in (wl.TINY, wl.QWEN3_0P6B, wl.GEMMA2_2B, wl.LONG_BATCH)] == [122, 3686, 7946, 58981]
    assert wl.CE_LOGITS.B - wl.CE_LOGITS.n_ignored == 7782


def test_tiny_inputs_deterministic_and_shaped():
    a = wl.make_fused_inputs(wl.TINY)
    b = wl.make_fused_inputs(wl.TINY)
    assert wl.digest(a["hidden"], a["W"], a["target"]) == wl.digest(b["hidden"], b["W"], b["target"])
    assert a["hidden"].shape == (128, 64) and a["hidden"].dtype == np.uint16
    assert a["W"].shape == (512, 64) and a["bias"] is None
    t = a["target"]
    assert int((t == -100).sum()) == 6
    assert t[t != -100].min() >= 0 and t.max() < 512
    w = wl.bf16_bits_to_f32(a["W"])
    assert 0.017 < float(w.std()) < 0.023
    h = wl.bf16_bits_to_f32(a["hidden"])
    assert 0.9 < float(h.std()) < 1.1


def test_zipf_targets():
    w = wl.FusedWorkload("zipf probe", BT=20000, H=8, V=1000, targets="zipf", ignore_frac=0.03, bias_std=0.1)
    d = wl.make_fused_inputs(w)
    t = d["target"]
    v = t[t != -100]
    counts = np.bincount(v, minlength=1000)
    assert counts.argmax() == 0
    # P(0)/P(1) = 2^1.1
    assert 1.6 < counts[0] / counts[1] < 2.8
    assert d["bias"].dtype == np.float32 and d["bias"].shape == (1000,)


def test_ce_rows_reproducible_alone():
    w = wl.CEWorkload("ce probe", B=300, V=1000)
    full = wl.make_ce_inputs(w)
    part = wl.make_ce_inputs(w, rows=slice(70, 135))
    assert np.array_equal(full["logits"][70:135], part["logits"])
    assert np.array_equal(full["labels"][70:135], part["labels"])
    x = wl.bf16_bits_to_f32(full["logits"])
    assert 1.9 < float(x.std()) < 2.1
    assert int((full["labels"] == -100).sum()) == 15
