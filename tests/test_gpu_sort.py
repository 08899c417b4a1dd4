"""The vocabulary sort ("Cut Cross Entropy visualized", "Vocabulary Sorting", keyed by the logit_avg of
"Forward pass") against the fp64 oracle on the GPU, through the C ABI.

  * logit_avg: within 1e-4 of sum_k |W[n, k]| |mean hidden_k| + |b_n| per entry (fp32 column sums of
    hidden and an fp32 dot product per row, against the oracle's fp64 mean of the logits);
  * the order: bit for bit the stable descending sort of the kernel's own fp32 logit_avg values (the
    order is a decision taken in the kernel's precision), ties included;
  * the sorted exact path: loss, n_valid, grad_input, grad_W and grad_bias (in the caller's vocabulary
    order) under the usual bars, with an ignore_index inside [0, V) and an out-of-range target;
  * with gradient filtering: a vocabulary whose high-probability entries are scattered skips almost no
    block unsorted and most blocks sorted, and the sorted result stays within the filter's bound.
"""
import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import (assert_grad_close, assert_scalar_close, assert_within_bound, bf16_tensor, bf16_to_numpy_f32)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def flce():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    import linear_cross_entropy_tma_gb300 as m
    m.load()
    return m


def _upload(hidden, W, target, bias):
    import torch
    return (bf16_tensor(hidden), bf16_tensor(W), torch.from_numpy(target).cuda(),
            torch.from_numpy(bias).cuda() if bias is not None else None)


def _case(BT, H, V, seed, bias_std=0.1):
    w = wl.FusedWorkload("sort", BT=BT, H=H, V=V, hidden_std=1.0, w_std=0.05, bias_std=bias_std, ignore_frac=0.0,
                         seed=seed)
    d = wl.make_fused_inputs(w)
    return d["hidden"], d["W"], d["target"], d["bias"]


def _expected_order(avg_f32: np.ndarray) -> np.ndarray:
    a = np.where(avg_f32 == 0.0, np.float32(0.0), avg_f32)   # -0 and +0 are one key
    return np.argsort(-a, kind="stable")


@pytest.mark.parametrize("shape", [(520, 512, 3000), (300, 128, 1000), (37, 64, 20000), (64, 64, 100003)])
def test_logit_avg_and_order(flce, shape):
    import torch
    BT, H, V = shape
    hidden, W, target, bias = _case(BT, H, V, seed=BT + V)
    # duplicated vocabulary rows with equal bias: exact ties in the key, which must keep index order
    for r in (10, V // 2, V - 1):
        W[r] = W[3]
        bias[r] = bias[3]
    h, w_, t, b = _upload(hidden, W, target, bias)
    out = flce.flce_fwd_bwd(h, w_, t, bias=b, sort_vocab=True, need_grad_input=False, need_grad_W=False)
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == 0
    got = out["logit_avg"].cpu().numpy()
    ref = oracle.logit_avg(hidden, W, bias=bias)
    hbar = np.abs(oracle.widen(hidden).mean(axis=0))
    scale = np.abs(oracle.widen(W)) @ hbar + np.abs(bias.astype(np.float64))
    assert np.all(np.abs(got - ref) <= 1e-4 * scale + 1e-30), float(np.max(np.abs(got - ref) / scale))
    order = out["vocab_order"].cpu().numpy().astype(np.int64)
    assert np.array_equal(order, _expected_order(got))
    tie = [int(np.nonzero(order == r)[0][0]) for r in (3, 10, V // 2, V - 1)]
    assert tie == sorted(tie) and tie[-1] - tie[0] == 3, "equal keys must sit together in index order"
    # and the oracle's own order agrees wherever the keys are not within rounding of each other
    ro = oracle.vocab_order(ref)
    gap = np.abs(np.diff(ref[ro]))
    sep = np.concatenate([[np.inf], gap]) > 1e-3 * np.max(scale)
    sep &= np.concatenate([gap, [np.inf]]) > 1e-3 * np.max(scale)
    assert np.array_equal(order[sep], ro[sep])


@pytest.mark.parametrize("shape", [(300, 128, 1000), (260, 512, 3000)])
def test_sorted_exact_path(flce, shape):
    import torch
    BT, H, V = shape
    hidden, W, target, bias = _case(BT, H, V, seed=3 * BT + H)
    ignore = 7
    target[[0, 5, 77]] = ignore          # an ignore_index inside [0, V)
    target[11] = V + 5                   # out of range: ignored, with the status bit
    h, w_, t, b = _upload(hidden, W, target, bias)
    out = flce.flce_fwd_bwd(h, w_, t, bias=b, ignore_index=ignore, z_loss=1e-4, sort_vocab=True, want_entropy=True)
    torch.cuda.synchronize()
    assert flce.read_device_status(out["workspace"]) == flce.STATUS_BAD_TARGET
    ref = oracle.flce_reference(hidden, W, target, bias=bias, ignore_index=ignore, z_loss=1e-4)
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(out["loss"].item(), ref["loss"], "loss")
    assert_grad_close(bf16_to_numpy_f32(out["grad_input"]), ref["grad_input"], "grad_input")
    assert_grad_close(out["grad_W"].cpu().numpy(), ref["grad_W"], "grad_W")
    assert_grad_close(out["grad_bias"].cpu().numpy(), ref["grad_bias"], "grad_bias")
    ent = out["entropy"].cpu().numpy().astype(np.float64)
    assert np.all(np.abs(ent - ref["entropy"]) <= 2e-4 * np.maximum(1.0, ref["lse"]))


def _popular_case(BT, H, V, n_pop, seed):
    # a few vocabulary entries carry almost all of the probability (bias +12) and every target is one of
    # them: the kind of vocabulary the sort is for; the popular entries are scattered over all blocks
    rng = np.random.Generator(np.random.PCG64(seed))
    hidden = wl.f32_to_bf16_bits(rng.standard_normal((BT, H), dtype=np.float32))
    W = wl.f32_to_bf16_bits((0.02 * rng.standard_normal((V, H))).astype(np.float32))
    pop = rng.choice(V, n_pop, replace=False)
    bias = np.zeros(V, dtype=np.float32)
    bias[pop] = 12.0
    target = pop[rng.integers(0, n_pop, BT)].astype(np.int64)
    target[[3, 100]] = -100
    return hidden, W, target, bias


def test_sort_raises_filter_skips(flce):
    import torch
    BT, H, V, eps = 520, 512, 4096, 2.0 ** -12
    hidden, W, target, bias = _popular_case(BT, H, V, 64, seed=41)
    h, w_, t, b = _upload(hidden, W, target, bias)
    # (the separate LSE pass keeps both gradient passes filtering; by default only the grad_W pass does)
    plain = flce.flce_fwd_bwd(h, w_, t, bias=b, filter_eps=eps, separate_lse_pass=True)
    srt = flce.flce_fwd_bwd(h, w_, t, bias=b, filter_eps=eps, sort_vocab=True, separate_lse_pass=True)
    torch.cuda.synchronize()
    assert flce.read_device_status(srt["workspace"]) == 0
    skips_plain = flce.read_filter_skips(plain["workspace"])
    skips_sorted = flce.read_filter_skips(srt["workspace"])
    # 3 row pairs x 32 column halves in the grad_input pass and 16 x 6 in the grad_W pass: unsorted
    # nearly every half holds a popular entry, sorted only the first ones do
    assert skips_sorted >= 200 and skips_sorted > 3 * max(skips_plain, 1), (skips_plain, skips_sorted)
    assert set(srt["vocab_order"][:64].cpu().numpy().tolist()) == set(np.nonzero(bias)[0].tolist())
    ref = oracle.flce_reference(hidden, W, target, bias=bias)
    dS = oracle.flce_dlogits(hidden, W, target, bias=bias)
    valid = (target >= 0) & (target < V)
    s_w = valid / max(int(valid.sum()), 1)
    unscaled = np.divide(np.abs(dS), s_w[:, None], out=np.zeros_like(dS), where=s_w[:, None] > 0)
    small = np.where(unscaled <= eps * (1.0 + 1.0 / 64), np.abs(dS), 0.0)
    assert int(srt["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(srt["loss"].item(), ref["loss"], "loss")
    assert_within_bound(bf16_to_numpy_f32(srt["grad_input"]), ref["grad_input"], small @ np.abs(oracle.widen(W)),
                        "grad_input")
    assert_within_bound(srt["grad_W"].cpu().numpy(), ref["grad_W"], small.T @ np.abs(oracle.widen(hidden)), "grad_W")
    assert_grad_close(srt["grad_bias"].cpu().numpy(), ref["grad_bias"], "grad_bias")
