"""Fused linear cross-entropy (flce_fwd_bwd) against the fp64 oracle on the GPU, through the C ABI.

Element-by-element parity at sizes the oracle finishes in seconds (several tiles, ragged tails in
BT, V and H, bias, z-loss, both reductions, degenerate cases), and at the full benchmark sizes on
sampled outputs: the loss and n_valid, grad_input rows of sampled tokens and grad_W / grad_bias rows
of sampled vocabulary entries (stored by tests/golden/make_expected.py, which calls only the oracle),
each row checked on its own, the rows of untargeted vocabulary entries against the softmax part alone.
"""
import functools
import os

import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32, check_full_size_rows

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


def _upload(d):
    import torch
    hidden = bf16_tensor(d["hidden"])
    W = bf16_tensor(d["W"])
    target = torch.from_numpy(d["target"]).cuda()
    bias = torch.from_numpy(d["bias"]).cuda() if d.get("bias") is not None else None
    return hidden, W, target, bias


def _run(flce, d, **kw):
    import torch
    hidden, W, target, bias = _upload(d)
    out = flce.flce_fwd_bwd(hidden, W, target, bias=bias, ignore_index=d.get("ignore_index", -100),
                            reduction=d["reduction"], z_loss=d["z_loss"], **kw)
    torch.cuda.synchronize()
    out["status"] = flce.read_device_status(out["workspace"])
    return out


def _synthetic(BT, H, V, bias, z_loss, reduction, ignore=(), bad=(), seed=0, h_std=1.0, w_std=0.02):
    w = wl.FusedWorkload("case", BT=BT, H=H, V=V, hidden_std=h_std, w_std=w_std,
                         bias_std=0.1 if bias else None, ignore_frac=0.0, z_loss=z_loss, reduction=reduction,
                         seed=seed)
    d = wl.make_fused_inputs(w)
    for r in ignore:
        d["target"][r] = -100
    for r in bad:
        d["target"][r] = V + 5
    return d


def _check_full(out, d):
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction=d["reduction"],
                                z_loss=d["z_loss"])
    assert int(out["n_valid"].item()) == ref["n_valid"]
    assert_scalar_close(out["loss"].item(), ref["loss"], "loss")
    if out["grad_input"] is not None:
        assert_grad_close(bf16_to_numpy_f32(out["grad_input"]), ref["grad_input"], "grad_input")
    if out["grad_W"] is not None:
        assert_grad_close(out["grad_W"].cpu().numpy(), ref["grad_W"], "grad_W")
    if out["grad_bias"] is not None:
        assert_grad_close(out["grad_bias"].cpu().numpy(), ref["grad_bias"], "grad_bias")
    return ref


CASES = {
    # name: (BT, H, V, bias, z_loss, reduction, ignored rows)
    "one-tile": (128, 64, 256, False, 0.0, "mean", (5,)),
    "ragged-BT-V-bias-zloss": (300, 128, 1000, True, 1e-3, "mean", (0, 150, 299)),
    "two-H-chunks-sum": (257, 320, 777, False, 0.0, "sum", (256,)),
    "H-not-multiple-of-64": (64, 200, 300, True, 1e-2, "mean", ()),
    "wide-H-bias": (96, 576, 513, True, 1e-4, "mean", (1, 2)),
    "V-equals-1": (130, 64, 1, True, 1e-2, "sum", (3,)),
    "many-vocab-tiles": (40, 64, 5000, False, 0.0, "mean", ()),
    # fewer vocabulary blocks than pairs per cluster: pairs that own no block (two and three pairs)
    "one-block-two-pairs": (64, 512, 100, True, 1e-3, "mean", (3,)),
    "one-block-three-pairs": (70, 768, 200, False, 0.0, "sum", ()),
    # four pairs per cluster (H a multiple of 1024, at least 64 column blocks per unit): in the grad_input
    # pass (17000 / 256 = 67 vocabulary blocks), with two H groups (H = 2048), and in the grad_W pass
    # (16400 / 256 = 65 token blocks); the other pass of each case runs with two pairs
    "four-pairs-grad-input": (700, 1024, 17000, True, 1e-3, "mean", (0, 699)),
    "four-pairs-two-groups": (300, 2048, 16500, True, 1e-4, "mean", (7,)),
    "four-pairs-grad-W": (16400, 1024, 2100, False, 0.0, "sum", (5, 16399)),
}


FLOWS = {
    # the default: LSE inside the grad_input pass, vocabulary-split clusters where the plan puts them
    "online": {},
    # the same pass with every cluster over the whole vocabulary
    "online-whole-vocab": {"vocab_splits": 1},
    "separate-lse-pass": {"separate_lse_pass": True},
}


@pytest.mark.parametrize("flow", sorted(FLOWS))
@pytest.mark.parametrize("name", sorted(CASES))
def test_flce_matches_oracle(flce, name, flow):
    BT, H, V, bias, zl, red, ign = CASES[name]
    d = _synthetic(BT, H, V, bias, zl, red, ignore=ign, seed=BT * 7 + V)
    out = _run(flce, d, **FLOWS[flow])
    assert out["status"] == 0
    _check_full(out, d)
    if flow != "online":
        assert flce.read_vocab_split_units(out["workspace"]) == 0


# vocabulary-split clusters of the grad_input pass, forced: (BT, H, V, bias, z_loss, reduction, ignored rows,
# parts asked for).  Two and three pairs per cluster, ragged BT / V / H, parts of unequal length.
SPLIT_CASES = {
    "H1024-two-parts": (600, 1024, 9000, True, 1e-4, "mean", (0, 599), 2),
    "H1024-max-parts": (300, 1024, 12000, False, 0.0, "sum", (7,), 8),
    "H768-three-pairs": (260, 768, 5000, True, 1e-3, "mean", (1,), 3),
    "H200-one-pair-ragged": (513, 200, 4100, True, 0.0, "mean", (), 5),
    "H2304-three-groups": (100, 2304, 3333, False, 1e-4, "mean", (50,), 3),
    "H256-sixteen-parts": (300, 256, 20000, True, 1e-4, "mean", (3,), 16),
}


@pytest.mark.parametrize("name", sorted(SPLIT_CASES))
def test_flce_vocab_split_units(flce, name):
    BT, H, V, bias, zl, red, ign, k = SPLIT_CASES[name]
    d = _synthetic(BT, H, V, bias, zl, red, ignore=ign, seed=BT + V + k)
    out = _run(flce, d, vocab_splits=k)
    assert out["status"] == 0
    assert flce.read_vocab_split_units(out["workspace"]) > 0, "the pass did not split the vocabulary"
    _check_full(out, d)


# token-split clusters of the grad_W pass, forced: (BT, H, V, bias, z_loss, reduction, ignored rows, parts).
# Their partial rows live in the workspace's LSE-partials area (256 bytes per token), so BT must be large
# enough for two or three units' rows of P x 256 fp32 columns (and V at most 256: one row block).
DW_SPLIT_CASES = {
    "H256-one-pair": (4096, 256, 250, True, 1e-4, "mean", (5,), 3),
    "H512-two-pairs": (4500, 512, 200, True, 0.0, "sum", (), 2),
    "H768-three-pairs": (6200, 768, 250, False, 1e-3, "mean", (1, 6199), 2),
    "H2304-three-groups": (20000, 2304, 250, True, 1e-4, "mean", (7,), 2),
}


@pytest.mark.parametrize("name", sorted(DW_SPLIT_CASES))
def test_flce_token_split_units(flce, name):
    BT, H, V, bias, zl, red, ign, k = DW_SPLIT_CASES[name]
    d = _synthetic(BT, H, V, bias, zl, red, ignore=ign, seed=BT + V + 3 * k)
    out = _run(flce, d, token_splits=k)
    assert out["status"] == 0
    assert flce.read_token_split_units(out["workspace"]) > 0, "the grad_W pass did not split the tokens"
    _check_full(out, d)


def test_flce_token_split_classic_flow(flce):
    # without grad_input the call takes the classic flow: the LSE pass's partials occupy the scratch the
    # grad_W pass's split clusters reuse once the merge has read them
    BT, H, V, bias, zl, red, ign, k = DW_SPLIT_CASES["H512-two-pairs"]
    d = _synthetic(BT, H, V, bias, zl, red, ignore=ign, seed=BT + V + 1)
    out = _run(flce, d, token_splits=k, need_grad_input=False)
    assert out["status"] == 0
    assert flce.read_token_split_units(out["workspace"]) > 0
    assert out["grad_input"] is None
    _check_full(out, d)


def test_flce_token_split_accumulate_sorted(flce):
    # accumulation and the vocabulary sort's row permutation through the grad_W merge kernel
    import torch
    BT, H, V = 4096, 256, 250
    d = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(9,), seed=31)
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="mean", z_loss=1e-4)
    rng = np.random.Generator(np.random.PCG64(4))
    gw0 = (rng.standard_normal((V, H)) * np.std(ref["grad_W"])).astype(np.float32)
    gb0 = (rng.standard_normal(V) * np.std(ref["grad_bias"])).astype(np.float32)
    gi0 = wl.f32_to_bf16_bits((rng.standard_normal((BT, H)) * np.std(ref["grad_input"])).astype(np.float32))
    acc = {"grad_input": bf16_tensor(gi0), "grad_W": torch.from_numpy(gw0.copy()).cuda(),
           "grad_bias": torch.from_numpy(gb0.copy()).cuda()}
    out = _run(flce, d, token_splits=3, sort_vocab=True, accumulate=True, out=acc)
    assert out["status"] == 0
    assert flce.read_token_split_units(out["workspace"]) > 0
    assert_grad_close(out["grad_W"].cpu().numpy(), ref["grad_W"] + gw0, "grad_W (accumulated)")
    assert_grad_close(out["grad_bias"].cpu().numpy(), ref["grad_bias"] + gb0, "grad_bias (accumulated)")


def test_flce_vocab_split_options(flce):
    # per-token upstream gradients, per-token losses, entropy and accumulation through the merge kernel
    import torch
    BT, H, V = 400, 1024, 7000
    d = _synthetic(BT, H, V, True, 1e-4, "none", ignore=(3, 399), seed=77)
    rng = np.random.Generator(np.random.PCG64(9))
    gtok = rng.standard_normal(BT).astype(np.float32)
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="none", z_loss=1e-4,
                                grad_loss_per_token=gtok)
    gi0 = wl.f32_to_bf16_bits((rng.standard_normal((BT, H)) * np.std(ref["grad_input"])).astype(np.float32))
    gw0 = (rng.standard_normal((V, H)) * np.std(ref["grad_W"])).astype(np.float32)
    gb0 = (rng.standard_normal(V) * np.std(ref["grad_bias"])).astype(np.float32)
    acc = {"grad_input": bf16_tensor(gi0), "grad_W": torch.from_numpy(gw0.copy()).cuda(),
           "grad_bias": torch.from_numpy(gb0.copy()).cuda()}
    out = _run(flce, d, vocab_splits=4, grad_loss_per_token=torch.from_numpy(gtok).cuda(), want_entropy=True,
               accumulate=True, out=acc)
    assert out["status"] == 0
    assert flce.read_vocab_split_units(out["workspace"]) > 0
    assert_grad_close(out["loss_per_token"].cpu().numpy(), ref["loss_per_token"], "loss_per_token")
    assert_grad_close(out["entropy"].cpu().numpy(), ref["entropy"], "entropy")
    assert_grad_close(bf16_to_numpy_f32(out["grad_input"]),
                      ref["grad_input"] + (gi0.astype(np.uint32) << 16).view(np.float32), "grad_input (accumulated)")
    assert_grad_close(out["grad_W"].cpu().numpy(), ref["grad_W"] + gw0, "grad_W (accumulated)")
    assert_grad_close(out["grad_bias"].cpu().numpy(), ref["grad_bias"] + gb0, "grad_bias (accumulated)")


# Both passes with four pairs per cluster and at least three waves of row pairs (65 token and 66 vocabulary
# row pairs against 15 resident 8-CTA clusters): persistent four-pair clusters plus side clusters
# on the SMs they leave idle, which take the last row pairs one 256-wide H chunk at a time.
PERSISTENT_SHAPE = (16400, 1024, 16700)


def test_flce_persistent_with_side_clusters(flce):
    """Element by element against the oracle; the side launches counted; and bit for bit the same as one
    cluster per unit (the side pairs keep the four pairs' partial sums apart and add them in order)."""
    import torch
    BT, H, V = PERSISTENT_SHAPE
    d = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(0, BT - 1), seed=41)
    out = _run(flce, d)
    assert out["status"] == 0
    assert flce.read_side_launches(out["workspace"]) == 2
    assert flce.read_vocab_split_units(out["workspace"]) == 0
    assert flce.read_token_split_units(out["workspace"]) == 0
    _check_full(out, d)
    plain = _run(flce, d, vocab_splits=1, token_splits=1)
    assert plain["status"] == 0
    assert flce.read_side_launches(plain["workspace"]) == 0
    for k in ("grad_input", "grad_W", "grad_bias"):
        assert torch.equal(out[k], plain[k]), f"{k} differs from one cluster per unit"
    assert out["loss"].item() == plain["loss"].item()


def test_flce_persistent_with_side_clusters_sorted_vocab(flce):
    # the vocabulary sort (its row permutation applied by the grad_W pass's epilogue) with both passes
    # persistent and side clusters: against the oracle, and bit for bit against the sorted call with one
    # cluster per unit
    import torch
    BT, H, V = PERSISTENT_SHAPE
    d = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(5,), seed=53)
    out = _run(flce, d, sort_vocab=True)
    assert out["status"] == 0
    assert flce.read_side_launches(out["workspace"]) == 2
    _check_full(out, d)
    plain = _run(flce, d, sort_vocab=True, vocab_splits=1, token_splits=1)
    assert plain["status"] == 0 and flce.read_side_launches(plain["workspace"]) == 0
    for k in ("grad_input", "grad_W", "grad_bias"):
        assert torch.equal(out[k], plain[k]), f"{k} differs from one cluster per unit"


def test_flce_short_units_four_pairs_with_side_clusters(flce):
    """A grad_W pass of short units (17 token blocks, under the 64 that four pairs otherwise need) with
    enough vocabulary row pairs (118: more than the 75 above the main clusters' that the single-pair
    clusters keep in reserve, beside 15 resident 8-CTA clusters) runs four pairs per cluster, persistent,
    with side and single-pair clusters: against the oracle, and against the same pass with one two-pair
    cluster per unit (the grad_input pass unsplit in both, so that both grad_W passes read the same
    statistics)."""
    import torch
    BT, H, V = 4100, 1024, 30000
    d = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(1, BT - 1), seed=47)
    out = _run(flce, d, vocab_splits=1)
    assert out["status"] == 0
    assert flce.read_side_launches(out["workspace"]) == 1, "the grad_W pass did not run with side clusters"
    assert flce.read_single_launches(out["workspace"]) == 1
    assert flce.read_single_units(out["workspace"])[1] > 0, "the single-pair clusters took no unit"
    _check_full(out, d)
    plain = _run(flce, d, vocab_splits=1, token_splits=1)
    assert plain["status"] == 0 and flce.read_side_launches(plain["workspace"]) == 0
    assert torch.equal(out["grad_input"], plain["grad_input"])
    # (four pairs against two: the same GEMM1 K order and GEMM2 block order; grad_bias adds the pairs'
    # partial sums in another grouping, so it is compared within the parity bound)
    assert torch.equal(out["grad_W"], plain["grad_W"])
    assert_grad_close(out["grad_bias"].cpu().numpy(), plain["grad_bias"].cpu().numpy().astype(np.float64), "grad_bias")


def test_flce_single_pair_clusters_grad_W(flce):
    """The grad_W pass with enough vocabulary row pairs (102) for the single-pair clusters to take units
    (each a row pair's two H chunks, one at a time, keeping the four pairs' owner-class sums apart): against
    the oracle element by element, and bit for bit against one four-pair cluster per unit (65 token
    blocks, so that the one-unit run has four pairs per cluster too).  The grad_input pass runs with side
    clusters only."""
    import torch
    BT, H, V = 16400, 1024, 26000
    d = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(2, BT - 2), seed=59)
    out = _run(flce, d)
    assert out["status"] == 0
    assert flce.read_side_launches(out["workspace"]) == 2 and flce.read_single_launches(out["workspace"]) == 1
    units = flce.read_single_units(out["workspace"])
    assert units[0] == 0 and units[1] > 0, f"single-pair units per pass: {units}"
    assert flce.read_single_clusters(out["workspace"]) > 0
    _check_full(out, d)
    plain = _run(flce, d, vocab_splits=1, token_splits=1)
    assert plain["status"] == 0 and flce.read_single_launches(plain["workspace"]) == 0
    for k in ("grad_input", "grad_W", "grad_bias"):
        assert torch.equal(out[k], plain[k]), f"{k} differs from one cluster per unit"
    assert out["loss"].item() == plain["loss"].item()


def test_flce_persistent_side_clusters_options(flce):
    # per-token upstream gradients and losses, entropy (the owner-class sums of the side pairs) and
    # accumulation, with the side clusters
    import torch
    BT, H, V = PERSISTENT_SHAPE
    d = _synthetic(BT, H, V, True, 1e-3, "none", ignore=(11,), seed=43)
    rng = np.random.Generator(np.random.PCG64(17))
    gtok = rng.standard_normal(BT).astype(np.float32)
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="none", z_loss=1e-3,
                                grad_loss_per_token=gtok)
    gi0 = wl.f32_to_bf16_bits((rng.standard_normal((BT, H)) * np.std(ref["grad_input"])).astype(np.float32))
    gw0 = (rng.standard_normal((V, H)) * np.std(ref["grad_W"])).astype(np.float32)
    gb0 = (rng.standard_normal(V) * np.std(ref["grad_bias"])).astype(np.float32)
    acc = {"grad_input": bf16_tensor(gi0), "grad_W": torch.from_numpy(gw0.copy()).cuda(),
           "grad_bias": torch.from_numpy(gb0.copy()).cuda()}
    out = _run(flce, d, grad_loss_per_token=torch.from_numpy(gtok).cuda(), want_entropy=True, accumulate=True, out=acc)
    assert out["status"] == 0
    assert flce.read_side_launches(out["workspace"]) == 2
    assert_grad_close(out["loss_per_token"].cpu().numpy(), ref["loss_per_token"], "loss_per_token")
    assert_grad_close(out["entropy"].cpu().numpy(), ref["entropy"], "entropy")
    assert_grad_close(bf16_to_numpy_f32(out["grad_input"]),
                      ref["grad_input"] + (gi0.astype(np.uint32) << 16).view(np.float32), "grad_input (accumulated)")
    assert_grad_close(out["grad_W"].cpu().numpy(), ref["grad_W"] + gw0, "grad_W (accumulated)")
    assert_grad_close(out["grad_bias"].cpu().numpy(), ref["grad_bias"] + gb0, "grad_bias (accumulated)")


def test_flce_tiny_workload(flce):
    d = wl.make_fused_inputs(wl.TINY)
    out = _run(flce, d)
    assert out["status"] == 0
    ref = _check_full(out, d)
    assert ref["n_valid"] == 122


@pytest.mark.parametrize("separate_lse", [False, True], ids=["lse-in-grad-input-pass", "separate-lse-pass"])
def test_flce_peaked_logits(flce, separate_lse):
    # logits std ~8: the online max matters and the softmax is far from uniform
    d = _synthetic(200, 256, 3000, True, 1e-4, "mean", ignore=(7,), seed=3, w_std=0.5)
    out = _run(flce, d, separate_lse_pass=separate_lse)
    _check_full(out, d)


def test_flce_confident_rows(flce):
    # rows whose target holds almost all of the probability (p_y near 1): grad_input is a small difference
    # (p_y f - 1) W_y + ...; the online pass adds the target term exactly at the end
    d = _synthetic(260, 512, 2000, False, 0.0, "sum", ignore=(3,), seed=23, w_std=0.02)
    W = oracle.widen(d["W"])
    h = oracle.widen(d["hidden"])
    for r in range(0, 260, 2):   # make half of the rows confident: hidden aligned with its target's W row
        y = int(d["target"][r])
        if y >= 0:
            v = (W[y] / np.linalg.norm(W[y]) * 40.0).astype(np.float32)
            d["hidden"][r] = wl.f32_to_bf16_bits(v)
    out = _run(flce, d)
    assert out["status"] == 0
    _check_full(out, d)


def test_flce_all_ignored(flce):
    d = _synthetic(150, 64, 700, True, 1e-3, "mean", ignore=range(150))
    out = _run(flce, d)
    assert int(out["n_valid"].item()) == 0 and out["loss"].item() == 0.0
    assert np.all(bf16_to_numpy_f32(out["grad_input"]) == 0.0)
    assert np.all(out["grad_W"].cpu().numpy() == 0.0)
    assert np.all(out["grad_bias"].cpu().numpy() == 0.0)


def test_flce_empty_batch(flce):
    import torch
    W = torch.randn(300, 64, device="cuda").to(torch.bfloat16)
    hidden = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    target = torch.empty((0,), dtype=torch.int64, device="cuda")
    bias = torch.randn(300, device="cuda")
    out = flce.flce_fwd_bwd(hidden, W, target, bias=bias)
    torch.cuda.synchronize()
    assert out["loss"].item() == 0.0 and out["n_valid"].item() == 0
    assert torch.count_nonzero(out["grad_W"]).item() == 0 and torch.count_nonzero(out["grad_bias"]).item() == 0


def test_flce_bad_targets_flagged_and_ignored(flce):
    d = _synthetic(140, 64, 400, False, 0.0, "mean", ignore=(2,), bad=(9, 130))
    out = _run(flce, d)
    assert out["status"] & flce.STATUS_BAD_TARGET
    ref = _check_full(out, d)
    assert ref["n_valid"] == 137


def test_flce_output_subsets(flce):
    d = _synthetic(160, 128, 900, True, 1e-3, "mean", ignore=(4,), seed=11)
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], z_loss=1e-3)
    only_gi = _run(flce, d, need_grad_W=False)
    assert only_gi["grad_W"] is None and only_gi["grad_bias"] is None
    assert_scalar_close(only_gi["loss"].item(), ref["loss"], "loss")
    assert_grad_close(bf16_to_numpy_f32(only_gi["grad_input"]), ref["grad_input"], "grad_input")
    only_gw = _run(flce, d, need_grad_input=False)
    assert only_gw["grad_input"] is None
    assert_grad_close(only_gw["grad_W"].cpu().numpy(), ref["grad_W"], "grad_W")
    assert_grad_close(only_gw["grad_bias"].cpu().numpy(), ref["grad_bias"], "grad_bias")
    # grad_bias alone (grad_W NULL) goes through the C ABI directly
    import torch
    from linear_cross_entropy_tma_gb300 import _lib
    hidden, W, target, bias = _upload(d)
    loss = torch.empty(1, device="cuda")
    gb = torch.empty(900, device="cuda")
    ws = torch.empty(_lib.workspace_size(160, 128, 900), dtype=torch.uint8, device="cuda")
    _lib.check(_lib.load().flce_fwd_bwd(hidden.data_ptr(), W.data_ptr(), bias.data_ptr(), target.data_ptr(), 160, 128,
                                        900, -100, 0, 1e-3, loss.data_ptr(), None, None, gb.data_ptr(), None,
                                        ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert_grad_close(gb.cpu().numpy(), ref["grad_bias"], "grad_bias only")


def _fallback_flag(ws) -> int:
    # word 6 of the workspace header: set when the grad_input pass that finds the LSE itself handed the
    # call to the classic passes
    return int(ws[24:28].cpu().view(__import__("torch").int32).item())


@pytest.mark.parametrize("H", [128, 512])
def test_flce_online_fallback(flce, H):
    # a bias of -200 on the first 128 columns puts every row's reference far below its other logits: the
    # sums overflow the online pass's safe range, and the classic passes must produce the exact result
    d = _synthetic(260, H, 1200, True, 1e-4, "mean", ignore=(1, 200), seed=17)
    d["bias"] = d["bias"].copy()
    d["bias"][:128] = -200.0
    d["target"][d["target"] < 128] = 300
    out = _run(flce, d)
    assert out["status"] == 0
    assert _fallback_flag(out["workspace"]) == 1
    _check_full(out, d)
    # the same with accumulation: rows the online pass left are written once, by the classic pass
    import torch
    rng = np.random.Generator(np.random.PCG64(5))
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], reduction="mean", z_loss=1e-4)
    gi0 = wl.f32_to_bf16_bits((rng.standard_normal((260, H)) * np.std(ref["grad_input"])).astype(np.float32))
    gw0 = (rng.standard_normal((1200, H)) * np.std(ref["grad_W"])).astype(np.float32)
    gb0 = (rng.standard_normal(1200) * np.std(ref["grad_bias"])).astype(np.float32)
    acc = {"grad_input": bf16_tensor(gi0), "grad_W": torch.from_numpy(gw0.copy()).cuda(),
           "grad_bias": torch.from_numpy(gb0.copy()).cuda()}
    out3 = _run(flce, d, accumulate=True, out=acc)
    assert out3["status"] == 0 and _fallback_flag(out3["workspace"]) == 1
    assert_grad_close(bf16_to_numpy_f32(out3["grad_input"]),
                      ref["grad_input"] + (gi0.astype(np.uint32) << 16).view(np.float32), "grad_input (accumulated)")
    assert_grad_close(out3["grad_W"].cpu().numpy(), ref["grad_W"] + gw0, "grad_W (accumulated)")
    assert_grad_close(out3["grad_bias"].cpu().numpy(), ref["grad_bias"] + gb0, "grad_bias (accumulated)")
    # and ordinary inputs stay on the online pass
    d2 = _synthetic(260, H, 1200, True, 1e-4, "mean", ignore=(1, 200), seed=18)
    out2 = _run(flce, d2)
    assert _fallback_flag(out2["workspace"]) == 0
    _check_full(out2, d2)


def test_flce_online_fallback_vocab_split(flce):
    # as above, with the vocabulary split: only the part whose reference comes from the -200 columns leaves
    # the safe range, and its rows go to the classic passes
    d = _synthetic(260, 512, 3000, True, 1e-4, "mean", ignore=(1, 200), seed=19)
    d["bias"] = d["bias"].copy()
    d["bias"][:128] = -200.0
    d["target"][d["target"] < 128] = 300
    out = _run(flce, d, vocab_splits=3)
    assert out["status"] == 0
    assert flce.read_vocab_split_units(out["workspace"]) > 0
    assert _fallback_flag(out["workspace"]) == 1
    _check_full(out, d)


@pytest.mark.parametrize("shape", [(600, 1024, 9000), (128, 64, 512), (16400, 1024, 16700)])
def test_flce_cuda_graph_replay(flce, shape):
    # the call captures into a CUDA graph (no host synchronisation, no allocation inside): a replay gives
    # the eager call's results bit for bit, and replays on new inputs in the same buffers match the oracle
    import torch
    from linear_cross_entropy_tma_gb300 import _lib
    BT, H, V = shape
    d = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(0,), seed=5)
    hidden, W, target, bias = _upload(d)
    ws = torch.empty(_lib.workspace_size(BT, H, V), dtype=torch.uint8, device="cuda")
    out = {"loss": torch.empty(1, device="cuda"), "n_valid": torch.empty(1, dtype=torch.int64, device="cuda"),
           "grad_input": torch.empty((BT, H), dtype=torch.bfloat16, device="cuda"),
           "grad_W": torch.empty((V, H), device="cuda"), "grad_bias": torch.empty(V, device="cuda")}
    kw = dict(bias=bias, z_loss=1e-4, workspace=ws, out=out)
    flce.flce_fwd_bwd(hidden, W, target, **kw)   # (one-time queries run outside the capture)
    torch.cuda.synchronize()
    eager = {k: v.clone() for k, v in out.items()}
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        flce.flce_fwd_bwd(hidden, W, target, **kw)
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert flce.read_device_status(ws) == 0
    if shape == PERSISTENT_SHAPE:
        # the side launches (programmatic dependent launch) are part of the graph
        assert flce.read_side_launches(ws) == 2
    for k in out:
        assert torch.equal(out[k], eager[k]), f"graph replay differs from the eager call in {k}"
    d2 = _synthetic(BT, H, V, True, 1e-4, "mean", ignore=(1, BT - 1), seed=6)
    h2, w2, t2, b2 = _upload(d2)
    hidden.copy_(h2)
    W.copy_(w2)
    target.copy_(t2)
    bias.copy_(b2)
    g.replay()
    torch.cuda.synchronize()
    assert flce.read_device_status(ws) == 0
    _check_full(dict(loss=out["loss"], n_valid=out["n_valid"], grad_input=out["grad_input"], grad_W=out["grad_W"],
                     grad_bias=out["grad_bias"]), d2)


def test_flce_cuda_graph_capture_of_the_first_call(flce):
    # in a fresh process the very first call is the captured one (its one-time occupancy queries are then
    # skipped, not made inside the capture): the replay must match an eager call made afterwards
    import subprocess
    import sys
    code = r"""
import sys, torch
sys.path.insert(0, %r)
import linear_cross_entropy_tma_gb300 as flce
from linear_cross_entropy_tma_gb300 import _lib
torch.manual_seed(0)
BT, H, V = 1000, 1024, 9000
h = torch.randn(BT, H, device="cuda").bfloat16()
W = (torch.randn(V, H, device="cuda") * 0.02).bfloat16()
t = torch.randint(0, V, (BT,), device="cuda")
ws = torch.empty(_lib.workspace_size(BT, H, V), dtype=torch.uint8, device="cuda")
out = {"loss": torch.empty(1, device="cuda"), "grad_input": torch.empty((BT, H), dtype=torch.bfloat16, device="cuda"),
       "grad_W": torch.empty((V, H), device="cuda")}
g = torch.cuda.CUDAGraph()
with torch.cuda.graph(g):
    flce.flce_fwd_bwd(h, W, t, workspace=ws, out=out)
g.replay()
torch.cuda.synchronize()
assert flce.read_device_status(ws) == 0
first = {k: v.clone() for k, v in out.items()}
r = flce.flce_fwd_bwd(h, W, t)   # eager, with the queries (and possibly a split plan) this time
torch.cuda.synchronize()
assert abs(r["loss"].item() - first["loss"].item()) <= 2e-4 * abs(first["loss"].item())
for k in ("grad_input", "grad_W"):
    a, b = first[k].float(), r[k].float()
    assert ((a - b).norm() / b.norm()).item() < 5e-3, k
print("ok")
""" % (os.path.dirname(os.path.dirname(os.path.abspath(__file__))),)
    p = subprocess.run([sys.executable, "-c", code], capture_output=True, text=True, timeout=600)
    assert p.returncode == 0 and p.stdout.strip().endswith("ok"), p.stdout + p.stderr


def test_flce_grad_input_and_bias_without_grad_W(flce):
    # grad_W NULL with a bias: the grad_W pass covers one H chunk (one pair per cluster) while the
    # grad_input pass at H = 512 has two, so the two passes run as separate launches
    import torch
    from linear_cross_entropy_tma_gb300 import _lib
    d = _synthetic(300, 512, 1500, True, 1e-4, "mean", ignore=(5, 299), seed=13)
    ref = oracle.flce_reference(d["hidden"], d["W"], d["target"], bias=d["bias"], z_loss=1e-4)
    hidden, W, target, bias = _upload(d)
    loss = torch.empty(1, device="cuda")
    gi = torch.empty((300, 512), dtype=torch.bfloat16, device="cuda")
    gb = torch.empty(1500, device="cuda")
    ws = torch.empty(_lib.workspace_size(300, 512, 1500), dtype=torch.uint8, device="cuda")
    _lib.check(_lib.load().flce_fwd_bwd(hidden.data_ptr(), W.data_ptr(), bias.data_ptr(), target.data_ptr(), 300, 512,
                                        1500, -100, 0, 1e-4, loss.data_ptr(), gi.data_ptr(), None, gb.data_ptr(), None,
                                        ws.data_ptr(), ws.numel(), torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    assert flce.read_device_status(ws) == 0
    assert_scalar_close(loss.item(), ref["loss"], "loss")
    assert_grad_close(bf16_to_numpy_f32(gi), ref["grad_input"], "grad_input")
    assert_grad_close(gb.cpu().numpy(), ref["grad_bias"], "grad_bias")


@functools.lru_cache(maxsize=1)
def _full_inputs(key):
    return wl.make_fused_inputs(wl.FUSED_WORKLOADS[key])


@pytest.mark.parametrize("key", ["qwen3", "gemma2", "long"])
def test_flce_full_size_sampled(flce, key):
    import torch
    w = wl.FUSED_WORKLOADS[key]
    exp = np.load(os.path.join(GOLDEN, f"expected_{key}.npz"))
    d = _full_inputs(key)
    assert wl.digest(d["hidden"], d["W"], d["bias"], d["target"]) == str(exp["digest"]), "input generator drifted"
    out = _run(flce, d)
    assert out["status"] == 0
    assert int(out["n_valid"].item()) == int(exp["n_valid"]) == w.n_valid
    assert_scalar_close(out["loss"].item(), float(exp["loss"]), "loss")
    # the grad_input pass's last row blocks ran as an automatic split tail or, where the pass has four pairs
    # per cluster and enough waves, on the side clusters beside the persistent ones (the sample holds
    # tokens and vocabulary entries among the last 512, where either form works)
    side = flce.read_side_launches(out["workspace"])
    assert flce.read_vocab_split_units(out["workspace"]) > 0 or side > 0
    if key == "long":
        assert side == 2, "both passes of the long workload run with side clusters beside"
        assert flce.read_single_launches(out["workspace"]) == 1, "the grad_W pass launches single-pair clusters"
        assert flce.read_single_units(out["workspace"])[1] > 0, "the single-pair clusters took no unit"
    rows = torch.from_numpy(exp["rows"]).cuda()
    vr = torch.from_numpy(exp["vocab_rows"]).cuda()
    check_full_size_rows(exp, bf16_to_numpy_f32(out["grad_input"][rows]), out["grad_W"][vr].cpu().numpy(),
                         out["grad_bias"][vr].cpu().numpy() if "grad_bias_rows" in exp.files else None)
    # no (BT, V) buffer: the workspace is O(BT)
    assert out["workspace"].numel() < 64 * 2**20
    first = out["loss"].item()
    del out
    again = _run(flce, d, need_grad_input=False, need_grad_W=False)
    assert again["loss"].item() == first, "loss is not deterministic"


@pytest.mark.parametrize("key", ["qwen3", "gemma2", "long"])
def test_flce_full_size_split_tails(flce, key):
    """The automatic scheduling at the full sizes (split tails, or side clusters beside persistent
    four-pair clusters): every row of the last row pairs (grad_input) and every vocabulary row of the last
    vocabulary row pairs (grad_W, grad_bias) against the same call with one cluster per unit and no
    splitting (whose rows the sampled test above checks against the oracle), within the parity bounds."""
    import torch
    d = _full_inputs(key)
    a = _run(flce, d)
    assert a["status"] == 0
    vs, side = flce.read_vocab_split_units(a["workspace"]), flce.read_side_launches(a["workspace"])
    assert vs > 0 or side > 0, "the grad_input pass neither split its last wave nor ran side clusters"
    b = _run(flce, d, vocab_splits=1, token_splits=1)
    assert b["status"] == 0
    assert flce.read_vocab_split_units(b["workspace"]) == 0 and flce.read_token_split_units(b["workspace"]) == 0
    assert flce.read_side_launches(b["workspace"]) == 0
    assert_scalar_close(a["loss"].item(), b["loss"].item(), "loss")
    w = wl.FUSED_WORKLOADS[key]
    # a pass that ran persistent with side clusters (no split units) gives the one-cluster-per-unit result
    # bit for bit; the grad_W pass only when the grad_input pass did not split either (its per-token
    # statistics, which every grad_W row sums over, carry the split tail's rounding)
    ts = flce.read_token_split_units(a["workspace"])
    if side > 0 and vs == 0:
        assert torch.equal(a["grad_input"], b["grad_input"]) and a["loss"].item() == b["loss"].item()
        if ts == 0:
            assert torch.equal(a["grad_W"], b["grad_W"])
            if a["grad_bias"] is not None:
                assert torch.equal(a["grad_bias"], b["grad_bias"])
    # the split row pairs are the last ones (at qwen3 all 16, split unevenly); compare the last 4096 rows
    # and the last 1280 vocabulary rows (5 vocabulary row pairs)
    r0 = max(0, w.BT - 4096)
    assert_grad_close(bf16_to_numpy_f32(a["grad_input"][r0:]), bf16_to_numpy_f32(b["grad_input"][r0:]).astype(np.float64),
                      "grad_input (split rows)")
    v0 = max(0, w.V - 1280)
    assert_grad_close(a["grad_W"][v0:].cpu().numpy(), b["grad_W"][v0:].cpu().numpy().astype(np.float64),
                      "grad_W (split vocabulary rows)")
    if a["grad_bias"] is not None:
        assert_grad_close(a["grad_bias"][v0:].cpu().numpy(), b["grad_bias"][v0:].cpu().numpy().astype(np.float64),
                          "grad_bias (split vocabulary rows)")

