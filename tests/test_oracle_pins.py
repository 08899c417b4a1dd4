"""Pins for the CPU oracle: each check ties it to something other than itself.

  * brute force: the element-by-element loop version of the same definitions;
  * calculus: central finite differences of the loss against the analytic gradients
    (the boxed identity dl/dz = softmax - onehot of "Fused Linear Cross-Entropy", "The identity ...");
  * an independent library: torch.nn.functional.cross_entropy in float64 on the CPU, with autograd;
  * closed forms: W = 0, V = 1, and the hand-evaluated values in tests/golden/ce_closed_forms.txt;
  * invariants: LSE shift, dlogits row sums, ignored rows, n_valid = 0, vocabulary permutation;
  * the unreduced loss with an upstream gradient against finite differences and torch autograd;
  * the per-row entropy against torch, plain loops, closed forms and its bounds;
  * the average logit per vocabulary entry against loops, closed forms and the linearity identity, and
    the vocabulary order against a hand-evaluated case and brute force;
  * the widening of bf16 bit patterns against hand-evaluated values (zeros, subnormals, infinities, the
    largest finite values) and torch's bfloat16 decoding of all 65536 patterns, and the loss and
    gradients from bit patterns against torch.

The same checks run against deliberately broken copies of the oracle (test_planted_mistakes) to show
that a dropped term, a wrong sign, a wrong index or a wrong scale fails at least one of them.
"""
from __future__ import annotations

import math
import os
import types

import numpy as np
import pytest
import torch

import oracle.flce_oracle as ORACLE

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rel(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    scale = max(float(np.max(np.abs(b))) if b.size else 0.0, 1e-300)
    return float(np.max(np.abs(a - b))) / scale if b.size else 0.0


def _tiny_case(seed=1, BT=6, H=5, V=7, bias=True, ignore_rows=(2,), logit_scale=1.0):
    rng = np.random.default_rng(seed)
    hidden = rng.standard_normal((BT, H)) * logit_scale
    W = rng.standard_normal((V, H))
    b = rng.standard_normal(V) if bias else None
    t = rng.integers(0, V, BT)
    for r in ignore_rows:
        t[r] = -100
    return hidden, W, b, t


# ----------------------------------------------------------------------------- pins (parameterised
# by the oracle module so that planted-mistake copies can be run through them)

def pin_loops_vs_vectorised(orc):
    for reduction in ("mean", "sum"):
        for zl in (0.0, 1e-2):
            hidden, W, b, t = _tiny_case()
            ref = orc.flce_reference_loops(hidden, W, t, bias=b, reduction=reduction, z_loss=zl)
            got = orc.flce_reference(hidden, W, t, bias=b, reduction=reduction, z_loss=zl, row_block=4)
            assert abs(got["loss"] - ref["loss"]) <= 1e-12 * abs(ref["loss"])
            assert got["n_valid"] == ref["n_valid"]
            for k in ("grad_input", "grad_W", "grad_bias", "lse"):
                assert _rel(got[k], ref[k]) < 1e-12, k


def pin_finite_differences(orc):
    h_step = 1e-6
    for reduction, zl in (("mean", 1e-2), ("sum", 0.0), ("mean", 0.0)):
        hidden, W, b, t = _tiny_case(seed=3)
        t[4] = 11  # out of range: read as ignored
        g = orc.flce_reference(hidden, W, t, bias=b, reduction=reduction, z_loss=zl, row_block=4)

        def loss_at(hh, ww, bb):
            return orc.flce_reference(hh, ww, t, bias=bb, reduction=reduction, z_loss=zl,
                                      want_grads=False, row_block=4)["loss"]

        for name, arr, grad in (("hidden", hidden, g["grad_input"]), ("W", W, g["grad_W"]),
                                ("bias", b, g["grad_bias"])):
            fd = np.zeros_like(arr)
            for idx in np.ndindex(arr.shape):
                plus = arr.copy()
                minus = arr.copy()
                plus[idx] += h_step
                minus[idx] -= h_step
                args_p = {"hidden": (plus, W, b), "W": (hidden, plus, b), "bias": (hidden, W, plus)}[name]
                args_m = {"hidden": (minus, W, b), "W": (hidden, minus, b), "bias": (hidden, W, minus)}[name]
                fd[idx] = (loss_at(*args_p) - loss_at(*args_m)) / (2 * h_step)
            assert _rel(grad, fd) < 1e-6, (name, reduction, zl)


def pin_torch_fp64(orc):
    for reduction in ("mean", "sum"):
        for zl in (0.0, 1e-3):
            hidden, W, b, t = _tiny_case(seed=5, BT=37, H=16, V=50, ignore_rows=(0, 9, 30))
            got = orc.flce_reference(hidden, W, t, bias=b, reduction=reduction, z_loss=zl, row_block=8)
            th = torch.tensor(hidden, requires_grad=True)
            tw = torch.tensor(W, requires_grad=True)
            tb = torch.tensor(b, requires_grad=True)
            tt = torch.tensor(t)
            z = th @ tw.T + tb
            ce = torch.nn.functional.cross_entropy(z, tt, ignore_index=-100, reduction=reduction)
            valid = (tt != -100).double()
            scale = 1.0 / valid.sum() if reduction == "mean" else 1.0
            loss = ce + zl * scale * (torch.logsumexp(z, dim=1) ** 2 * valid).sum()
            loss.backward()
            assert abs(got["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
            assert _rel(got["grad_input"], th.grad.numpy()) < 1e-10
            assert _rel(got["grad_W"], tw.grad.numpy()) < 1e-10
            assert _rel(got["grad_bias"], tb.grad.numpy()) < 1e-10
            assert _rel(got["lse"], torch.logsumexp(z, dim=1).detach().numpy()) < 1e-13


def pin_closed_forms(orc):
    # W = 0, no bias: z = 0, LSE = log V, grad_input = 0,
    # grad_W[n] = s * sum_valid ((1 + 2 zl log V)/V - [y_t = n]) hidden[t]
    rng = np.random.default_rng(7)
    BT, H, V, zl = 9, 4, 7, 1e-2
    hidden = rng.standard_normal((BT, H))
    t = rng.integers(0, V, BT)
    t[3] = -100
    g = orc.flce_reference(hidden, np.zeros((V, H)), t, z_loss=zl, row_block=4)
    valid = t != -100
    n = int(valid.sum())
    lv = math.log(V)
    assert abs(g["loss"] - (lv + zl * lv * lv)) < 1e-13
    assert np.all(g["grad_input"] == 0.0)
    expect = np.zeros((V, H))
    for i in range(BT):
        if valid[i]:
            for j in range(V):
                expect[j] += ((1 + 2 * zl * lv) / V - (1.0 if j == t[i] else 0.0)) * hidden[i] / n
    assert _rel(g["grad_W"], expect) < 1e-12
    # V = 1: the CE part vanishes; loss = s * sum_valid zl z^2; grad row = s * 2 zl z * W[0]
    W1 = rng.standard_normal((1, H))
    t1 = np.zeros(BT, dtype=np.int64)
    t1[5] = -100
    g1 = orc.flce_reference(hidden, W1, t1, z_loss=zl, reduction="sum", row_block=4)
    z = hidden @ W1[0]
    v1 = t1 != -100
    assert abs(g1["loss"] - zl * float(np.sum(z[v1] ** 2))) < 1e-12
    assert _rel(g1["grad_input"], (2 * zl * z * v1)[:, None] * W1[0][None, :]) < 1e-12
    # golden closed-form CE values
    with open(os.path.join(GOLDEN, "ce_closed_forms.txt")) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            name, logit_s, tgt, lse_s, loss_s = [x.strip() for x in line.split("|")]
            if "*" in logit_s:
                val, cnt = logit_s.split("*")
                row = [float(val)] * int(cnt)
            else:
                row = [float(x) for x in logit_s.split(",")]
            r = orc.ce_reference(np.array([row]), np.array([int(tgt)]))
            assert abs(r["lse"][0] - float(lse_s)) < 1e-14 * max(1.0, float(lse_s)), name
            assert abs(r["ce_sum"] - float(loss_s)) < 1e-14 * max(1.0, float(loss_s)), name


def pin_invariants(orc):
    hidden, W, b, t = _tiny_case(seed=11, BT=10, H=6, V=9, ignore_rows=(1, 7))
    # LSE shift: a constant added to every bias entry shifts LSE and leaves loss / grads (zl = 0)
    g0 = orc.flce_reference(hidden, W, t, bias=b, row_block=3)
    g1 = orc.flce_reference(hidden, W, t, bias=b + 3.25, row_block=3)
    assert _rel(g1["lse"] - 3.25, g0["lse"]) < 1e-13
    assert abs(g1["loss"] - g0["loss"]) < 1e-12
    for k in ("grad_input", "grad_W", "grad_bias"):
        assert _rel(g1[k], g0[k]) < 1e-11, k
    # dlogits row sums: 0 with zl = 0, s * 2 zl LSE on valid rows with zl > 0 (summed: grad_bias)
    zl = 0.05
    for reduction in ("mean", "sum"):
        g = orc.flce_reference(hidden, W, t, bias=b, z_loss=zl, reduction=reduction, row_block=3)
        valid = t != -100
        s = 1.0 / valid.sum() if reduction == "mean" else 1.0
        assert abs(g["grad_bias"].sum() - s * 2 * zl * g["lse"][valid].sum()) < 1e-12
    assert abs(g0["grad_bias"].sum()) < 1e-13
    # ignored rows: zero grad_input rows; changing them changes nothing else
    assert np.all(g0["grad_input"][[1, 7]] == 0.0)
    h2 = hidden.copy()
    h2[[1, 7]] += 5.0
    g2 = orc.flce_reference(h2, W, t, bias=b, row_block=3)
    assert abs(g2["loss"] - g0["loss"]) < 1e-13
    assert _rel(g2["grad_W"], g0["grad_W"]) < 1e-13
    assert _rel(g2["grad_bias"], g0["grad_bias"]) < 1e-13
    # n_valid = 0: loss 0, all gradients 0
    gz = orc.flce_reference(hidden, W, np.full_like(t, -100), bias=b, z_loss=zl, row_block=3)
    assert gz["n_valid"] == 0 and gz["loss"] == 0.0
    for k in ("grad_input", "grad_W", "grad_bias"):
        assert np.all(gz[k] == 0.0)
    # vocabulary permutation: permute W rows, bias and relabel targets
    perm = np.random.default_rng(0).permutation(W.shape[0])
    inv = np.argsort(perm)
    tp = np.where(t == -100, -100, inv[np.where(t == -100, 0, t)])
    gp = orc.flce_reference(hidden, W[perm], tp, bias=b[perm], row_block=3)
    assert abs(gp["loss"] - g0["loss"]) < 1e-12
    assert _rel(gp["grad_W"], g0["grad_W"][perm]) < 1e-12
    assert _rel(gp["grad_bias"], g0["grad_bias"][perm]) < 1e-12
    assert _rel(gp["grad_input"], g0["grad_input"]) < 1e-12


def pin_ce(orc):
    rng = np.random.default_rng(13)
    B, V, zl = 11, 23, 1e-2
    x = rng.standard_normal((B, V)) * 2
    lab = rng.integers(0, V, B)
    lab[[2, 8]] = -100
    got = orc.ce_reference(x, lab, z_loss=zl, row_block=4)
    loops = orc.ce_reference_loops(x, lab, z_loss=zl)
    assert abs(got["ce_sum"] - loops["ce_sum"]) < 1e-12 * abs(loops["ce_sum"])
    assert abs(got["z_sum"] - loops["z_sum"]) < 1e-12 * abs(loops["z_sum"])
    assert got["n_valid"] == loops["n_valid"] == B - 2
    assert _rel(got["dlogits"], loops["dlogits"]) < 1e-12
    tx = torch.tensor(x, requires_grad=True)
    tl = torch.tensor(lab)
    ce = torch.nn.functional.cross_entropy(tx, tl, ignore_index=-100, reduction="sum")
    valid = (tl != -100).double()
    zs = (torch.logsumexp(tx, dim=1) ** 2 * valid).sum()
    (ce + zl * zs).backward()
    assert abs(got["ce_sum"] - ce.item()) < 1e-12 * abs(ce.item())
    assert abs(got["z_sum"] - zs.item()) < 1e-12 * abs(zs.item())
    assert _rel(got["dlogits"], tx.grad.numpy()) < 1e-12
    assert np.all(got["dlogits"][[2, 8]] == 0.0)


def pin_sampled_matches_full(orc):
    hidden, W, b, t = _tiny_case(seed=17, BT=40, H=12, V=33, ignore_rows=(3, 4, 20))
    zl = 1e-3
    full = orc.flce_reference(hidden, W, t, bias=b, z_loss=zl, row_block=7)
    L = orc.flce_lse(hidden, W, bias=b, row_block=6)
    assert _rel(L, full["lse"]) < 1e-14
    rows = [0, 3, 17, 39]
    vrows = [0, 5, 32]
    smp = orc.flce_sampled(hidden, W, t, L, rows, vrows, bias=b, z_loss=zl)
    assert abs(smp["loss"] - full["loss"]) < 1e-12 * abs(full["loss"])
    assert _rel(smp["grad_input_rows"], full["grad_input"][rows]) < 1e-12
    assert _rel(smp["grad_W_rows"], full["grad_W"][vrows]) < 1e-12
    assert _rel(smp["grad_bias_rows"], full["grad_bias"][vrows]) < 1e-12
    # the softmax parts: the full rows minus the onehot term, written out with loops from the targets
    # (grad_input: -s W[y_t] on valid rows; grad_W[n]: -s sum of hidden[t] over valid t with y_t = n;
    # grad_bias[n]: -s times that count)
    s = 1.0 / full["n_valid"]
    for i, r in enumerate(rows):
        one = -s * W[t[r]] if t[r] != -100 else np.zeros(W.shape[1])
        assert np.allclose(smp["grad_input_rows"][i] - smp["grad_input_rows_softmax"][i], one, rtol=0, atol=1e-13)
    for i, n in enumerate(vrows):
        one = np.zeros(hidden.shape[1])
        cnt = 0
        for tt in range(len(t)):
            if t[tt] == n:
                one -= s * hidden[tt]
                cnt += 1
        assert np.allclose(smp["grad_W_rows"][i] - smp["grad_W_rows_softmax"][i], one, rtol=0, atol=1e-13)
        assert abs(smp["grad_bias_rows"][i] - smp["grad_bias_rows_softmax"][i] + s * cnt) < 1e-13
    assert (t[:, None] == np.array(vrows)[None, :]).any(axis=0).any(), "the sample must hold a targeted entry"


def pin_unreduced_and_upstream(orc):
    # reduction "none" with an upstream gradient g (negative and zero entries included) and a scalar
    # grad_scale: the gradients are those of grad_scale * sum_t g_t l_t
    hidden, W, b, t = _tiny_case(seed=19)
    g = np.array([0.7, -1.3, 2.0, 0.0, 0.25, -0.5])
    zl, gs = 1e-2, -0.75
    got = orc.flce_reference(hidden, W, t, bias=b, reduction="none", z_loss=zl, grad_scale=gs,
                             grad_loss_per_token=g, row_block=4)
    h_step = 1e-6

    def fun(hh, ww, bb):
        r = orc.flce_reference(hh, ww, t, bias=bb, reduction="none", z_loss=zl, want_grads=False, row_block=4)
        return gs * float(np.dot(g, r["loss_per_token"]))

    for name, arr, grad in (("hidden", hidden, got["grad_input"]), ("W", W, got["grad_W"]),
                            ("bias", b, got["grad_bias"])):
        fd = np.zeros_like(arr)
        for idx in np.ndindex(arr.shape):
            plus = arr.copy()
            minus = arr.copy()
            plus[idx] += h_step
            minus[idx] -= h_step
            args_p = {"hidden": (plus, W, b), "W": (hidden, plus, b), "bias": (hidden, W, plus)}[name]
            args_m = {"hidden": (minus, W, b), "W": (hidden, minus, b), "bias": (hidden, W, minus)}[name]
            fd[idx] = (fun(*args_p) - fun(*args_m)) / (2 * h_step)
        assert _rel(grad, fd) < 1e-6, name
    # an independent library: per-token cross entropy + z-loss in torch, backward with g * grad_scale
    th = torch.tensor(hidden, requires_grad=True)
    tw = torch.tensor(W, requires_grad=True)
    tb = torch.tensor(b, requires_grad=True)
    tt = torch.tensor(t)
    z = th @ tw.T + tb
    valid = (tt != -100).double()
    per = torch.nn.functional.cross_entropy(z, tt, ignore_index=-100, reduction="none") + \
        zl * torch.logsumexp(z, dim=1) ** 2 * valid
    per.backward(torch.tensor(g * gs))
    assert _rel(got["loss_per_token"], per.detach().numpy()) < 1e-13
    assert _rel(got["grad_input"], th.grad.numpy()) < 1e-10
    assert _rel(got["grad_W"], tw.grad.numpy()) < 1e-10
    assert _rel(got["grad_bias"], tb.grad.numpy()) < 1e-10
    # consistency of the reductions: sum of per-token losses, and mean = none with g = 1/n_valid
    m = orc.flce_reference(hidden, W, t, bias=b, reduction="mean", z_loss=zl, row_block=4)
    n = orc.flce_reference(hidden, W, t, bias=b, reduction="none", z_loss=zl, row_block=4,
                           grad_loss_per_token=np.full(len(t), 1.0 / m["n_valid"]))
    assert abs(n["loss"] - m["loss"] * m["n_valid"]) < 1e-12 * abs(n["loss"])
    for k in ("grad_input", "grad_W", "grad_bias"):
        assert _rel(n[k], m[k]) < 1e-12, k


def pin_entropy(orc):
    # torch: -(softmax * log_softmax).sum over the vocabulary, for every row (ignored ones included)
    hidden, W, b, t = _tiny_case(seed=23, BT=21, H=9, V=40, ignore_rows=(0, 4))
    got = orc.flce_reference(hidden, W, t, bias=b, row_block=5, want_grads=False)
    z = torch.tensor(hidden) @ torch.tensor(W).T + torch.tensor(b)
    ref = -(torch.softmax(z, dim=1) * torch.log_softmax(z, dim=1)).sum(dim=1).numpy()
    assert _rel(got["entropy"], ref) < 1e-13
    # brute force per row from the definition, in plain loops
    for r in (0, 7, 20):
        zr = hidden[r] @ W.T + b
        pr = [math.exp(v - max(zr)) for v in zr]
        tot = math.fsum(pr)
        h = -math.fsum((q / tot) * math.log(q / tot) for q in pr)
        assert abs(got["entropy"][r] - h) < 1e-12
    # closed forms and bounds: W = 0 gives the uniform distribution (log V); V = 1 gives 0; a constant
    # added to every logit changes nothing; 0 <= H <= log V
    g0 = orc.flce_reference(hidden, np.zeros_like(W), t, want_grads=False, row_block=5)
    assert np.max(np.abs(g0["entropy"] - math.log(W.shape[0]))) < 1e-13
    g1 = orc.flce_reference(hidden, W[:1], np.zeros_like(t), want_grads=False, row_block=5)
    assert np.max(np.abs(g1["entropy"])) < 1e-15
    g2 = orc.flce_reference(hidden, W, t, bias=b + 7.5, row_block=5, want_grads=False)
    assert _rel(g2["entropy"], got["entropy"]) < 1e-12
    assert np.all(got["entropy"] >= 0) and np.all(got["entropy"] <= math.log(W.shape[0]) + 1e-12)


def pin_dlogits_matrix(orc):
    # the dlogits matrix against torch autograd of the logits, and against the oracle's own GEMMs
    hidden, W, b, t = _tiny_case(seed=29, BT=15, H=7, V=19, ignore_rows=(2, 11))
    for reduction, zl in (("mean", 1e-2), ("sum", 0.0)):
        d = orc.flce_dlogits(hidden, W, t, bias=b, reduction=reduction, z_loss=zl)
        z = torch.tensor(hidden @ W.T + b, requires_grad=True)
        tt = torch.tensor(t)
        valid = (tt != -100).double()
        scale = 1.0 / valid.sum() if reduction == "mean" else 1.0
        loss = torch.nn.functional.cross_entropy(z, tt, ignore_index=-100, reduction=reduction) + \
            zl * scale * (torch.logsumexp(z, dim=1) ** 2 * valid).sum()
        loss.backward()
        assert _rel(d, z.grad.numpy()) < 1e-12
        g = orc.flce_reference(hidden, W, t, bias=b, reduction=reduction, z_loss=zl, row_block=4)
        assert _rel(d @ W, g["grad_input"]) < 1e-12
        assert _rel(d.T @ hidden, g["grad_W"]) < 1e-12


def pin_widen_bf16_bits(orc):
    # bf16 bit patterns (uint16) widen to the exact value they encode: against hand-evaluated values
    # (sign, exponent field e, fraction f: (-1)^s 2^(e-127) (1 + f/128), subnormals 2^-126 f/128) and
    # against torch's own bfloat16 decoding
    cases = {
        0x0000: 0.0, 0x8000: -0.0, 0x0001: math.ldexp(1.0, -133), 0x8001: -math.ldexp(1.0, -133),
        0x007F: math.ldexp(127.0, -133), 0x0080: math.ldexp(1.0, -126), 0x3F80: 1.0, 0xBF80: -1.0,
        0x3FC0: 1.5, 0xC000: -2.0, 0x4049: 3.140625, 0x3DCD: 0.10009765625, 0x477F: 65280.0,
        0x4780: 65536.0, 0x7F7F: math.ldexp(255.0, 120), 0xFF7F: -math.ldexp(255.0, 120),
        0x7F80: math.inf, 0xFF80: -math.inf,
    }
    bits = np.array(sorted(cases), dtype=np.uint16)
    got = orc.widen(bits)
    assert got.dtype == np.float64 and got.shape == bits.shape
    for b_, v in zip(bits.tolist(), got.tolist()):
        assert v == cases[b_] and math.copysign(1.0, v) == math.copysign(1.0, cases[b_]), (hex(b_), v, cases[b_])
    assert np.isnan(orc.widen(np.array([0x7FC0, 0xFFC1], dtype=np.uint16))).all()
    rng = np.random.default_rng(29)
    every = np.arange(65536, dtype=np.uint32).astype(np.uint16)
    ref = torch.from_numpy(every.view(np.int16).copy()).view(torch.bfloat16).double().numpy()
    with np.errstate(invalid="ignore"):   # (the NaN patterns)
        w = orc.widen(every)
    fin = ~np.isnan(ref)
    assert np.array_equal(np.isnan(w), ~fin)
    assert np.array_equal(w[fin], ref[fin]) and np.array_equal(np.signbit(w[fin]), np.signbit(ref[fin]))
    # the fused loss from bf16 bit patterns equals the loss from the values they encode (torch, float64)
    hb = rng.integers(0x3C00, 0x4000, (9, 8)).astype(np.uint16) ^ (rng.integers(0, 2, (9, 8)).astype(np.uint16) << 15)
    wb = rng.integers(0x3A00, 0x3E00, (13, 8)).astype(np.uint16) ^ (rng.integers(0, 2, (13, 8)).astype(np.uint16) << 15)
    t = rng.integers(0, 13, 9)
    got = orc.flce_reference(hb, wb, t, row_block=4)
    th = torch.from_numpy(hb.view(np.int16).copy()).view(torch.bfloat16).double().requires_grad_(True)
    tw = torch.from_numpy(wb.view(np.int16).copy()).view(torch.bfloat16).double().requires_grad_(True)
    loss = torch.nn.functional.cross_entropy(th @ tw.T, torch.tensor(t))
    loss.backward()
    assert abs(got["loss"] - loss.item()) <= 1e-12 * abs(loss.item())
    assert _rel(got["grad_input"], th.grad.numpy()) < 1e-10
    assert _rel(got["grad_W"], tw.grad.numpy()) < 1e-10
    cb = rng.integers(0x3F00, 0x4100, (5, 11)).astype(np.uint16)
    lab = rng.integers(0, 11, 5)
    gce = orc.ce_reference(cb, lab)
    tx = torch.from_numpy(cb.view(np.int16).copy()).view(torch.bfloat16).double()
    assert abs(gce["ce_sum"] - torch.nn.functional.cross_entropy(tx, torch.tensor(lab), reduction="sum").item()) \
        <= 1e-12 * abs(gce["ce_sum"])


def pin_logit_avg_and_order(orc):
    # logit_avg: plain loops with exactly rounded sums; closed forms (W = 0 gives the bias, equal rows
    # give one matrix-vector product); the linearity identity mean_t z[t, n] = W[n] . mean_t hidden[t]
    # + b[n] (a different route to the same number); an empty batch
    hidden, W, b, _ = _tiny_case(seed=31, BT=9, H=4, V=6)
    got = orc.logit_avg(hidden, W, bias=b, row_block=4)
    for n in range(W.shape[0]):
        zs = [math.fsum(hidden[t, k] * W[n, k] for k in range(W.shape[1])) + b[n] for t in range(hidden.shape[0])]
        assert abs(got[n] - math.fsum(zs) / len(zs)) < 1e-13 * max(1.0, abs(got[n]))
    assert _rel(orc.logit_avg(hidden, np.zeros_like(W), bias=b), b) < 1e-15
    same = np.repeat(hidden[:1], 5, axis=0)
    assert _rel(orc.logit_avg(same, W, bias=b), W @ hidden[0] + b) < 1e-13
    assert _rel(orc.logit_avg(hidden, W, bias=b), W @ hidden.mean(axis=0) + b) < 1e-13
    assert _rel(orc.logit_avg(hidden, W), W @ hidden.mean(axis=0)) < 1e-13
    assert np.array_equal(orc.logit_avg(hidden[:0], W, bias=b), b)
    # the order: a hand-evaluated case with ties (largest first, ties by index), then brute force
    assert orc.vocab_order(np.array([0.0, 5.0, -1.0, 5.0, 2.0])).tolist() == [1, 3, 4, 0, 2]
    rng = np.random.default_rng(32)
    keys = rng.integers(-3, 4, 40).astype(np.float64) / 2.0
    order = orc.vocab_order(keys)
    assert order.tolist() == sorted(range(40), key=lambda n: (-keys[n], n))
    assert sorted(order.tolist()) == list(range(40))
    assert np.all(np.diff(keys[order]) <= 0)


PINS = [pin_loops_vs_vectorised, pin_finite_differences, pin_torch_fp64, pin_closed_forms,
        pin_invariants, pin_ce, pin_sampled_matches_full, pin_unreduced_and_upstream, pin_entropy,
        pin_dlogits_matrix, pin_logit_avg_and_order, pin_widen_bf16_bits]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_oracle_pin(pin):
    pin(ORACLE)


# ----------------------------------------------------------------------------- planted mistakes

MUTATIONS = {
    "z-loss factor dropped from gradient": ("d = p * (1.0 + 2.0 * z_loss * L)[:, None]", "d = p * (1.0 + z_loss * L)[:, None]"),
    "onehot sign flipped": ("            d[rows, y] -= 1.0\n            d *= (s * v)", "            d[rows, y] += 1.0\n            d *= (s * v)"),
    "grad_W accumulation dropped": ("grad_W += d.T @ h[r0:r1]", "grad_W = d.T @ h[r0:r1]"),
    "max term dropped from LSE": ("L = m + np.log(denom)", "L = np.log(denom)"),
    "z-loss term not squared": ("(L - z_y) + z_loss * L * L, 0.0))\n        if want_grads", "(L - z_y) + z_loss * L, 0.0))\n        if want_grads"),
    "target index shifted": ("y = np.where(v, t[r0:r1], 0)", "y = np.where(v, t[r0:r1], 0)[::-1]"),
    "mean over all rows": ("    n_valid = int(valid.sum())\n    s = _scale(n_valid, reduction)\n\n    loss_terms", "    n_valid = int(valid.sum())\n    s = _scale(BT, reduction)\n\n    loss_terms"),
    "bias sign flipped": ("        z = h[r0:r1] @ w.T\n        if b is not None:\n            z += b[None, :]\n        m = z.max", "        z = h[r0:r1] @ w.T\n        if b is not None:\n            z -= b[None, :]\n        m = z.max"),
    "ignored CE rows not zeroed": ("dl[r0:r1] = d * v[:, None]", "dl[r0:r1] = d"),
    "CE target column not adjusted": ("        d[rows, y[r0:r1]] -= 1.0\n        dl[r0:r1]", "        dl[r0:r1]"),
    "upstream gradient ignored": ("d *= (grad_scale * u[r0:r1])[:, None]", "d *= grad_scale"),
    "grad_scale applied twice": ("d *= (grad_scale * u[r0:r1])[:, None]", "d *= (grad_scale * grad_scale * u[r0:r1])[:, None]"),
    "entropy sign flipped": ("ent_all[r0:r1] = L - (e * z).sum(axis=1) / denom", "ent_all[r0:r1] = (e * z).sum(axis=1) / denom - L"),
    "entropy unnormalised": ("ent_all[r0:r1] = L - (e * z).sum(axis=1) / denom", "ent_all[r0:r1] = L - (e * z).sum(axis=1)"),
    "dlogits matrix target column not adjusted": ("    d[rows, t[rows]] -= 1.0\n    return d * (s * valid)", "    return d * (s * valid)"),
    "logit_avg bias dropped": ("            z += b[None, :]\n        col_sum", "            pass\n        col_sum"),
    "logit_avg divided by V": ("return col_sum / BT", "return col_sum / w.shape[0]"),
    "vocabulary order ascending": ('np.argsort(-a, kind="stable")', 'np.argsort(a, kind="stable")'),
    "vocabulary ties in reverse index order": ('np.argsort(-a, kind="stable")',
                                               '(len(a) - 1 - np.argsort(-a[::-1], kind="stable"))'),
    "bf16 bits widened with a 15-bit shift": ("(a.astype(np.uint32) << 16)", "(a.astype(np.uint32) << 15)"),
    "bf16 bit patterns read as integers": ("    if a.dtype == np.uint16:\n", "    if False:\n"),
    "sampled softmax part keeps the target column": (
        "    dc_soft = dc * (s * valid)[:, None]\n",
        "    dc_soft = (dc - (y[:, None] == vr[None, :])) * (s * valid)[:, None]\n"),
    "grad_input uses transposed product": ("grad_input[r0:r1] = d @ w", "grad_input[r0:r1] = (w.T @ d.T).T * 0 + d @ w[::-1]"),
}


def _mutated_oracle(src: str, old: str, new: str):
    assert src.count(old) == 1, f"mutation anchor must be unique: {old!r}"
    mod = types.ModuleType("oracle_mutant")
    exec(compile(src.replace(old, new), "oracle_mutant", "exec"), mod.__dict__)
    return mod


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistakes(name):
    with open(ORACLE.__file__) as f:
        src = f.read()
    mutant = _mutated_oracle(src, *MUTATIONS[name])
    failures = 0
    for pin in PINS:
        try:
            pin(mutant)
        except (AssertionError, ValueError, IndexError):
            failures += 1
    assert failures > 0, f"no pin caught the planted mistake: {name}"
