"""Seeded synthetic inputs for the fused linear cross-entropy path and the standalone CE kernel.

This module only draws random numbers and rounds them to the storage types.  It holds none of the
method's arithmetic (no logits, no softmax, no loss), so both the CPU oracle and the CUDA path can be
fed from it without sharing any of the computation.

Recipe (the same on every machine; NumPy PCG64 streams derived from one seed):
  * normal draws use ``Generator.standard_normal`` in float64, multiplied by the standard deviation
    (the second parameter of N(mean, std) is read as a standard deviation), cast to float32;
  * bf16 values are the float32 values rounded to nearest-even (what ``tensor.to(torch.bfloat16)``
    does), stored as raw uint16 bit patterns;
  * exactly ``rint(p * BT)`` rows get the ignore label, picked by a seeded permutation;
  * uniform targets are integers drawn uniformly from [0, V);
  * Zipf(s) targets use P(k) proportional to (k + 1)^-s over k in [0, V), drawn by inverse CDF from
    seeded uniforms, token id = rank (id 0 is the most frequent).

The five workloads mirror the shapes the pages discuss: the LM heads of Qwen3-0.6B (p1 "The setting"),
Gemma-2 2B with 8192 tokens (p2 "Naive CE is expensive"), the BT=65535, H=1024, V=176245 shape p1
benchmarks ("The engineering wall", "Putting numbers on it"), and the [8192, 128256] bf16 logits of the
Greyhound usage example (p3 "Usage").
"""
from __future__ import annotations

import dataclasses
import hashlib

import numpy as np

IGNORE_INDEX = -100


@dataclasses.dataclass(frozen=True)
class FusedWorkload:
    """One fused linear cross-entropy problem: hidden [BT, H], W [V, H], optional bias [V]."""

    name: str
    BT: int
    H: int
    V: int
    hidden_std: float = 1.0
    w_std: float = 0.02
    bias_std: float | None = None       # None: no bias
    ignore_frac: float = 0.05
    targets: str = "uniform"            # "uniform" or "zipf"
    zipf_s: float = 1.1
    reduction: str = "mean"
    z_loss: float = 0.0
    seed: int = 0

    @property
    def n_ignored(self) -> int:
        return int(np.rint(self.ignore_frac * self.BT))

    @property
    def n_valid(self) -> int:
        return self.BT - self.n_ignored

    def flops(self) -> int:
        """Algorithmic work of one fused forward+backward: 8*BT*V*H (logits, grad_input GEMM,
        logits recompute, grad_W GEMM)."""
        return 8 * self.BT * self.V * self.H


@dataclasses.dataclass(frozen=True)
class CEWorkload:
    """One standalone CE problem over materialised bf16 logits [B, V]."""

    name: str
    B: int
    V: int
    logit_std: float = 2.0
    ignore_frac: float = 0.05
    z_loss: float = 1e-4
    seed: int = 0

    @property
    def n_ignored(self) -> int:
        return int(np.rint(self.ignore_frac * self.B))

    def bytes_moved(self) -> int:
        """Algorithmic HBM traffic: one read of the logits plus one write of dlogits (bf16)."""
        return 2 * self.B * self.V * 2


TINY = FusedWorkload("tiny BT=128 H=64 V=512", BT=128, H=64, V=512, ignore_frac=0.05)
QWEN3_0P6B = FusedWorkload("Qwen3-0.6B LM head BT=4096 H=1024 V=151936", BT=4096, H=1024, V=151936,
                           ignore_frac=0.10)
GEMMA2_2B = FusedWorkload("Gemma-2-2B LM head BT=8192 H=2304 V=256128 bias zipf z_loss=1e-4",
                          BT=8192, H=2304, V=256128, bias_std=0.1, ignore_frac=0.03, targets="zipf",
                          z_loss=1e-4)
LONG_BATCH = FusedWorkload("long-batch LM head BT=65535 H=1024 V=176245", BT=65535, H=1024, V=176245,
                           ignore_frac=0.10)
CE_LOGITS = CEWorkload("standalone CE logits bf16 [8192, 128256] sum z_loss=1e-4", B=8192, V=128256)

FUSED_WORKLOADS = {"tiny": TINY, "qwen3": QWEN3_0P6B, "gemma2": GEMMA2_2B, "long": LONG_BATCH}


def _streams(seed: int, n: int) -> list[np.random.Generator]:
    return [np.random.Generator(np.random.PCG64(s)) for s in np.random.SeedSequence(seed).spawn(n)]


def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); returns the uint16 bit patterns."""
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32).astype(np.uint64)
    u = u + 0x7FFF + ((u >> 16) & 1)
    return (u >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    """Widen bfloat16 bit patterns to float32 exactly."""
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def normal_bf16(rng: np.random.Generator, shape, std: float, chunk_rows: int = 8192) -> np.ndarray:
    """N(0, std) samples rounded to bf16 (uint16 bits), generated in row chunks to bound memory."""
    shape = tuple(int(s) for s in shape)
    out = np.empty(shape, dtype=np.uint16)
    rows = shape[0]
    cols = int(np.prod(shape[1:])) if len(shape) > 1 else 1
    flat = out.reshape(rows, cols)
    for r0 in range(0, rows, chunk_rows):
        r1 = min(rows, r0 + chunk_rows)
        x = rng.standard_normal((r1 - r0, cols), dtype=np.float64) * std
        flat[r0:r1] = f32_to_bf16_bits(x.astype(np.float32))
    return out


def _targets(rng_t: np.random.Generator, rng_i: np.random.Generator, n: int, V: int, kind: str,
             zipf_s: float, n_ignored: int) -> np.ndarray:
    if kind == "uniform":
        t = rng_t.integers(0, V, size=n, dtype=np.int64)
    elif kind == "zipf":
        w = np.arange(1, V + 1, dtype=np.float64) ** (-zipf_s)
        cdf = np.cumsum(w)
        cdf /= cdf[-1]
        u = rng_t.random(n)
        t = np.minimum(np.searchsorted(cdf, u, side="right"), V - 1).astype(np.int64)
    else:
        raise ValueError(f"unknown target distribution {kind!r}")
    if n_ignored:
        t[rng_i.permutation(n)[:n_ignored]] = IGNORE_INDEX
    return t


def make_fused_inputs(wl: FusedWorkload) -> dict:
    """Inputs of one fused workload as host arrays.

    Returns a dict with ``hidden`` and ``W`` (uint16 bf16 bits), ``bias`` (float32 or None) and
    ``target`` (int64), plus the workload's scalar settings.
    """
    g_h, g_w, g_b, g_t, g_i = _streams(wl.seed, 5)
    hidden = normal_bf16(g_h, (wl.BT, wl.H), wl.hidden_std)
    W = normal_bf16(g_w, (wl.V, wl.H), wl.w_std)
    bias = None
    if wl.bias_std is not None:
        bias = (g_b.standard_normal(wl.V, dtype=np.float64) * wl.bias_std).astype(np.float32)
    target = _targets(g_t, g_i, wl.BT, wl.V, wl.targets, wl.zipf_s, wl.n_ignored)
    return dict(hidden=hidden, W=W, bias=bias, target=target, ignore_index=IGNORE_INDEX,
                reduction=wl.reduction, z_loss=wl.z_loss)


def make_ce_inputs(wl: CEWorkload, rows: slice | None = None) -> dict:
    """Inputs of one standalone CE workload: ``logits`` (uint16 bf16 bits [B, V]) and ``labels``.

    ``rows`` selects a contiguous block of rows; the values of a row do not depend on which rows are
    generated, so a sample equals the same rows of the full tensor.
    """
    g_l, g_t, g_i = _streams(wl.seed, 3)
    labels = _targets(g_t, g_i, wl.B, wl.V, "uniform", 0.0, wl.n_ignored)
    r = rows if rows is not None else slice(0, wl.B)
    r0, r1 = r.start or 0, r.stop if r.stop is not None else wl.B
    logits = np.empty((r1 - r0, wl.V), dtype=np.uint16)
    # Each block of 64 rows has its own child stream, so any row range is reproducible alone.
    block = 64
    for b0 in range((r0 // block) * block, r1, block):
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([wl.seed, 1, b0 // block])))
        x = g.standard_normal((block, wl.V), dtype=np.float64) * wl.logit_std
        xb = f32_to_bf16_bits(x.astype(np.float32))
        lo, hi = max(b0, r0), min(b0 + block, r1)
        logits[lo - r0:hi - r0] = xb[lo - b0:hi - b0]
    del g_l
    return dict(logits=logits, labels=labels[r0:r1], ignore_index=IGNORE_INDEX, z_loss=wl.z_loss)


def digest(*arrays) -> str:
    """sha256 over the raw bytes of the given arrays (None entries are skipped)."""
    h = hashlib.sha256()
    for a in arrays:
        if a is not None:
            h.update(np.ascontiguousarray(a).view(np.uint8).tobytes())
    return h.hexdigest()
