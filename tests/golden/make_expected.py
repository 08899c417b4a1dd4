"""Write the stored expected values for the full-size parity tests.

Calls only the CPU oracle (``oracle/``) and the seeded input generators.  For every full-size workload
it records a digest of the generated inputs (the GPU test regenerates them and checks the digest
first), the oracle's loss and n_valid, and sampled outputs the oracle computes one by one:
grad_input rows for sampled tokens, grad_W / grad_bias rows for sampled vocabulary entries (these
need the float64 LSE of every token, which this script computes), and for the standalone CE
workload ce_sum, z_sum, n_valid and the dlogits of sampled rows.

The samples: tokens 0, BT - 1, the first ignored token, random tokens, and 8 tokens among the last 512
(the row blocks that the grad_input pass splits over the vocabulary when its last wave is partly
filled); vocabulary entries 0, V - 1, the most frequent target, the first token's target, random
entries, 16 entries that no token targets (their grad_W rows are the softmax part alone), and 8 entries
among the last 512 (the rows the grad_W pass splits over the tokens).  Besides the full rows the file
holds the oracle's softmax parts (the rows without the onehot term of dlogits), in float64, and each
sampled entry's target count.

Usage:  python tests/golden/make_expected.py [name ...]     (names: qwen3 gemma2 long ce)
"""
from __future__ import annotations

import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, os.path.dirname(os.path.dirname(HERE)))

import oracle  # noqa: E402
from linear_cross_entropy_tma_gb300 import workloads as wl  # noqa: E402

N_ROWS = 32
N_VOCAB = 16
N_UNTARGETED = 16
N_TAIL = 8
TAIL = 512


def sample_rows(BT: int, target: np.ndarray, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    ign = np.flatnonzero(target == wl.IGNORE_INDEX)
    rows = {0, BT - 1, int(ign[0])} if ign.size else {0, BT - 1}
    while len(rows) < N_ROWS:
        rows.add(int(rng.integers(0, BT)))
    tail = rng.choice(np.arange(max(0, BT - TAIL), BT), size=min(N_TAIL, BT), replace=False)
    rows.update(int(r) for r in tail)
    return np.array(sorted(rows), dtype=np.int64)


def sample_vocab(V: int, target: np.ndarray, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed + 1)
    t = target[target != wl.IGNORE_INDEX]
    counts = np.bincount(t, minlength=V)
    vs = {0, V - 1, int(counts.argmax()), int(t[0])}
    while len(vs) < N_VOCAB:
        vs.add(int(rng.integers(0, V)))
    free = np.flatnonzero(counts == 0)
    vs.update(int(v) for v in rng.choice(free, size=min(N_UNTARGETED, free.size), replace=False))
    tail = np.arange(max(0, V - TAIL), V)
    tail_free = tail[counts[tail] == 0]
    tail_hit = tail[counts[tail] > 0]
    # tail entries: untargeted ones and targeted ones
    vs.update(int(v) for v in rng.choice(tail_free, size=min(N_TAIL // 2, tail_free.size), replace=False))
    vs.update(int(v) for v in rng.choice(tail_hit, size=min(N_TAIL - N_TAIL // 2, tail_hit.size), replace=False))
    return np.array(sorted(vs), dtype=np.int64)


def make_fused(key: str) -> None:
    w = wl.FUSED_WORKLOADS[key]
    t0 = time.time()
    d = wl.make_fused_inputs(w)
    dig = wl.digest(d["hidden"], d["W"], d["bias"], d["target"])
    L = oracle.flce_lse(d["hidden"], d["W"], bias=d["bias"], row_block=256)
    rows = sample_rows(w.BT, d["target"], w.seed)
    vocab = sample_vocab(w.V, d["target"], w.seed)
    smp = oracle.flce_sampled(d["hidden"], d["W"], d["target"], L, rows, vocab, bias=d["bias"],
                              reduction=w.reduction, z_loss=w.z_loss)
    t = d["target"]
    counts = np.bincount(t[(t >= 0) & (t < w.V)], minlength=w.V)
    out = dict(digest=np.array(dig), loss=np.float64(smp["loss"]), n_valid=np.int64(smp["n_valid"]),
               rows=rows, vocab_rows=vocab, lse_rows=L[rows], vocab_target_count=counts[vocab].astype(np.int64),
               grad_input_rows=smp["grad_input_rows"], grad_W_rows=smp["grad_W_rows"],
               grad_input_rows_softmax=smp["grad_input_rows_softmax"],
               grad_W_rows_softmax=smp["grad_W_rows_softmax"])
    if smp["grad_bias_rows"] is not None:
        out["grad_bias_rows"] = smp["grad_bias_rows"]
        out["grad_bias_rows_softmax"] = smp["grad_bias_rows_softmax"]
    np.savez_compressed(os.path.join(HERE, f"expected_{key}.npz"), **out)
    print(f"{key}: loss={smp['loss']:.12f} n_valid={smp['n_valid']} ({time.time() - t0:.1f} s)")


def make_ce() -> None:
    w = wl.CE_LOGITS
    t0 = time.time()
    d = wl.make_ce_inputs(w)
    dig = wl.digest(d["logits"], d["labels"])
    rows = sample_rows(w.B, d["labels"], w.seed)
    ce_sum = z_sum = 0.0
    n_valid = 0
    parts_ce, parts_z = [], []
    block = 512
    for r0 in range(0, w.B, block):
        r = oracle.ce_reference(d["logits"][r0:r0 + block], d["labels"][r0:r0 + block], z_loss=w.z_loss)
        parts_ce.append(r["ce_sum"])
        parts_z.append(r["z_sum"])
        n_valid += r["n_valid"]
    import math
    ce_sum = math.fsum(parts_ce)
    z_sum = math.fsum(parts_z)
    # sampled dlogits rows are cheap and are computed by the test itself
    np.savez_compressed(os.path.join(HERE, "expected_ce.npz"), digest=np.array(dig), ce_sum=np.float64(ce_sum),
                        z_sum=np.float64(z_sum), n_valid=np.int64(n_valid), rows=rows)
    print(f"ce: ce_sum={ce_sum:.6f} z_sum={z_sum:.6f} n_valid={n_valid} ({time.time() - t0:.1f} s)")


if __name__ == "__main__":
    names = sys.argv[1:] or ["qwen3", "gemma2", "long", "ce"]
    for n in names:
        make_ce() if n == "ce" else make_fused(n)
