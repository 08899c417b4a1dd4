"""Data parallelism over tokens, on CPU: two gloo ranks each compute their token shard with the fp64
oracle (sum reduction), compose_token_shards reduces them, and the result must equal the unsharded
oracle.  The GPU path of the composition is the same host code around flce_fwd_bwd."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

from linear_cross_entropy_tma_gb300 import workloads as wl
from linear_cross_entropy_tma_gb300.data_parallel import compose_token_shards
import oracle

WORLD = 2


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _inputs(BT, H, V, bias, ignored, seed):
    rng = np.random.Generator(np.random.PCG64(seed))
    hidden = wl.f32_to_bf16_bits(rng.standard_normal((BT, H), dtype=np.float32))
    W = wl.f32_to_bf16_bits((0.5 * rng.standard_normal((V, H))).astype(np.float32))
    b = (0.1 * rng.standard_normal(V)).astype(np.float32) if bias else None
    target = rng.integers(0, V, BT).astype(np.int64)
    for i in ignored:
        target[i] = -100
    return hidden, W, b, target


def _rank(rank, port, case, split, result_path):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=WORLD)
    try:
        BT, H, V, bias, zl, red, ignored, seed = case
        hidden, W, b, target = _inputs(BT, H, V, bias, ignored, seed)
        lo, hi = (0, split) if rank == 0 else (split, BT)
        r = oracle.flce_reference(hidden[lo:hi], W, target[lo:hi], bias=b, reduction="sum", z_loss=zl, row_block=64)
        loss = torch.tensor([r["loss"]], dtype=torch.float64)
        n_valid = torch.tensor([r["n_valid"]], dtype=torch.int64)
        gi = torch.from_numpy(r["grad_input"].copy())
        gw = torch.from_numpy(r["grad_W"].copy())
        gb = torch.from_numpy(r["grad_bias"].copy()) if r["grad_bias"] is not None else None
        compose_token_shards(loss, n_valid, gi, gw, gb, reduction=red)
        np.savez(f"{result_path}.{rank}.npz", loss=loss.numpy(), n_valid=n_valid.numpy(), gi=gi.numpy(),
                 gw=gw.numpy(), gb=gb.numpy() if gb is not None else np.zeros(0))
    finally:
        dist.destroy_process_group()


CASES = {
    # name: (BT, H, V, bias, z_loss, reduction, ignored rows, seed), split point
    "mean-bias-zloss": ((37, 16, 50, True, 1e-2, "mean", (0, 5, 30), 1), 20),
    "sum": ((24, 8, 31, False, 0.0, "sum", (3,), 2), 7),
    "mean-shard-all-ignored": ((12, 8, 20, True, 0.0, "mean", (0, 1, 2, 3, 4), 3), 5),
    "mean-uneven": ((33, 12, 17, False, 1e-3, "mean", (), 4), 1),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_token_sharded_matches_unsharded(name, tmp_path):
    case, split = CASES[name]
    port = _free_port()
    ctx = mp.get_context("spawn")
    procs = [ctx.Process(target=_rank, args=(r, port, case, split, str(tmp_path / "res"))) for r in range(WORLD)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0, f"rank exited with {p.exitcode}"
    BT, H, V, bias, zl, red, ignored, seed = case
    hidden, W, b, target = _inputs(BT, H, V, bias, ignored, seed)
    ref = oracle.flce_reference(hidden, W, target, bias=b, reduction=red, z_loss=zl, row_block=64)
    res = [np.load(tmp_path / f"res.{r}.npz") for r in range(WORLD)]
    for r in range(WORLD):
        assert int(res[r]["n_valid"][0]) == ref["n_valid"]
        assert abs(float(res[r]["loss"][0]) - ref["loss"]) <= 1e-12 * max(1.0, abs(ref["loss"]))
        np.testing.assert_allclose(res[r]["gw"], ref["grad_W"], rtol=1e-12, atol=1e-14)
        if bias:
            np.testing.assert_allclose(res[r]["gb"], ref["grad_bias"], rtol=1e-12, atol=1e-14)
    gi = np.concatenate([res[0]["gi"], res[1]["gi"]], axis=0)
    np.testing.assert_allclose(gi, ref["grad_input"], rtol=1e-12, atol=1e-14)


def test_compose_rejects_unknown_reduction():
    with pytest.raises(ValueError):
        compose_token_shards(torch.zeros(1), torch.zeros(1, dtype=torch.int64), reduction="none")
