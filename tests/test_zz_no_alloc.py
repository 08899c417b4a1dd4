"""ce_with_grad_noalloc: the standalone CE entry point for callers that cannot allocate device memory
(for example a plugin that receives only its input and output buffers from an engine that plans all
device memory ahead).  It takes its scratch from a fixed array inside the library instead of a
workspace.  Checked through the C ABI against ce_with_grad on the same inputs and against the fp64
oracle, on two calls in a row (the second call finds the first call's leftovers in the shared array).  This file is collected last
so that a run stopping at the first failure has run every other test before it."""
import ctypes

import numpy as np
import pytest

import oracle
from linear_cross_entropy_tma_gb300 import _lib
from linear_cross_entropy_tma_gb300 import workloads as wl
from parity import assert_grad_close, assert_scalar_close, bf16_tensor, bf16_to_numpy_f32

pytestmark = pytest.mark.gpu

MAX_ROWS = 262144  # FLCE_CE_NOALLOC_MAX_ROWS in include/flce.h


def _inputs(B, V, seed):
    rng = np.random.default_rng(seed)
    x = wl.f32_to_bf16_bits((rng.standard_normal((B, V)) * 2.0).astype(np.float32))
    lab = rng.integers(0, V, B).astype(np.int64)
    lab[rng.permutation(B)[: B // 20]] = -100
    return x, lab


def _call_noalloc(lib, logits, labels, z_loss):
    import torch
    ce_sum = torch.empty(1, device="cuda")
    z_sum = torch.empty(1, device="cuda")
    n_valid = torch.empty(1, dtype=torch.int64, device="cuda")
    B, V = logits.shape
    _lib.check(lib.ce_with_grad_noalloc(logits.data_ptr(), labels.data_ptr(), B, V, -100, z_loss, ce_sum.data_ptr(),
                                        z_sum.data_ptr(), n_valid.data_ptr(),
                                        torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return ce_sum.item(), z_sum.item(), int(n_valid.item())


def _call_workspace(lib, logits, labels, z_loss):
    import torch
    ce_sum = torch.empty(1, device="cuda")
    z_sum = torch.empty(1, device="cuda")
    n_valid = torch.empty(1, dtype=torch.int64, device="cuda")
    B, V = logits.shape
    ws = torch.empty(_lib.ce_workspace_size(B, V), dtype=torch.uint8, device="cuda")
    _lib.check(lib.ce_with_grad(logits.data_ptr(), labels.data_ptr(), B, V, -100, z_loss, ce_sum.data_ptr(),
                                z_sum.data_ptr(), n_valid.data_ptr(), ws.data_ptr(), ws.numel(),
                                torch.cuda.current_stream().cuda_stream))
    torch.cuda.synchronize()
    return ce_sum.item(), z_sum.item(), int(n_valid.item())


def test_noalloc_matches_workspace_entry_point_twice():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA device is required for -m gpu tests")
    lib = _lib.load()
    for call, (B, V, seed) in enumerate([(700, 5003, 1), (2048, 32000, 2)]):
        x, lab = _inputs(B, V, seed)
        labels = torch.from_numpy(lab).cuda()
        a = bf16_tensor(x)
        b = bf16_tensor(x)
        got = _call_noalloc(lib, a, labels, 1e-4)
        ref = _call_workspace(lib, b, labels, 1e-4)
        assert got[2] == ref[2], f"call {call}: n_valid {got[2]} vs {ref[2]}"
        assert_scalar_close(got[0], ref[0], f"call {call}: ce_sum")
        assert_scalar_close(got[1], ref[1], f"call {call}: z_sum")
        assert_grad_close(bf16_to_numpy_f32(a), bf16_to_numpy_f32(b), f"call {call}: dlogits")
        orc = oracle.ce_reference(x, lab, z_loss=1e-4)
        assert got[2] == orc["n_valid"], f"call {call}: n_valid {got[2]} vs oracle {orc['n_valid']}"
        assert_scalar_close(got[0], orc["ce_sum"], f"call {call}: ce_sum vs oracle")
        assert_scalar_close(got[1], orc["z_sum"], f"call {call}: z_sum vs oracle")
        assert_grad_close(bf16_to_numpy_f32(a), orc["dlogits"], f"call {call}: dlogits vs oracle")


def test_noalloc_rejects_too_many_rows():
    lib = _lib.load()
    # rejected on the host before any device work, so the pointers are never dereferenced
    st = lib.ce_with_grad_noalloc(ctypes.c_void_p(256), ctypes.c_void_p(256), MAX_ROWS + 1, 128, -100, 0.0,
                                  ctypes.c_void_p(256), ctypes.c_void_p(256), ctypes.c_void_p(256), None)
    assert st == 4  # FLCE_ERR_UNSUPPORTED
    assert b"at most" in lib.flce_last_error()
