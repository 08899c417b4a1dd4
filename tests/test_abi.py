"""The C ABI without a GPU: the library loads, exports every symbol include/flce.h declares, sizes
its workspaces, and rejects bad arguments with the documented codes before touching a device."""
import ctypes
import os
import re

import pytest

from linear_cross_entropy_tma_gb300 import _lib

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

INVALID_ARG, MISALIGNED, WS_SMALL, UNSUPPORTED, NO_DEVICE = 1, 2, 3, 4, 6


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(_lib.LIB_PATH):
        from linear_cross_entropy_tma_gb300 import build
        build.build()
    return _lib.load()


def declared_functions():
    src = open(os.path.join(ROOT, "include", "flce.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", src, flags=re.M)) - {"defined"})


def test_header_symbols_exported(lib):
    names = declared_functions()
    assert set(names) == set(_lib.EXPORTED), names
    for n in names:
        assert hasattr(lib, n), n


def test_library_has_no_driver_dependency():
    # the runtime is linked statically and the driver is reached through the runtime's entry-point
    # query, so the library loads where no GPU driver exists
    out = os.popen(f"ldd {_lib.LIB_PATH}").read()
    assert "libcuda.so" not in out and "libcudart.so" not in out


def test_workspace_sizes(lib):
    assert lib.flce_workspace_size(-1, 8, 8) == 0
    a = lib.flce_workspace_size(128, 64, 512)
    b = lib.flce_workspace_size(65535, 1024, 176245)
    assert 0 < a < b
    # O(BT + V): no (BT, V) term; independent of H
    assert b < 64 * 1024 * 1024
    assert lib.flce_workspace_size(65535, 1024, 176245) == lib.flce_workspace_size(65535, 64, 176245)
    assert lib.flce_workspace_size(65535, 64, 176245) - lib.flce_workspace_size(65535, 64, 8) == 4 * (176384 - 256)
    assert lib.ce_workspace_size(8192, 128256) == 256 + 16 * 8192
    # the vocabulary sort adds a sorted copy of W (V x H bf16) and O(V + BT + H) scratch
    plain = _lib.FwdBwdOptions(1.0, None, None, 0, None, 0.0, 0, None, None, 0)
    sort = _lib.FwdBwdOptions(1.0, None, None, 0, None, 0.0, 1, None, None, 0)
    assert lib.flce_workspace_size_ex(128, 64, 512, None) == a
    assert lib.flce_workspace_size_ex(128, 64, 512, ctypes.byref(plain)) == a
    extra = lib.flce_workspace_size_ex(65535, 1024, 176245, ctypes.byref(sort)) - b
    assert 176245 * 1024 * 2 <= extra < 176245 * 1024 * 2 + 16 * 1024 * 1024
    assert lib.flce_workspace_size_ex(-1, 64, 512, ctypes.byref(sort)) == 0


def _fwd(lib, hidden=0x1000, W=0x2000, bias=None, target=0x3000, BT=128, H=64, V=512, red=0, loss=0x4000,
         gi=0x5000, gw=0x6000, gb=None, nv=None, ws=0x7000, wsb=1 << 30):
    return lib.flce_fwd_bwd(hidden, W, bias, target, BT, H, V, -100, red, 0.0, loss, gi, gw, gb, nv, ws, wsb, None)


def test_fwd_bwd_argument_errors(lib):
    # (all of these are rejected before any CUDA call, so no GPU is needed)
    assert _fwd(lib, W=None) == INVALID_ARG
    assert _fwd(lib, loss=None) == INVALID_ARG
    assert _fwd(lib, ws=None) == INVALID_ARG
    assert _fwd(lib, BT=-1) == INVALID_ARG
    assert _fwd(lib, V=0) == INVALID_ARG
    assert _fwd(lib, red=2) == INVALID_ARG
    assert _fwd(lib, gb=0x8000) == INVALID_ARG          # grad_bias without bias
    assert _fwd(lib, gi=0x1000) == INVALID_ARG          # grad_input aliases hidden
    assert _fwd(lib, H=60) == UNSUPPORTED               # H % 8 != 0
    assert _fwd(lib, V=1 << 31) == UNSUPPORTED
    assert _fwd(lib, hidden=0x1008) == MISALIGNED
    assert _fwd(lib, ws=0x7010) == MISALIGNED
    assert _fwd(lib, wsb=16) == WS_SMALL
    assert b"workspace" in lib.flce_last_error()


def _fwd_ex(lib, red=2, loss=None, grad_scale=1.0, gtok=None, ltok=None, acc=0, gi=0x5000, ent=None, eps=0.0,
            sort=0, la=None, vo=None, wsb=1 << 30, splits=0, tsplits=0, stall=0):
    opts = _lib.FwdBwdOptions(grad_scale, gtok, ltok, acc, ent, eps, sort, la, vo, 0, splits, tsplits, stall)
    return lib.flce_fwd_bwd_ex(0x1000, 0x2000, None, 0x3000, 128, 64, 512, -100, red, 0.0, loss, gi, 0x6000, None,
                               None, 0x7000, wsb, ctypes.byref(opts), None)


def test_fwd_bwd_ex_argument_errors(lib):
    assert _fwd_ex(lib, red=3) == INVALID_ARG
    assert _fwd_ex(lib, red=0, loss=None) == INVALID_ARG                 # mean needs the scalar loss
    assert _fwd_ex(lib, red=0, loss=0x4000, gtok=0x9000) == INVALID_ARG  # per-token upstream grads: none only
    assert _fwd_ex(lib, grad_scale=float("nan")) == INVALID_ARG
    assert _fwd_ex(lib, grad_scale=float("inf")) == INVALID_ARG
    assert _fwd_ex(lib, eps=-1e-3) == INVALID_ARG
    assert _fwd_ex(lib, eps=float("nan")) == INVALID_ARG
    assert _fwd_ex(lib, splits=-1) == INVALID_ARG
    assert _fwd_ex(lib, splits=3) == NO_DEVICE
    assert _fwd_ex(lib, splits=1000) == NO_DEVICE                         # (clamped, not an error)
    assert _fwd_ex(lib, tsplits=-2) == INVALID_ARG
    assert _fwd_ex(lib, tsplits=4) == NO_DEVICE
    assert _fwd_ex(lib, ltok=0x9002) == MISALIGNED
    assert _fwd_ex(lib, gtok=0x9001) == MISALIGNED
    assert _fwd_ex(lib, ent=0x9003) == MISALIGNED
    # the vocabulary sort: its outputs need sort_vocab, 4-byte alignment and the larger workspace
    assert _fwd_ex(lib, la=0xC000) == INVALID_ARG
    assert _fwd_ex(lib, vo=0xD000) == INVALID_ARG
    assert _fwd_ex(lib, sort=1, la=0xC002) == MISALIGNED
    assert _fwd_ex(lib, sort=1, vo=0xD001) == MISALIGNED
    assert _fwd_ex(lib, sort=1, wsb=lib.flce_workspace_size(128, 64, 512)) == WS_SMALL
    assert _fwd_ex(lib, sort=1, la=0xC000, vo=0xD000, eps=1e-3) == NO_DEVICE
    # valid argument sets get as far as the device check (no GPU here)
    assert _fwd_ex(lib) == NO_DEVICE
    assert _fwd_ex(lib, gtok=0x9000, ltok=0xA000, acc=1, grad_scale=-2.0) == NO_DEVICE
    assert _fwd_ex(lib, red=1, loss=0x4000, acc=1) == NO_DEVICE
    assert _fwd_ex(lib, red=0, loss=0x4000, ent=0xB000) == NO_DEVICE
    assert _fwd_ex(lib, red=0, loss=0x4000, eps=2.0 ** -12) == NO_DEVICE
    # the plain entry points do not take reduction none
    assert _fwd(lib, red=2) == INVALID_ARG
    # the test-only stall of the bounded waits: at most one second
    assert _fwd_ex(lib, stall=1000001) == INVALID_ARG
    assert b"debug_stall_us" in lib.flce_last_error()
    assert _fwd_ex(lib, stall=1000) == NO_DEVICE


def test_scale_and_reduce_argument_errors(lib):
    def scale(g=0x1000, dtype=0, n=100, up=0x2000, div=None):
        return lib.flce_scale_gradient(g, dtype, n, up, div, None)

    assert scale(dtype=3) == INVALID_ARG
    assert scale(n=-1) == INVALID_ARG
    assert scale(up=None) == INVALID_ARG
    assert scale(g=None) == INVALID_ARG
    assert scale(g=0x1008) == MISALIGNED
    assert scale(up=0x2002) == MISALIGNED
    assert scale(div=0x3004) == MISALIGNED
    assert scale() == NO_DEVICE
    assert scale(g=None, n=0, div=0x3000, dtype=2) == NO_DEVICE

    def red(cs=0x1000, zs=0x1004, nv=0x1008, reduction=0, loss=0x1010):
        return lib.ce_reduce_loss(cs, zs, nv, 1e-4, reduction, loss, None)

    assert red(reduction=2) == INVALID_ARG
    assert red(loss=None) == INVALID_ARG
    assert red(nv=None) == INVALID_ARG
    assert red(nv=0x100C) == MISALIGNED
    assert red() == NO_DEVICE
    assert red(reduction=1) == NO_DEVICE


def test_ce_noalloc_argument_errors(lib):
    def na(logits=0x1000, labels=0x2000, B=8, V=16, cs=0x3000, zs=0x3004, nv=0x3008):
        return lib.ce_with_grad_noalloc(logits, labels, B, V, -100, 0.0, cs, zs, nv, None)

    assert na(logits=None) == INVALID_ARG and b"non-NULL" in lib.flce_last_error()
    assert na(V=0) == INVALID_ARG and b"V > 0" in lib.flce_last_error()
    assert na(V=1 << 31) == UNSUPPORTED and b"V must be below 2^31" in lib.flce_last_error()
    assert na(B=262145) == UNSUPPORTED and b"at most 262144 rows" in lib.flce_last_error()
    assert na(logits=0x1008) == MISALIGNED and b"misaligned" in lib.flce_last_error()
    assert na() == NO_DEVICE and b"10.3" in lib.flce_last_error()


def test_ce_argument_errors(lib):
    def ce(logits=0x1000, labels=0x2000, B=8, V=16, cs=0x3000, zs=0x3100, nv=0x3200, ws=0x4000, wsb=1 << 20):
        return lib.ce_with_grad(logits, labels, B, V, -100, 0.0, cs, zs, nv, ws, wsb, None)

    assert ce(logits=None) == INVALID_ARG
    assert ce(nv=None) == INVALID_ARG
    assert ce(V=0) == INVALID_ARG
    assert ce(B=1 << 31) == UNSUPPORTED
    assert ce(logits=0x1002) == MISALIGNED
    assert ce(wsb=100) == WS_SMALL
    assert lib.flce_read_device_status(None, None, None) == INVALID_ARG


def test_ce_ex_argument_errors(lib):
    def ce(logits=0x10000, dl=0x10000, dtype=1, B=8, V=16, ws=0x40000):
        return lib.ce_with_grad_ex(logits, dl, dtype, 0x2000, B, V, -100, 0.0, 0x3000, 0x3100, 0x3200, ws, 1 << 20,
                                   None)

    assert ce(dtype=3) == INVALID_ARG
    assert ce(dtype=-1) == INVALID_ARG
    assert ce(dl=0x10010) == INVALID_ARG          # separate buffer overlapping the logits (8 x 16 x 2 bytes)
    assert ce(dl=0x10000 + 8 * 16 * 2 + 8) == MISALIGNED
    assert ce(logits=0x10008, dl=None) == MISALIGNED
    # in place, out of place right after the logits, and no gradient reach the device check
    assert ce() == NO_DEVICE
    assert ce(dl=0x10000 + 8 * 16 * 2) == NO_DEVICE
    assert ce(dl=None, dtype=2) == NO_DEVICE
    assert ce(dl=0x10000 + 8 * 16 * 4, dtype=2) == NO_DEVICE
    assert ce(dl=0x10000 + 8 * 16 * 2, dtype=2) == INVALID_ARG   # overlaps at 4 bytes per element


def test_status_strings(lib):
    assert lib.flce_status_string(0) == b"FLCE_OK"
    assert lib.flce_status_string(3) == b"FLCE_ERR_WORKSPACE_TOO_SMALL"
    assert lib.flce_status_string(99) == b"FLCE_ERR_UNKNOWN"


def test_binding_fails_loudly_without_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "_lib", None)
    monkeypatch.setattr(_lib, "LIB_PATH", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="missing"):
        _lib.load()
