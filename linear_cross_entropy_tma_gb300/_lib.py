"""ctypes binding of libflce.so (argument marshalling only; every step runs in the CUDA kernels).

The functions below take torch CUDA tensors, check dtypes/shapes/devices, allocate the outputs and the
workspace with torch (PyTorch is only the memory and stream provider), and call the C ABI declared
in include/flce.h.  There is no fallback: if the library is missing, or the call returns an error,
a RuntimeError is raised.
"""
from __future__ import annotations

import ctypes
import os

PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(PKG, "libflce.so")

FLCE_OK = 0
STATUS_BAD_TARGET = 0x1
STATUS_TIMEOUT = 0x2
STATUS_INTERNAL = 0x4
EXPORTED = ("flce_workspace_size", "flce_workspace_size_ex", "flce_fwd_bwd", "flce_fwd_bwd_timed", "flce_fwd_bwd_ex", "ce_workspace_size",
            "ce_with_grad", "ce_with_grad_ex", "flce_read_device_status", "flce_status_string", "flce_last_error",
            "ce_with_grad_noalloc", "ce_reduce_loss", "flce_scale_gradient")
REDUCTIONS = {"mean": 0, "sum": 1, "none": 2}

_lib = None

c_p = ctypes.c_void_p
c_i64 = ctypes.c_int64
c_sz = ctypes.c_size_t


class FwdBwdOptions(ctypes.Structure):
    """flce_fwd_bwd_options of include/flce.h."""
    _fields_ = [("grad_scale", ctypes.c_float), ("grad_loss_per_token", c_p), ("loss_per_token", c_p),
                ("accumulate", ctypes.c_int), ("entropy", c_p), ("filter_eps", ctypes.c_float),
                ("sort_vocab", ctypes.c_int), ("logit_avg", c_p), ("vocab_order", c_p),
                ("separate_lse_pass", ctypes.c_int), ("vocab_splits", ctypes.c_int),
                ("token_splits", ctypes.c_int), ("debug_stall_us", ctypes.c_uint32)]


def load() -> ctypes.CDLL:
    """Load libflce.so once; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIB_PATH):
        raise RuntimeError(f"{LIB_PATH} is missing: build it with `python -m linear_cross_entropy_tma_gb300.build` "
                           "(needs nvcc from CUDA 13)")
    lib = ctypes.CDLL(LIB_PATH)
    lib.flce_workspace_size.restype = c_sz
    lib.flce_workspace_size.argtypes = [c_i64, c_i64, c_i64]
    lib.flce_workspace_size_ex.restype = c_sz
    lib.flce_workspace_size_ex.argtypes = [c_i64, c_i64, c_i64, ctypes.POINTER(FwdBwdOptions)]
    lib.flce_fwd_bwd.restype = ctypes.c_int
    lib.flce_fwd_bwd.argtypes = [c_p, c_p, c_p, c_p, c_i64, c_i64, c_i64, c_i64, ctypes.c_int, ctypes.c_float,
                                 c_p, c_p, c_p, c_p, c_p, c_p, c_sz, c_p]
    lib.flce_fwd_bwd_timed.restype = ctypes.c_int
    lib.flce_fwd_bwd_timed.argtypes = lib.flce_fwd_bwd.argtypes + [ctypes.POINTER(c_p), ctypes.c_int]
    lib.flce_fwd_bwd_ex.restype = ctypes.c_int
    lib.flce_fwd_bwd_ex.argtypes = lib.flce_fwd_bwd.argtypes[:-1] + [ctypes.POINTER(FwdBwdOptions), c_p]
    lib.ce_workspace_size.restype = c_sz
    lib.ce_workspace_size.argtypes = [c_i64, c_i64]
    lib.ce_with_grad.restype = ctypes.c_int
    lib.ce_with_grad.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, ctypes.c_float, c_p, c_p, c_p, c_p, c_sz, c_p]
    lib.ce_with_grad_ex.restype = ctypes.c_int
    lib.ce_with_grad_ex.argtypes = [c_p, c_p, ctypes.c_int, c_p, c_i64, c_i64, c_i64, ctypes.c_float, c_p, c_p, c_p,
                                    c_p, c_sz, c_p]
    lib.ce_with_grad_noalloc.restype = ctypes.c_int
    lib.ce_with_grad_noalloc.argtypes = [c_p, c_p, c_i64, c_i64, c_i64, ctypes.c_float, c_p, c_p, c_p, c_p]
    lib.ce_reduce_loss.restype = ctypes.c_int
    lib.ce_reduce_loss.argtypes = [c_p, c_p, c_p, ctypes.c_float, ctypes.c_int, c_p, c_p]
    lib.flce_scale_gradient.restype = ctypes.c_int
    lib.flce_scale_gradient.argtypes = [c_p, ctypes.c_int, c_i64, c_p, c_p, c_p]
    lib.flce_read_device_status.restype = ctypes.c_int
    lib.flce_read_device_status.argtypes = [c_p, ctypes.POINTER(ctypes.c_uint32), c_p]
    lib.flce_status_string.restype = ctypes.c_char_p
    lib.flce_status_string.argtypes = [ctypes.c_int]
    lib.flce_last_error.restype = ctypes.c_char_p
    lib.flce_last_error.argtypes = []
    _lib = lib
    return lib


def check(status: int) -> None:
    if status != FLCE_OK:
        lib = load()
        raise RuntimeError(f"{lib.flce_status_string(status).decode()}: {lib.flce_last_error().decode()}")


def _ptr(t) -> int | None:
    return None if t is None else t.data_ptr()


def _stream_ptr(stream) -> int | None:
    import torch
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def workspace_size(BT: int, H: int, V: int, sort_vocab: bool = False) -> int:
    """Workspace bytes of flce_fwd_bwd; with ``sort_vocab`` those of the vocabulary-sorting call."""
    if not sort_vocab:
        return int(load().flce_workspace_size(BT, H, V))
    opts = FwdBwdOptions(1.0, None, None, 0, None, 0.0, 1, None, None, 0)
    return int(load().flce_workspace_size_ex(BT, H, V, ctypes.byref(opts)))


def ce_workspace_size(B: int, V: int) -> int:
    return int(load().ce_workspace_size(B, V))


def _bf16_ptr_ok(t, name):
    import torch
    if t.dtype != torch.bfloat16 or not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA bfloat16 tensor")


def flce_fwd_bwd(hidden, W, target, bias=None, ignore_index: int = -100, reduction: str = "mean",
                 z_loss: float = 0.0, need_grad_input: bool = True, need_grad_W: bool = True, workspace=None,
                 out=None, stream=None, pass_events=None, grad_scale: float = 1.0, grad_loss_per_token=None,
                 accumulate: bool = False, want_loss_per_token: bool = False, want_entropy: bool = False,
                 filter_eps: float = 0.0, sort_vocab: bool = False, separate_lse_pass: bool = False,
                 vocab_splits: int = 0, token_splits: int = 0, debug_stall_us: int = 0) -> dict:
    """Fused linear cross-entropy forward + backward on the current CUDA device.

    hidden [BT, H] bf16, W [V, H] bf16, target [BT] int64, bias [V] fp32 or None.  Returns a dict with
    ``loss`` (fp32 [1]; for reduction "none" the plain sum of the per-token losses), ``n_valid``
    (int64 [1]), ``grad_input`` (bf16 [BT, H] or None), ``grad_W`` (fp32 [V, H] or None),
    ``grad_bias`` (fp32 [V] or None), ``loss_per_token`` (fp32 [BT], for reduction "none" or when
    ``want_loss_per_token``; else None) and ``entropy`` (fp32 [BT], the entropy of each row's softmax,
    when ``want_entropy``; else None).  ``out`` may supply preallocated outputs with the same keys;
    ``workspace`` a uint8 CUDA tensor of at least ``workspace_size`` bytes.

    ``grad_scale`` multiplies every gradient; ``grad_loss_per_token`` (fp32 [BT], reduction "none"
    only) is the upstream gradient of each token's loss; ``accumulate`` adds the gradients to the
    tensors given in ``out`` instead of overwriting them; ``filter_eps`` > 0 turns on gradient filtering
    (GEMM2 of dS blocks whose entries are all below it is skipped; see include/flce.h for the error
    bound); ``sort_vocab`` runs every pass on the vocabulary sorted by average logit (adds ``logit_avg``,
    fp32 [V], and ``vocab_order``, int32 [V], to the result); ``separate_lse_pass`` computes the LSE in a
    pass of its own first instead of inside the grad_input pass; ``vocab_splits`` sets how that pass splits
    the vocabulary of its row blocks (0 automatic, 1 never, k >= 2 up to k parts each), ``token_splits`` the
    same for the grad_W pass over token ranges (flce_fwd_bwd_ex).  ``debug_stall_us`` (test-only) makes the
    gradient passes' bounded waits give up on purpose (FLCE_STATUS_TIMEOUT; results invalid).
    ``pass_events``: five
    recorded ``torch.cuda.Event(enable_timing=True)`` objects; the library re-records them at the pass
    boundaries (flce_fwd_bwd_timed) for per-kernel timing; only with the default options.
    """
    import torch
    _bf16_ptr_ok(hidden, "hidden")
    _bf16_ptr_ok(W, "W")
    BT, H = hidden.shape
    V, H2 = W.shape
    if H2 != H or target.shape != (BT,) or target.dtype != torch.int64 or not target.is_cuda:
        raise ValueError("shapes must be hidden [BT, H], W [V, H], target [BT] int64 on the GPU")
    if bias is not None and (bias.dtype != torch.float32 or bias.shape != (V,) or not bias.is_cuda):
        raise ValueError("bias must be a CUDA float32 tensor of shape [V]")
    if grad_loss_per_token is not None and (grad_loss_per_token.dtype != torch.float32 or
                                            grad_loss_per_token.shape != (BT,) or not grad_loss_per_token.is_cuda
                                            or not grad_loss_per_token.is_contiguous()):
        raise ValueError("grad_loss_per_token must be a contiguous CUDA float32 tensor of shape [BT]")
    red = REDUCTIONS[reduction]
    dev = hidden.device
    o = dict(out or {})
    if "loss" not in o:
        o["loss"] = torch.empty(1, dtype=torch.float32, device=dev)
    if "n_valid" not in o:
        o["n_valid"] = torch.empty(1, dtype=torch.int64, device=dev)
    if (reduction == "none" or want_loss_per_token) and o.get("loss_per_token") is None:
        o["loss_per_token"] = torch.empty(BT, dtype=torch.float32, device=dev)
    if want_entropy and o.get("entropy") is None:
        o["entropy"] = torch.empty(BT, dtype=torch.float32, device=dev)
    if accumulate and ((need_grad_input and o.get("grad_input") is None) or (need_grad_W and o.get("grad_W") is None)
                       or (need_grad_W and bias is not None and o.get("grad_bias") is None)):
        raise ValueError("accumulate needs the gradient tensors to add to in `out`")
    if need_grad_input and o.get("grad_input") is None:
        o["grad_input"] = torch.empty((BT, H), dtype=torch.bfloat16, device=dev)
    if need_grad_W and o.get("grad_W") is None:
        o["grad_W"] = torch.empty((V, H), dtype=torch.float32, device=dev)
    if need_grad_W and bias is not None and o.get("grad_bias") is None:
        o["grad_bias"] = torch.empty(V, dtype=torch.float32, device=dev)
    gi = o.get("grad_input") if need_grad_input else None
    gw = o.get("grad_W") if need_grad_W else None
    gb = o.get("grad_bias") if (need_grad_W and bias is not None) else None
    lt = o.get("loss_per_token")
    ent = o.get("entropy") if want_entropy else None
    if sort_vocab:
        if o.get("logit_avg") is None:
            o["logit_avg"] = torch.empty(V, dtype=torch.float32, device=dev)
        if o.get("vocab_order") is None:
            o["vocab_order"] = torch.empty(V, dtype=torch.int32, device=dev)
    la = o.get("logit_avg") if sort_vocab else None
    vo = o.get("vocab_order") if sort_vocab else None
    need = workspace_size(BT, H, V, sort_vocab=sort_vocab)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device=dev)
    args = (_ptr(hidden), _ptr(W), _ptr(bias), _ptr(target), BT, H, V, ignore_index, red, float(z_loss),
            _ptr(o["loss"]), _ptr(gi), _ptr(gw), _ptr(gb), _ptr(o["n_valid"]), _ptr(workspace), workspace.numel())
    plain = (red != 2 and grad_scale == 1.0 and grad_loss_per_token is None and not accumulate and lt is None
             and ent is None and filter_eps == 0.0 and not sort_vocab and not separate_lse_pass
             and vocab_splits == 0 and token_splits == 0 and debug_stall_us == 0)
    if pass_events is not None:
        if not plain:
            raise ValueError("pass_events only with the default options")
        if len(pass_events) != 5:
            raise ValueError("pass_events needs exactly 5 events")
        handles = (c_p * 5)(*[ev.cuda_event for ev in pass_events])
        check(load().flce_fwd_bwd_timed(*args, _stream_ptr(stream), handles, 5))
    elif plain:
        check(load().flce_fwd_bwd(*args, _stream_ptr(stream)))
    else:
        opts = FwdBwdOptions(float(grad_scale), _ptr(grad_loss_per_token), _ptr(lt), 1 if accumulate else 0, _ptr(ent),
                             float(filter_eps), 1 if sort_vocab else 0, _ptr(la), _ptr(vo),
                             1 if separate_lse_pass else 0, int(vocab_splits), int(token_splits),
                             int(debug_stall_us))
        check(load().flce_fwd_bwd_ex(*args, ctypes.byref(opts), _stream_ptr(stream)))
    res = dict(loss=o["loss"], n_valid=o["n_valid"], grad_input=gi, grad_W=gw, grad_bias=gb, loss_per_token=lt,
               entropy=ent, workspace=workspace)
    if sort_vocab:
        res["logit_avg"] = la
        res["vocab_order"] = vo
    return res


def _ce_dtype(t) -> int:
    import torch
    codes = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
    if t.dtype not in codes or not t.is_cuda or not t.is_contiguous() or t.dim() != 2:
        raise ValueError("logits must be a contiguous 2-D CUDA bfloat16, float16 or float32 tensor")
    return codes[t.dtype]


def _ce_call(logits, dlogits, labels, ignore_index, z_loss, workspace, out, stream) -> dict:
    import torch
    dtype = _ce_dtype(logits)
    B, V = logits.shape
    if labels.shape != (B,) or labels.dtype != torch.int64 or not labels.is_cuda:
        raise ValueError("labels must be a CUDA int64 tensor of shape [B]")
    dev = logits.device
    o = dict(out or {})
    for k, dt in (("ce_sum", torch.float32), ("z_sum", torch.float32), ("n_valid", torch.int64)):
        if k not in o:
            o[k] = torch.empty(1, dtype=dt, device=dev)
    if workspace is None:
        workspace = torch.empty(ce_workspace_size(B, V), dtype=torch.uint8, device=dev)
    if dtype == 0 and dlogits is not None and dlogits.data_ptr() == logits.data_ptr():
        check(load().ce_with_grad(_ptr(logits), _ptr(labels), B, V, ignore_index, float(z_loss), _ptr(o["ce_sum"]),
                                  _ptr(o["z_sum"]), _ptr(o["n_valid"]), _ptr(workspace), workspace.numel(),
                                  _stream_ptr(stream)))
    else:
        check(load().ce_with_grad_ex(_ptr(logits), _ptr(dlogits), dtype, _ptr(labels), B, V, ignore_index,
                                     float(z_loss), _ptr(o["ce_sum"]), _ptr(o["z_sum"]), _ptr(o["n_valid"]),
                                     _ptr(workspace), workspace.numel(), _stream_ptr(stream)))
    return dict(ce_sum=o["ce_sum"], z_sum=o["z_sum"], n_valid=o["n_valid"], workspace=workspace)


def ce_with_grad(logits, labels, ignore_index: int = -100, z_loss: float = 0.0, workspace=None, out=None,
                 stream=None) -> dict:
    """Row-wise CE over logits [B, V] (bf16, fp16 or fp32); overwrites ``logits`` with dlogits in place.

    Returns ``ce_sum`` (fp32 [1]), ``z_sum`` (fp32 [1]) and ``n_valid`` (int64 [1]).
    """
    return _ce_call(logits, logits, labels, ignore_index, z_loss, workspace, out, stream)


def cross_entropy(logits, labels, ignore_index: int = -100, z_loss: float = 0.0, want_grad: bool = True,
                  workspace=None, out=None, stream=None) -> dict:
    """Non-mutating form of ce_with_grad: the logits are left unchanged and dlogits (same dtype and shape)
    is returned as a new tensor (or written into ``out["dlogits"]``), or not computed at all when
    ``want_grad`` is False.  Returns ``ce_sum``, ``z_sum``, ``n_valid`` and ``dlogits`` (or None)."""
    import torch
    o = dict(out or {})
    dl = None
    if want_grad:
        dl = o.get("dlogits")
        if dl is None:
            dl = torch.empty_like(logits)
        elif dl.dtype != logits.dtype or dl.shape != logits.shape or not dl.is_contiguous():
            raise ValueError("out['dlogits'] must match the logits' dtype and shape")
    r = _ce_call(logits, dl, labels, ignore_index, z_loss, workspace, o, stream)
    r["dlogits"] = dl
    return r


def ce_reduce_loss(ce_sum, z_sum, n_valid, z_loss: float = 0.0, reduction: str = "mean", loss=None,
                   stream=None):
    """The reduced loss of the standalone CE from its device sums (ce_reduce_loss of include/flce.h):
    (ce_sum + z_loss z_sum) / max(n_valid, 1) for "mean", ce_sum + z_loss z_sum for "sum".  Returns a
    fp32 [1] CUDA tensor (``loss`` if given)."""
    import torch
    if reduction not in ("mean", "sum"):
        raise ValueError("reduction must be 'mean' or 'sum'")
    if loss is None:
        loss = torch.empty(1, dtype=torch.float32, device=ce_sum.device)
    check(load().ce_reduce_loss(_ptr(ce_sum), _ptr(z_sum), _ptr(n_valid), float(z_loss), REDUCTIONS[reduction],
                                _ptr(loss), _stream_ptr(stream)))
    return loss


def scale_gradient_(grad, upstream, divisor=None, stream=None):
    """grad *= upstream / max(divisor, 1) in place, with ``upstream`` a fp32 CUDA scalar tensor and
    ``divisor`` an int64 CUDA scalar tensor or None (flce_scale_gradient of include/flce.h).  ``grad``:
    a contiguous CUDA bf16, fp16 or fp32 tensor.  Returns ``grad``."""
    import torch
    codes = {torch.bfloat16: 0, torch.float16: 1, torch.float32: 2}
    if grad.dtype not in codes or not grad.is_cuda or not grad.is_contiguous():
        raise ValueError("grad must be a contiguous CUDA bfloat16, float16 or float32 tensor")
    if upstream.dtype != torch.float32 or upstream.numel() != 1 or not upstream.is_cuda:
        raise ValueError("upstream must be a CUDA float32 scalar tensor")
    if divisor is not None and (divisor.dtype != torch.int64 or divisor.numel() != 1 or not divisor.is_cuda):
        raise ValueError("divisor must be a CUDA int64 scalar tensor")
    up = upstream.contiguous()
    check(load().flce_scale_gradient(_ptr(grad), codes[grad.dtype], grad.numel(), _ptr(up), _ptr(divisor),
                                     _stream_ptr(stream)))
    return grad


def read_filter_skips(workspace) -> int:
    """dS blocks whose GEMM2 the gradient filter skipped in the last flce_fwd_bwd on this workspace
    (the 32-bit word at byte 20; synchronises the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[20:24].cpu().view(torch.int32).item())


def read_vocab_split_units(workspace) -> int:
    """Vocabulary-split clusters the grad_input pass of the last flce_fwd_bwd on this workspace ran
    (the 32-bit word at byte 28; synchronises the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[28:32].cpu().view(torch.int32).item())


def read_token_split_units(workspace) -> int:
    """Token-split clusters the grad_W pass of the last flce_fwd_bwd on this workspace ran (the 32-bit
    word at byte 32; synchronises the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[32:36].cpu().view(torch.int32).item())


def read_side_launches(workspace) -> int:
    """Launches of side clusters (two pairs) that ran beside the persistent four-pair clusters in the last
    flce_fwd_bwd on this workspace, one per pass that used them (the 32-bit word at byte 56; synchronises
    the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[56:60].cpu().view(torch.int32).item())


def read_side_clusters(workspace) -> int:
    """Side clusters that took at least one unit in the last flce_fwd_bwd on this workspace, over both
    passes (the 32-bit word at byte 60; synchronises the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[60:64].cpu().view(torch.int32).item())


def read_single_launches(workspace) -> int:
    """Launches of single-pair clusters that ran beside the persistent four-pair and side clusters in the
    last flce_fwd_bwd on this workspace, one per pass that used them (the 32-bit word at byte 72;
    synchronises the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[72:76].cpu().view(torch.int32).item())


def read_single_clusters(workspace) -> int:
    """Single-pair clusters that took at least one unit in the last flce_fwd_bwd on this workspace, over
    both passes (the 32-bit word at byte 76; synchronises the device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return int(workspace[76:80].cpu().view(torch.int32).item())


def read_single_units(workspace) -> list:
    """Units (one row pair, two H chunks) the single-pair clusters took in the last flce_fwd_bwd on this
    workspace: [grad_input pass, grad_W pass] (the 32-bit words at bytes 64 and 68; synchronises the
    device)."""
    import torch
    torch.cuda.synchronize(workspace.device)
    return [int(x) for x in workspace[64:72].cpu().view(torch.int32).tolist()]


def read_device_status(workspace, stream=None) -> int:
    """Status word of a workspace after the call that used it (synchronises the stream)."""
    v = ctypes.c_uint32(0)
    check(load().flce_read_device_status(_ptr(workspace), ctypes.byref(v), _stream_ptr(stream)))
    return int(v.value)
