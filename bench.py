#!/usr/bin/env python
"""Benchmark of the fused linear cross-entropy library on one GB300 (or N independent replicas).

One step = one flce_fwd_bwd call (every pass: LSE tiles, merge, loss reduction, grad_input pass,
grad_W pass) over one batch of the long-batch LM-head workload (BT=65535, H=1024, V=176245, bf16,
seeded synthetic inputs, mean reduction).  Prints ONE JSON line on rank 0.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference] [--workload NAME]

Timing: W untimed steps, then K steps bracketed by a barrier and torch.cuda.synchronize() on both
sides, measured with CUDA events on the launching stream; the maximum over ranks is reported.
The inputs (hidden 128 MiB + W 344 MiB) are larger than the 126 MB L2, so no explicit flush is done.
Per-kernel times come from CUDA events the library records at its pass boundaries inside the same
timed region (flce_fwd_bwd_timed).  ``--impl reference`` times the fp64 CPU oracle instead, on
bounded row samples of the same workload.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from linear_cross_entropy_tma_gb300 import workloads as wl  # noqa: E402

# verl _Split_Dlogits_N, tuned: 356 ms fwd+bwd at BT=65535, H=1024, V=176245 on an H100 ("Fused Linear
# Cross-Entropy", "Putting numbers on it") -> 65535 / 0.356 s tokens/s.  Another machine: context only.
PAGES_TOKENS_PER_S = {"long": 65535 / 0.356}
KERNELS_PER_STEP = 5  # lse_partial, lse_merge, loss_reduce, dgrad(grad_input), dgrad(grad_W); the two dgrad passes are one launch when both run
# online flow: bias table, count, grad_input pass with the LSE, loss reduction, four gated classic kernels
# (launched, exit at once unless the online pass asked for them), grad_W pass; plus the merge of the
# vocabulary-split clusters when the grad_input pass splits its last wave (and the same for the grad_W
# pass's token-split clusters), and one launch of side clusters per pass that runs them
KERNELS_PER_STEP_ONLINE = 9


def pairs_per_cluster(h_chunks: int, n_blocks: int, side: bool) -> int:
    """CTA pairs per cluster of an exact gradient pass, as the library picks them (four when the 256-wide
    H chunks divide by 4 and a unit runs over at least 64 column blocks, or at least 16 when the pass ran
    with side clusters; else two, three or one)."""
    if h_chunks % 4 == 0 and (n_blocks >= 64 or (side and n_blocks >= 16)):
        return 4
    return 2 if h_chunks % 2 == 0 else 3 if h_chunks % 3 == 0 else 1


def pass_tflops(w, passes, queues, single_units):
    """Algorithmic (logits + one GEMM, 4*BT*V*H) and executed TFLOP/s of the two gradient passes of the
    default flow.  Executed counts the logits once per cluster that covers a row block: h_chunks / P times
    per row block (P pairs per cluster), once per side unit (two H chunks) the two-pair side clusters
    took, and twice per side unit the single-pair clusters took (one chunk at a time)."""
    h_chunks = -(-w.H // 256)
    out = {}
    for name, rows, cols, q, su in (("dgrad_grad_input_online", w.BT, w.V, queues[0], single_units[0]),
                                    ("dgrad_grad_W", w.V, w.BT, queues[1], single_units[1])):
        rp = -(-rows // 256)
        side_units = q >> 32
        P = pairs_per_cluster(h_chunks, -(-cols // 256), side_units > 0)
        if P != 4:
            side_units = su = 0
        side_rp = side_units // (h_chunks // 2)
        g1 = ((rp - side_rp) * (h_chunks // P) + (side_units - su) + 2 * su) / rp
        gemm = 2.0 * w.BT * w.V * w.H
        sec = passes[name] * 1e-3
        out[name] = {"algorithmic": 2 * gemm / sec / 1e12, "executed": (g1 + 1) * gemm / sec / 1e12,
                     "logits_computed_per_row_block": g1, "pairs_per_cluster": P, "side_row_blocks": side_rp,
                     "single_pair_units": su}
    return out


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm_gbs=d["hbm_gbs"], bf16_tflops=d["bf16_tflops"],
                    bf16_tflops_sustained=d.get("bf16_tflops_sustained", d["bf16_tflops"]), source="measured")
    return dict(hbm_gbs=6800.0, bf16_tflops=1900.0, bf16_tflops_sustained=1700.0, source="fallback")


def strip_comments(src: str) -> str:
    """C/CUDA source without its comments, every run of white space made one space (string and character
    literals kept), so that a digest of it changes with the code's tokens only."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            i = n if j < 0 else j + 2
        elif c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def kernel_source_digest(files):
    """Digest of the kernel sources' code (comments and layout stripped): the key under which
    profiles/traffic.json stores the DRAM counters taken on that code."""
    h = hashlib.sha256()
    for f in files:
        with open(os.path.join(ROOT, "linear_cross_entropy_tma_gb300", "csrc", f), encoding="utf-8") as fh:
            h.update(strip_comments(fh.read()).encode())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, workload: str, src_digest: str):
    """Per-launch DRAM bytes of a kernel from the committed ncu summary, if the kernel source has not
    changed since the counters were taken; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        d = json.load(f)
    e = d.get(workload, {}).get(kernel)
    if not e or e.get("source_digest") != src_digest:
        return None
    return e["dram_bytes_per_launch"]


class ClockSampler:
    """nvidia-smi clock / throttle sampling (200 ms) while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.out = None

    def start(self):
        try:
            self.out = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-i", str(self.gpu), "-lms", "200"], stdout=self.out,
                                         stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.out.flush()
        with open(self.out.name) as f:
            rows = [r.strip().split(", ") for r in f if r.strip()]
        os.unlink(self.out.name)
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for r in rows:
            if len(r) < 9:
                continue
            try:
                sm.append(float(r[1]))
                mx.append(float(r[2]))
            except ValueError:
                continue
            for name, val in zip(names, r[5:9]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_info():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x: float, world: int) -> float:
    if world == 1:
        return x
    import torch
    import torch.distributed as dist
    t = torch.tensor([x], dtype=torch.float64, device="cuda")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def to_device_bf16(bits, device):
    import numpy as np
    import torch
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).to(device)


# ----------------------------------------------------------------------------------- our arm
def bench_fused(w: wl.FusedWorkload, steps: int, warmup: int, world: int, local: int, peaks: dict,
                filter_eps: float = 0.0):
    import torch
    import linear_cross_entropy_tma_gb300 as flce

    dev = torch.device("cuda", local)
    d = wl.make_fused_inputs(w)
    hidden = to_device_bf16(d["hidden"], dev)
    W = to_device_bf16(d["W"], dev)
    target = torch.from_numpy(d["target"]).to(dev)
    bias = torch.from_numpy(d["bias"]).to(dev) if d["bias"] is not None else None
    out = {"loss": torch.empty(1, device=dev), "n_valid": torch.empty(1, dtype=torch.int64, device=dev),
           "grad_input": torch.empty((w.BT, w.H), dtype=torch.bfloat16, device=dev),
           "grad_W": torch.empty((w.V, w.H), dtype=torch.float32, device=dev)}
    if bias is not None:
        out["grad_bias"] = torch.empty(w.V, device=dev)
    ws = torch.empty(flce.workspace_size(w.BT, w.H, w.V), dtype=torch.uint8, device=dev)
    kw = dict(bias=bias, reduction=w.reduction, z_loss=w.z_loss, workspace=ws, out=out)

    def ev():
        e = torch.cuda.Event(enable_timing=True)
        e.record()
        return e

    pass_ev = [[ev() for _ in range(5)] for _ in range(steps)]
    torch.cuda.synchronize()
    torch.cuda.reset_peak_memory_stats(dev)
    for _ in range(warmup):
        flce.flce_fwd_bwd(hidden, W, target, **kw)
    torch.cuda.synchronize()
    assert flce.read_device_status(ws) == 0, "device status word non-zero after warm-up"

    sampler = ClockSampler(local)
    barrier(world)
    torch.cuda.synchronize()
    sampler.start()
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    for k in range(steps):
        flce.flce_fwd_bwd(hidden, W, target, pass_events=pass_ev[k], **kw)
    t1.record()
    torch.cuda.synchronize()
    barrier(world)
    clocks = sampler.stop()
    elapsed_ms = max_over_ranks(t0.elapsed_time(t1), world)
    peak_mem = torch.cuda.max_memory_allocated(dev)
    passes = {name: statistics.mean(pass_ev[k][i].elapsed_time(pass_ev[k][i + 1]) for k in range(steps))
              for i, name in enumerate(("lse_partial", "lse_merge+loss_reduce", "dgrad_grad_input", "dgrad_grad_W"))}
    loss = out["loss"].item()
    # vocabulary-split clusters the grad_input pass ran (its merge kernel is one more launch per step)
    split_units = flce.read_vocab_split_units(ws)
    token_split_units = flce.read_token_split_units(ws)
    # launches of side clusters beside the persistent four-pair clusters (one per pass that used them), and
    # the side clusters that took work (both passes)
    side_launches = flce.read_side_launches(ws)
    side_clusters = flce.read_side_clusters(ws)
    # the same for the single-pair clusters on the SMs where no side cluster finds room, and the units
    # (row pair, two H chunks) they took per pass
    single_launches = flce.read_single_launches(ws)
    single_clusters = flce.read_single_clusters(ws)
    single_units = flce.read_single_units(ws)
    # the two passes' work queues (workspace header bytes 40 and 48: main units | side units << 32), for the
    # executed GEMM1 work of passes that ran side clusters
    queues = [int(x) for x in ws[40:56].cpu().view(torch.int64).tolist()]

    # the same call captured once into a CUDA graph and replayed (what a training loop that captures its
    # step sees: no per-launch host overhead); same buffers, same inputs
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        flce.flce_fwd_bwd(hidden, W, target, **kw)
    graph.replay()
    torch.cuda.synchronize()
    g0 = torch.cuda.Event(enable_timing=True)
    g1 = torch.cuda.Event(enable_timing=True)
    g0.record()
    for _ in range(steps):
        graph.replay()
    g1.record()
    torch.cuda.synchronize()
    graph_ms = max_over_ranks(g0.elapsed_time(g1), world) / steps
    assert flce.read_device_status(ws) == 0, "device status word non-zero after the graph replays"
    del graph

    # end to end through the same public call from pinned host buffers: every step copies its inputs
    # host -> device, runs the call and copies the loss and both gradients device -> host.  The copies run
    # on two copy streams with double-buffered device inputs and outputs, so step k's copies overlap the
    # compute of its neighbours (a training loop's prefetch and write-back); the timed region runs from
    # the first copy in to the last copy out.  The serial form (copy in, call, copy out on one stream)
    # is reported beside it.
    h_hidden = torch.from_numpy(d["hidden"].view("int16")).pin_memory()
    h_W = torch.from_numpy(d["W"].view("int16")).pin_memory()
    h_target = torch.from_numpy(d["target"]).pin_memory()
    h_bias = torch.from_numpy(d["bias"]).pin_memory() if bias is not None else None
    r_loss = torch.empty(1).pin_memory()
    r_gi = torch.empty((w.BT, w.H), dtype=torch.int16).pin_memory()
    r_gw = torch.empty((w.V, w.H), dtype=torch.float32).pin_memory()
    r_gb = torch.empty(w.V).pin_memory() if bias is not None else None
    h2d = h_hidden.numel() * 2 + h_W.numel() * 2 + h_target.numel() * 8 + (h_bias.numel() * 4 if h_bias is not None else 0)
    d2h = 4 + r_gi.numel() * 2 + r_gw.numel() * 4 + (r_gb.numel() * 4 if r_gb is not None else 0)
    dev_in = [dict(hidden=hidden, W=W, target=target, bias=bias),
              dict(hidden=torch.empty_like(hidden), W=torch.empty_like(W), target=torch.empty_like(target),
                   bias=torch.empty_like(bias) if bias is not None else None)]
    dev_out = [out, {k: torch.empty_like(v) for k, v in out.items()}]

    def copy_in(buf):
        buf["hidden"].view(torch.int16).copy_(h_hidden, non_blocking=True)
        buf["W"].view(torch.int16).copy_(h_W, non_blocking=True)
        buf["target"].copy_(h_target, non_blocking=True)
        if h_bias is not None:
            buf["bias"].copy_(h_bias, non_blocking=True)

    def copy_out(o):
        r_loss.copy_(o["loss"], non_blocking=True)
        r_gi.copy_(o["grad_input"].view(torch.int16), non_blocking=True)
        r_gw.copy_(o["grad_W"], non_blocking=True)
        if r_gb is not None:
            r_gb.copy_(o["grad_bias"], non_blocking=True)

    def call(buf, o, stream=None):
        flce.flce_fwd_bwd(buf["hidden"], buf["W"], buf["target"], bias=buf["bias"], reduction=w.reduction,
                          z_loss=w.z_loss, workspace=ws, out=o, stream=stream)

    def e2e_serial(n):
        for _ in range(n):
            copy_in(dev_in[0])
            call(dev_in[0], dev_out[0])
            copy_out(dev_out[0])

    s_comp = torch.cuda.current_stream(dev)
    s_in = torch.cuda.Stream(dev)
    s_out = torch.cuda.Stream(dev)

    def e2e_pipelined(n, start_ev=None, end_ev=None):
        comp_done, out_done = [], []
        if start_ev is not None:
            start_ev.record(s_in)
        for k in range(n):
            buf, o = dev_in[k % 2], dev_out[k % 2]
            with torch.cuda.stream(s_in):
                if k >= 2:
                    s_in.wait_event(comp_done[k - 2])      # the call two steps back has read these inputs
                copy_in(buf)
                ready = torch.cuda.Event()
                ready.record(s_in)
            s_comp.wait_event(ready)
            if k >= 2:
                s_comp.wait_event(out_done[k - 2])         # these outputs have been copied out
            call(buf, o, stream=s_comp)
            done = torch.cuda.Event()
            done.record(s_comp)
            comp_done.append(done)
            with torch.cuda.stream(s_out):
                s_out.wait_event(done)
                copy_out(o)
                fin = torch.cuda.Event()
                fin.record(s_out)
                out_done.append(fin)
        if end_ev is not None:
            end_ev.record(s_out)

    e2e_steps = max(3, min(steps, 10))
    e2e_serial(1)
    e2e_pipelined(2)
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    e2e_serial(e2e_steps)
    b.record()
    torch.cuda.synchronize()
    barrier(world)
    e2e_serial_ms = max_over_ranks(a.elapsed_time(b), world) / e2e_steps
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    e2e_sampler = ClockSampler(local)
    e2e_sampler.start()
    e2e_pipelined(e2e_steps, start_ev=a, end_ev=b)
    torch.cuda.synchronize()
    e2e_clocks = e2e_sampler.stop()
    barrier(world)
    e2e_ms = max_over_ranks(a.elapsed_time(b), world) / e2e_steps
    del h_hidden, h_W, r_gi, r_gw, dev_in, dev_out

    # the gradient-filtering variant (not the headline: it skips GEMM2 work the exact path does)
    filt = None
    if filter_eps > 0:
        for _ in range(warmup):
            flce.flce_fwd_bwd(hidden, W, target, filter_eps=filter_eps, **kw)
        torch.cuda.synchronize()
        a.record()
        for _ in range(steps):
            flce.flce_fwd_bwd(hidden, W, target, filter_eps=filter_eps, **kw)
        b.record()
        torch.cuda.synchronize()
        f_ms = a.elapsed_time(b) / steps
        skips = flce.read_filter_skips(ws)
        hb = -(-w.H // 256)
        halves = 2 * (-(-w.BT // 256) * hb * -(-w.V // 256) + -(-w.V // 256) * hb * -(-w.BT // 256))
        filt = {"filter_eps": filter_eps, "ms_per_step": f_ms, "tokens_per_s": world * w.BT / (f_ms * 1e-3),
                "skipped_dS_blocks": skips, "skipped_fraction": skips / halves,
                "note": "CCE-style gradient filtering; error bound in include/flce.h; not the headline"}
        # the same with the vocabulary sorted by average logit first (its own workspace: + a sorted W)
        ws_sort = torch.empty(flce.workspace_size(w.BT, w.H, w.V, sort_vocab=True), dtype=torch.uint8, device=dev)
        kw_sort = dict(kw, workspace=ws_sort)
        for _ in range(warmup):
            flce.flce_fwd_bwd(hidden, W, target, filter_eps=filter_eps, sort_vocab=True, **kw_sort)
        torch.cuda.synchronize()
        a.record()
        for _ in range(steps):
            flce.flce_fwd_bwd(hidden, W, target, filter_eps=filter_eps, sort_vocab=True, **kw_sort)
        b.record()
        torch.cuda.synchronize()
        s_ms = a.elapsed_time(b) / steps
        s_skips = flce.read_filter_skips(ws_sort)
        filt["with_vocab_sort"] = {"ms_per_step": s_ms, "tokens_per_s": world * w.BT / (s_ms * 1e-3),
                                   "skipped_dS_blocks": s_skips, "skipped_fraction": s_skips / halves,
                                   "workspace_bytes": ws_sort.numel()}
        del ws_sort
    return dict(elapsed_ms=elapsed_ms, passes=passes, clocks=clocks, peak_mem=peak_mem, loss=loss, e2e_ms=e2e_ms,
                e2e_clocks=e2e_clocks,
                e2e_serial_ms=e2e_serial_ms, h2d=h2d, d2h=d2h, workspace_bytes=ws.numel(), filter=filt,
                split_units=split_units, token_split_units=token_split_units, side_launches=side_launches,
                side_clusters=side_clusters, single_launches=single_launches, single_clusters=single_clusters,
                single_units=single_units, queues=queues, graph_ms=graph_ms)


def bench_workload(w: wl.FusedWorkload, steps: int, warmup: int, local: int, peaks: dict, oracle_rows: int | None):
    """One more fused workload, timed like the headline (same call, W warm-up steps, K steps between two
    CUDA events on the launching stream, clocks sampled), and the fp64 oracle's rate on it: all BT tokens
    when oracle_rows is None, else a sample of that many tokens (labelled row-sampled)."""
    import torch
    import linear_cross_entropy_tma_gb300 as flce
    dev = torch.device("cuda", local)
    d = wl.make_fused_inputs(w)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    torch.cuda.reset_peak_memory_stats(dev)
    hidden = to_device_bf16(d["hidden"], dev)
    W = to_device_bf16(d["W"], dev)
    target = torch.from_numpy(d["target"]).to(dev)
    bias = torch.from_numpy(d["bias"]).to(dev) if d["bias"] is not None else None
    res = flce.flce_fwd_bwd(hidden, W, target, bias=bias, reduction=w.reduction, z_loss=w.z_loss)
    kw = dict(bias=bias, reduction=w.reduction, z_loss=w.z_loss, workspace=res["workspace"],
              out={k: v for k, v in res.items() if k in ("loss", "n_valid", "grad_input", "grad_W", "grad_bias")
                   and v is not None})
    for _ in range(warmup):
        flce.flce_fwd_bwd(hidden, W, target, **kw)
    torch.cuda.synchronize()
    assert flce.read_device_status(res["workspace"]) == 0, f"device status word non-zero ({w.name})"
    sampler = ClockSampler(local)
    sampler.start()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        flce.flce_fwd_bwd(hidden, W, target, **kw)
    b.record()
    torch.cuda.synchronize()
    clocks = sampler.stop()
    ms = a.elapsed_time(b) / steps
    peak = torch.cuda.max_memory_allocated(dev)
    tf = w.flops() / (ms * 1e-3) / 1e12
    del hidden, W, target, bias, res, kw
    torch.cuda.empty_cache()
    dw = widened(d)
    n = w.BT if oracle_rows is None else min(oracle_rows, w.BT)
    t = time_oracle_tokens(w, dw, n)
    return {"workload": w.name, "ms_per_step": ms, "tokens_per_s": w.BT / (ms * 1e-3), "tflops": tf,
            "frac_of_burst": tf / peaks["bf16_tflops"], "frac_of_sustained": tf / peaks["bf16_tflops_sustained"],
            "flops_per_step": w.flops(), "peak_allocated_bytes": peak, "avoided_fp32_logits_bytes": 4 * w.BT * w.V,
            "clocks": clocks,
            "oracle": {"tokens_per_s": n / t, "cores": cpu_cores(), "seconds": t,
                       "sample": "full: every token" if n == w.BT else
                                 f"row-sampled: the first {n} of {w.BT} tokens (full V and H per token)"}}


def bench_ce(steps: int, warmup: int, local: int, peaks: dict):
    import torch
    import linear_cross_entropy_tma_gb300 as flce
    w = wl.CE_LOGITS
    dev = torch.device("cuda", local)
    c = wl.make_ce_inputs(w)
    logits = to_device_bf16(c["logits"], dev)
    labels = torch.from_numpy(c["labels"]).to(dev)
    ws = torch.empty(flce.ce_workspace_size(w.B, w.V), dtype=torch.uint8, device=dev)
    out = {"ce_sum": torch.empty(1, device=dev), "z_sum": torch.empty(1, device=dev),
           "n_valid": torch.empty(1, dtype=torch.int64, device=dev)}
    # every call rewrites the buffer in place (logits -> dlogits); the work per call is the same
    for _ in range(warmup):
        flce.ce_with_grad(logits, labels, z_loss=w.z_loss, workspace=ws, out=out)
    torch.cuda.synchronize()
    a = torch.cuda.Event(enable_timing=True)
    b = torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(steps):
        flce.ce_with_grad(logits, labels, z_loss=w.z_loss, workspace=ws, out=out)
    b.record()
    torch.cuda.synchronize()
    ms = a.elapsed_time(b) / steps
    gbs = w.bytes_moved() / (ms * 1e-3) / 1e9
    src = kernel_source_digest(["ce_kernel.cu"])
    return {"workload": w.name, "value": gbs, "unit": "GB/s", "ms_per_call": ms,
            "rows_per_s": w.B / (ms * 1e-3),
            "roofline": {"bound": "hbm", "achieved": gbs, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": gbs / peaks["hbm_gbs"], "traffic": dram_traffic("ce_rows_kernel", "ce", src),
                         "peak_source": peaks["source"], "algorithmic_bytes": w.bytes_moved()}}


# ----------------------------------------------------------------------------------- oracle timing
def widened(d: dict) -> dict:
    """The inputs with W (and the bias) widened to float64 once, outside any timed region: the oracle then
    uses them as they are, so a timed call does the method's work and not a 1.4 GB conversion of W."""
    import oracle
    e = dict(d)
    e["W"] = oracle.widen(d["W"])
    e["bias"] = None if d["bias"] is None else oracle.widen(d["bias"])
    return e


def time_oracle_tokens(w: wl.FusedWorkload, d: dict, n_rows: int, offset: int = 0):
    """Seconds the fp64 oracle takes for the full loss + gradient work of n_rows tokens (d from widened())."""
    import oracle
    rows = slice(offset, offset + n_rows)
    t = time.perf_counter()
    oracle.flce_reference(d["hidden"][rows], d["W"], d["target"][rows], bias=d["bias"], reduction=w.reduction,
                          z_loss=w.z_loss, row_block=min(n_rows, 256))
    return time.perf_counter() - t


def cpu_cores():
    n = len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()
    for var in ("OPENBLAS_NUM_THREADS", "OMP_NUM_THREADS"):
        if os.environ.get(var):
            n = min(n, int(os.environ[var]))
    return n


def cpu_baseline(w: wl.FusedWorkload, target_s: float = 12.0):
    d = widened(wl.make_fused_inputs(w))
    time_oracle_tokens(w, d, 32)
    t256 = time_oracle_tokens(w, d, 256)
    n = int(max(256, min(w.BT - 64, 256 * target_s / max(t256, 1e-3))))
    t = time_oracle_tokens(w, d, n, offset=64)
    return {"value": n / t, "unit": "tokens/s", "cores": cpu_cores(), "kind": "oracle",
            "sample": f"fp64 oracle, full loss + grad_input + grad_W work for {n} of the {w.BT} tokens "
                      f"(rows 64..{64 + n - 1}), full V={w.V} and H={w.H}; {t:.1f} s (W widened to fp64 once, "
                      f"before timing)"}


def run_reference(args, w):
    rank, world, local = dist_info()
    if rank != 0:
        return 0
    d = widened(wl.make_fused_inputs(w))
    # 512 tokens a step (about 2.5 s of the oracle on 16 cores at the long workload): enough that its fixed
    # cost per call (the zeroed fp64 grad_W, V x H) is small beside the per-token work, as in cpu_baseline
    per_step = min(512, max(1, w.BT))
    for k in range(args.warmup):
        time_oracle_tokens(w, d, per_step, offset=(k * per_step) % max(1, w.BT - per_step))
    times = []
    for k in range(args.steps):
        times.append(time_oracle_tokens(w, d, per_step, offset=((args.warmup + k) * per_step) % max(1, w.BT - per_step)))
    total = sum(times)
    value = per_step * args.steps / total
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": config_of(w),
            "cpu_baseline": {"value": value, "unit": "tokens/s", "kind": "oracle", "cores": cpu_cores(),
                             "sample": f"each step: the fp64 oracle's full per-token work for {per_step} tokens of the "
                                       f"workload (rows advance each step), full V and H"},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


METRIC = "fused LM-head CE fwd+bwd tokens/s & % bf16 tensor peak; CE-only GB/s % HBM"


def config_of(w):
    return {"workload": w.name, "BT": w.BT, "H": w.H, "V": w.V, "reduction": w.reduction, "z_loss": w.z_loss,
            "bias": w.bias_std is not None, "targets": w.targets,
            "l2": "no flush: hidden + W (472 MiB at this shape) exceed the 126 MB L2",
            "parallelism": "independent replica per GPU"}


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--workload", choices=sorted(wl.FUSED_WORKLOADS), default="long")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-ce", action="store_true")
    ap.add_argument("--no-workloads", action="store_true", help="skip the other fused workloads")
    ap.add_argument("--tokens", type=int, default=0,
                    help="run the workload with this BT instead (a smaller case of the same shape; not the headline)")
    ap.add_argument("--filter-eps", type=float, default=2.0 ** -12,
                    help="also time the gradient-filtering variant at this threshold (0: skip)")
    args = ap.parse_args()
    w = wl.FUSED_WORKLOADS[args.workload]
    if args.tokens:
        # a smaller case of the same shape (for profiler captures): the first N tokens' worth of the workload
        import dataclasses
        w = dataclasses.replace(w, name=f"{w.name}, BT reduced to {args.tokens}", BT=args.tokens)
    if args.warmup < 3:
        raise SystemExit("--warmup must be at least 3")
    if args.impl == "reference":
        return run_reference(args, w)

    import torch
    rank, world, local = dist_info()
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    else:
        torch.cuda.set_device(local)
    import linear_cross_entropy_tma_gb300 as flce
    flce.load()
    peaks = load_peaks()

    r = bench_fused(w, args.steps, args.warmup, world, local, peaks, filter_eps=args.filter_eps)
    ms = r["elapsed_ms"] / args.steps
    value = world * w.BT / (ms * 1e-3)
    passes = r["passes"]
    # which flow ran: the timed calls request grad_input with default options, so the library takes the
    # flow whose grad_input pass finds the LSE itself (its first interval holds two small kernels) whenever
    # there are tokens; in the classic flow both gradient passes are one launch when both run (the grad_W
    # event is then recorded right after the grad_input one): report that launch as one kernel
    online = w.BT > 0
    merged = not online and passes["dgrad_grad_W"] < 0.01 * passes["dgrad_grad_input"]
    if online:
        passes = {"online_prep": passes["lse_partial"], "dgrad_grad_input_online": passes["lse_merge+loss_reduce"],
                  "loss_reduce+gated_classic": passes["dgrad_grad_input"], "dgrad_grad_W": passes["dgrad_grad_W"]}
    if merged:
        passes = {"lse_partial": passes["lse_partial"], "lse_merge+loss_reduce": passes["lse_merge+loss_reduce"],
                  "dgrad_both_passes": passes["dgrad_grad_input"] + passes["dgrad_grad_W"]}
    tensor_kernels = [k for k in ("lse_partial", "dgrad_grad_input", "dgrad_grad_W", "dgrad_both_passes",
                                  "dgrad_grad_input_online") if k in passes]
    dominant = max(tensor_kernels, key=lambda k: passes[k])
    # algorithmic work per launch of each tensor-core kernel: logits 2*BT*V*H; each gradient pass
    # recomputes the logits (2*BT*V*H) and runs its GEMM (2*BT*V*H)
    alg = {"lse_partial": 2 * w.BT * w.V * w.H, "dgrad_grad_input": 4 * w.BT * w.V * w.H,
           "dgrad_grad_W": 4 * w.BT * w.V * w.H, "dgrad_both_passes": 8 * w.BT * w.V * w.H,
           "dgrad_grad_input_online": 4 * w.BT * w.V * w.H}
    kname = {"lse_partial": "lse_pair_kernel", "dgrad_grad_input": "dgrad_pair_kernel<false>",
             "dgrad_grad_W": "dgrad_pair_kernel<true>", "dgrad_both_passes": "dgrad_both_kernel",
             "dgrad_grad_input_online": "dgrad_online_kernel"}
    src = kernel_source_digest(["flce_fwd.cu", "flce_bwd.cu", "sm100.cuh"])
    peak_tf = peaks["bf16_tflops_sustained"]
    achieved = alg[dominant] / (passes[dominant] * 1e-3) / 1e12
    step_tflops = w.flops() / (ms * 1e-3) / 1e12
    line = {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": (value / world) / PAGES_TOKENS_PER_S[args.workload]
        if args.workload in PAGES_TOKENS_PER_S and not args.tokens else None,
        "vs_baseline_note": "value per GPU / verl tuned _Split_Dlogits_N on an H100 (356 ms, pages' table); context only",
        "dtype": "bf16", "data": "synthetic (seeded; hidden N(0,1), W N(0,0.02), uniform targets, 10% ignored)",
        "config": config_of(w),
        "roofline": {"bound": "tensor", "kernel": kname[dominant], "achieved": achieved, "peak": peak_tf,
                     "unit": "TFLOP/s", "frac": achieved / peak_tf, "traffic": dram_traffic(kname[dominant], args.workload, src),
                     "peak_source": f"{peaks['source']} bf16_tflops_sustained (kernel timed inside a long step)",
                     "algorithmic_flops_per_launch": alg[dominant], "ms_per_launch": passes[dominant]},
        "step_roofline": {"flops_per_step": w.flops(), "achieved_tflops": step_tflops,
                          "frac_of_sustained": step_tflops / peak_tf, "frac_of_burst": step_tflops / peaks["bf16_tflops"],
                          "convention": "8*BT*V*H per fused forward+backward"},
        "pass_ms": passes,
        "pass_tflops": pass_tflops(w, passes, r["queues"], r["single_units"]) if online else None,
        "gpu_launches": ((KERNELS_PER_STEP_ONLINE + (1 if r["split_units"] else 0)) if online
                         else KERNELS_PER_STEP - 1 if merged else KERNELS_PER_STEP)
                        * args.steps + (args.steps if r["token_split_units"] else 0)
                        + (r["side_launches"] + r["single_launches"]) * args.steps,
        "graph_replay": {"ms_per_step": r["graph_ms"], "tokens_per_s": world * w.BT / (r["graph_ms"] * 1e-3),
                         "note": "the same call captured once into a CUDA graph, replayed steps times"},
        "vocab_split_clusters": r["split_units"],
        "token_split_clusters": r["token_split_units"],
        "side_launches_per_step": r["side_launches"],
        "side_clusters_with_work_per_step": r["side_clusters"],
        "single_pair_launches_per_step": r["single_launches"],
        "single_pair_clusters_with_work_per_step": r["single_clusters"],
        "clocks": r["clocks"],
        "e2e": {"value": world * w.BT / (r["e2e_ms"] * 1e-3), "unit": "tokens/s", "h2d_bytes_per_step": r["h2d"],
                "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e_ms"],
                "copies": "double-buffered on two copy streams, overlapping the neighbouring steps' compute",
                "ms_per_step_serial": r["e2e_serial_ms"], "clocks": r["e2e_clocks"]},
        "memory": {"peak_allocated_bytes": r["peak_mem"], "workspace_bytes": r["workspace_bytes"],
                   "avoided_fp32_logits_bytes": 4 * w.BT * w.V},
        "loss": r["loss"],
        "filter_variant": r["filter"],
    }
    if not args.no_ce and world == 1:
        line["ce_standalone"] = bench_ce(args.steps, args.warmup, local, peaks)
    if not args.no_workloads and world == 1:
        # the other fused workloads in the same run (the headline value stays on this one); the oracle in
        # full for the two small ones, row-sampled for the large ones
        others = {"tiny": None, "qwen3": None, "gemma2": 256, "long": 256}
        line["workloads"] = {k: bench_workload(wl.FUSED_WORKLOADS[k], args.steps, args.warmup, local, peaks, rows)
                             for k, rows in others.items() if k != args.workload}
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(w)
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
