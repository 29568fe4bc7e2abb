#!/usr/bin/env python3
"""Benchmark of the DiT attention hot path on GB300.

One step = the whole path on one batch of synthetic input, resident in HBM,
as one dit_attention call: QK-RMSNorm + interleaved RoPE on Q and K, flash
attention over the workload's KV chunks, and the LSE merge (in the last
chunk's epilogue, or by the merge kernel over stacked partials).  Default
workload: Qwen-Image joint attention (B1 H24 D128 S4312 = 256 text + 78x52
image tokens), KV in 2 chunks.

Timing: the step region records events around whole steps only (events
between a step's kernels would stall the stream); roofline.achieved comes
from a second region of the same steps whose events bracket the attention
launches; e2e runs the public host-buffer call with the copies inside the
timed region.

Prints one JSON line (rank 0).  `--impl reference` times the fp64 CPU oracle
(the only reference this method has) on a bounded sample of the same workload.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl ours|reference]
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time
from pathlib import Path

import numpy as np

ROOT = Path(__file__).resolve().parent
sys.path.insert(0, str(ROOT))

from diffusion_transformer_attention_dit_gb300 import inputs  # noqa: E402

METRIC = "attention TFLOP/s (4·B·H·Sq·Skv·D/t) and % of GB300 dense bf16 peak"
FALLBACK_TFLOPS = 1900.0
FALLBACK_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
ATTN_TIMED_STEPS = 1000  # steps of the separate attention-timing region (roofline.achieved)
PARTIAL = {"tiny": "f32", "qwen_image": "f32", "qwen_image_edit": "f32", "wan480": "f32", "wan720": "bf16"}
# How the KV chunks are combined: "update" folds each later chunk into the running (O, LSE) in its attention
# epilogue; "kernel" writes stacked per-chunk partials and runs the LSE-merge kernel (Wan720's workload
# specifies per-chunk bf16 partials merged by the merge kernel).
MERGE = {"tiny": "update", "qwen_image": "update", "qwen_image_edit": "update", "wan480": "kernel",
         "wan720": "kernel"}
# DRAM bytes (read + write) of the attention launches of one bench step, from an ncu capture
# (profiles/launch_list_qwen_image_step.md): chunk 0 (fp32 running O) and chunk 1 (update form,
# bf16 O), averaged per launch; valid for the attention source it was taken on.
ATTN_TRAFFIC = {"source_sha256_prefix": "5f5d8b30479990a5",
                "qwen_image": ((30.54 + 56.23) + (97.52 + 58.01)) / 2 * 1e6}


def peaks():
    path = ROOT / "MEASURED_PEAKS.json"
    if path.exists():
        try:
            d = json.loads(path.read_text())
            tf = d.get("bf16_tflops") or d.get("bf16_tflops_burst")
            gbs = d.get("hbm_gbs") or d.get("hbm_GBs")
            if tf and gbs:
                return float(tf), float(gbs), "measured"
        except (ValueError, OSError):
            pass
    return FALLBACK_TFLOPS, FALLBACK_GBS, "fallback"


class ClockSampler:
    """nvidia-smi samples (every 200 ms) taken while the timed region runs."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.lines: list[str] = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", "200"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        rows = [l.split(", ") for l in self.lines if l]
        if self.uuid:
            mine = [r for r in rows if r and self.uuid in r[0]]
            rows = mine or rows
        sm, smax, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm)}


# ----------------------------------------------------------------------------- CPU oracle (reference arm)

def oracle_step(inp, rows: np.ndarray, chunks: int):
    """The hot path on the CPU oracle for a sample of query rows (all heads, all keys): prologue, chunked attention, merge."""
    import oracle

    orc = oracle.get()
    w = inp.w
    c64, s64 = inp.cos.astype(np.float64), inp.sin.astype(np.float64)
    q = inputs.bf16_bits_to_f64(inp.q[:, rows])
    k = inputs.bf16_bits_to_f64(inp.k)
    v = inputs.bf16_bits_to_f64(inp.v)
    if w.prologue:
        q = oracle.round_bf16(orc.qk_norm_rope(q, inp.wq.astype(np.float64), c64[rows], s64[rows], w.eps))
        k = oracle.round_bf16(orc.qk_norm_rope(k, inp.wk.astype(np.float64), c64, s64, w.eps))
    parts = [orc.attention(q, k, v, w.scale, lo, hi) for lo, hi in w.chunk_bounds(chunks)]
    return orc.merge_lse(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))


def cpu_sample_rows(w, n: int) -> np.ndarray:
    return np.linspace(0, w.S - 1, n).round().astype(np.int64)


def cpu_baseline(inp, chunks: int, budget_s: float = 15.0):
    """Time the oracle on growing row samples until about budget_s of CPU work has been measured."""
    import oracle

    w = inp.w
    n, total_t, total_f = 16, 0.0, 0.0
    while True:
        rows = cpu_sample_rows(w, min(n, w.S))
        t0 = time.perf_counter()
        oracle_step(inp, rows, chunks)
        dt = time.perf_counter() - t0
        total_t += dt
        total_f += 4.0 * w.B * w.H * len(rows) * w.S * w.D
        if total_t >= budget_s or n >= w.S:
            break
        n = min(w.S, max(2 * n, int(n * budget_s / max(dt, 1e-3) / 2)))
    return {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{w.name}: prologue on all keys + attention over {chunks} KV chunks + merge for evenly spaced "
                      f"query rows (all {w.H} heads, all {w.S} keys), row counts doubling to {len(rows)}; "
                      f"{total_t:.1f} s of fp64 C/OpenMP work in total"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    inp = inputs.make_inputs(args.workload)
    w = inp.w
    chunks = args.chunks or w.chunks
    rows = cpu_sample_rows(w, args.ref_rows)
    for _ in range(args.warmup):
        oracle_step(inp, rows, chunks)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle_step(inp, rows, chunks)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.B * w.H * len(rows) * w.S * w.D * args.steps
    value = flops / dt / 1e12
    sample = (f"{w.name}: {len(rows)} evenly spaced query rows per (b, h) against all {w.S} keys; prologue, "
              f"{chunks} KV chunks and merge on the fp64 oracle")
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": config_of(w, chunks, args),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }))


def merge_mode(w, args):
    return args.merge if args.merge != "auto" else MERGE[w.name]


def config_of(w, chunks, args):
    return {"workload": w.description, "name": w.name, "B": w.B, "H": w.H, "D": w.D, "Sq": w.S, "Skv": w.S,
            "kv_chunks": chunks, "partial_o": PARTIAL[w.name],
            "merge": (merge_mode(w, args) + (" (fused in the last chunk's epilogue)" if merge_mode(w, args) == "update"
                                             else " (LSE-merge kernel)")) if chunks > 1 else "none",
            "prologue": w.prologue, "causal": False,
            "launch_overlap": not getattr(args, "no_launch_overlap", False),
            "attention_variant": getattr(args, "attention_variant", 0),
            "scale": "1/sqrt(D)", "l2": "flushed before every timed step (512 MiB write)",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


# ----------------------------------------------------------------------------- GPU arm

def attn_traffic(name: str):
    """ncu DRAM bytes per attention launch, or None if the kernel source changed since the capture."""
    import hashlib

    src = ROOT / "diffusion_transformer_attention_dit_gb300" / "csrc" / "attn_fwd.cu"
    if hashlib.sha256(src.read_bytes()).hexdigest()[:16] != ATTN_TRAFFIC["source_sha256_prefix"]:
        return None
    return ATTN_TRAFFIC.get(name)


def aggregate(t_local: float, flops_per_step: float, steps: int, world: int, device=None):
    """Replica timing across ranks: max of the per-rank timed seconds, and whole-job TFLOP/s.

    Each rank runs its own full copy of the workload (no data-path collective);
    the process group only carries this max-reduction.
    """
    import torch
    import torch.distributed as dist

    t = torch.tensor([t_local], dtype=torch.float64, device=device)
    if world > 1:
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
    t_max = float(t.item())
    return t_max, flops_per_step * steps * world / t_max / 1e12


def run_ours(args):
    import torch
    import torch.distributed as dist

    from diffusion_transformer_attention_dit_gb300 import build, ops

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    build.build()
    ops.load_library()
    ops.set_launch_overlap(not args.no_launch_overlap)
    ops.set_attention_variant(args.attention_variant)

    inp = inputs.make_inputs(args.workload)
    w = inp.w
    chunks = args.chunks or w.chunks
    pdt = torch.float32 if PARTIAL[w.name] == "f32" else torch.bfloat16
    dev = torch.device("cuda", torch.cuda.current_device())

    def to_dev(a, dtype=None):
        t = torch.from_numpy(np.ascontiguousarray(a))
        return t.to(dev).view(torch.bfloat16) if dtype is None else t.to(dev)

    host = {"q": inp.q, "k": inp.k, "v": inp.v}
    q, k, v = (to_dev(host[n].view(np.int16)) for n in ("q", "k", "v"))
    wq, wk, cos, sin = (torch.from_numpy(a).to(dev) for a in (inp.wq, inp.wk, inp.cos, inp.sin))
    B, S, H, D = w.B, w.S, w.H, w.D
    o = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)  # noqa: E731
    merge = merge_mode(w, args)
    launches_per_step = (1 if w.prologue else 0) + chunks + (1 if chunks > 1 and merge == "kernel" else 0)
    # one C call per step (dit_attention): prologue into the workspace, the KV chunks (chunk c covers keys
    # [c*S/chunks, (c+1)*S/chunks)), then the merge -- in the update form in the last chunk's epilogue, else by
    # the merge kernel over stacked partials.  The events bracket the attention launches alone.
    ws = torch.empty(max(1, ops.attention_workspace_bytes(B, S, H, D, chunks, w.prologue, pdt, merge)),
                     dtype=torch.uint8, device=dev)

    def step(attn_events=None):
        ops.dit_attention(q, k, v, wq, wk, cos, sin, eps=w.eps, chunks=chunks, partial_dtype=pdt,
                          prologue=w.prologue, merge=merge, o=o, lse=lse, workspace=ws, attn_events=attn_events)

    for _ in range(args.warmup):
        step()
    ops.poll_device_error()
    if not args.steps:
        # enough steps for about 2 s of timed work (so the clock sampler sees the region)
        e0, e1 = ev(), ev()
        flush.zero_()
        e0.record(stream)
        step()
        e1.record(stream)
        torch.cuda.synchronize()
        args.steps = int(min(4000, max(10, 2000.0 / max(e0.elapsed_time(e1), 1e-3))))

    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        pass
    def made(n):  # events created (recorded once) before a timed region, so none is created inside it
        evs = [ev() for _ in range(n)]
        for e in evs:
            e.record(stream)
        return evs

    # Timed region: whole steps only.  Events between the kernels of a step stall the stream and cut the launch
    # overlap between them (about 11 us per Qwen-Image step), so the step region carries none; the attention
    # launches are timed in a second region of the same steps below.
    step_ev = made(2 * args.steps)
    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    wall0 = time.perf_counter()
    with ClockSampler(uuid) as clocks:
        for i in range(args.steps):
            flush.zero_()
            step_ev[2 * i].record(stream)
            step()
            step_ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
    wall = time.perf_counter() - wall0
    if world > 1:
        dist.barrier()
    ops.poll_device_error()
    t_steps = sum(step_ev[2 * i].elapsed_time(step_ev[2 * i + 1]) for i in range(args.steps)) / 1e3
    # Attention region: the same steps with events recorded (by dit_attention, on this stream) right before the
    # first and after the last attention launch; achieved = attention flops / the time between them.
    attn_steps = min(args.steps, ATTN_TIMED_STEPS)
    attn_ev = made(2 * attn_steps)
    torch.cuda.synchronize()
    for i in range(attn_steps):
        flush.zero_()
        step((attn_ev[2 * i], attn_ev[2 * i + 1]))
    torch.cuda.synchronize()
    ops.poll_device_error()
    t_attn = sum(attn_ev[2 * i].elapsed_time(attn_ev[2 * i + 1]) for i in range(attn_steps)) / 1e3
    flops_step = w.attention_flops()
    t_max, value = aggregate(t_steps, flops_step, args.steps, world, dev)

    # end to end through the public API: pinned host inputs in, O and LSE back to pinned host memory
    pin = {n: torch.from_numpy(np.ascontiguousarray(host[n]).view(np.int16)).pin_memory() for n in host}
    pin_small = [torch.from_numpy(a).pin_memory() for a in (inp.wq, inp.wk, inp.cos, inp.sin)]
    o_host = torch.empty((B, S, H, D), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    h2d = sum(t_.numel() * t_.element_size() for t_ in list(pin.values()) + pin_small)
    d2h = o_host.numel() * 2 + lse_host.numel() * 4
    dq, dk, dv = (torch.empty((B, S, H, D), dtype=torch.int16, device=dev) for _ in range(3))
    dsmall = [torch.empty_like(t_, device=dev) for t_ in pin_small]

    host_path = merge == "update" or chunks == 1
    if host_path:
        # dit_attention_host: the C entry point that copies the inputs in (value rows chunk by chunk on a copy
        # stream, overlapping the kernels), runs the path and copies O and LSE out
        hq, hk, hv = (pin[n].view(torch.bfloat16).view(B, S, H, D) for n in ("q", "k", "v"))
        ws = torch.empty(ops.attention_host_workspace_bytes(B, S, H, D, chunks, w.prologue, pdt), dtype=torch.uint8,
                         device=dev)

    def e2e_step():
        if host_path:
            ops.dit_attention_host(hq, hk, hv, *pin_small, eps=w.eps, chunks=chunks, partial_dtype=pdt,
                                   prologue=w.prologue, o=o_host, lse=lse_host, workspace=ws)
            return
        for src, dst in zip((pin["q"], pin["k"], pin["v"]), (dq, dk, dv)):
            dst.copy_(src, non_blocking=True)
        for src, dst in zip(pin_small, dsmall):
            dst.copy_(src, non_blocking=True)
        oo, ll = ops.dit_attention(dq.view(torch.bfloat16), dk.view(torch.bfloat16), dv.view(torch.bfloat16),
                                   *dsmall, eps=w.eps, chunks=chunks, partial_dtype=pdt, prologue=w.prologue,
                                   merge=merge)
        o_host.copy_(oo, non_blocking=True)
        lse_host.copy_(ll, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        e2e_step()
    torch.cuda.synchronize()
    e2e_t = 0.0
    for _ in range(args.steps):
        flush.zero_()
        e0, e1 = ev(), ev()
        e0.record(stream)
        e2e_step()
        e1.record(stream)
        torch.cuda.synchronize()
        e2e_t += e0.elapsed_time(e1) / 1e3
    _, e2e_value = aggregate(e2e_t, flops_step, args.steps, world, dev)

    if rank == 0:
        peak_tf, peak_gbs, src = peaks()
        achieved = flops_step * attn_steps / t_attn / 1e12
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, chunks, args),
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel", "achieved": achieved, "peak": peak_tf,
                         "unit": "TFLOP/s", "frac": achieved / peak_tf, "peak_source": src,
                         "traffic": args.traffic if args.traffic is not None else attn_traffic(w.name),
                         "timing": f"{attn_steps} further steps with events right before the first and after the "
                                   "last attention launch (the step region carries no events between kernels)"},
            "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "dit_attention_host (copies pipelined per KV chunk)" if host_path
                    else "torch copies + ops.dit_attention"},
            "gpu_launches": launches_per_step * args.steps,
            "clocks": clocks.summary(),
            "wall_s_timed_region": wall,
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(inp, chunks, args.cpu_budget)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_ring_overlap(args):
    """Diagnostic: the ring-overlap emulation (local attention || gather of the remote key shards, attention over
    the gathered keys, merge) against the same steps run back to back on one stream."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import build, ops

    build.build()
    ops.load_library()
    inp = inputs.make_inputs(args.workload)
    w = inp.w
    dev = torch.device("cuda")
    q, k, v = (torch.from_numpy(np.ascontiguousarray(getattr(inp, n)).view(np.int16)).to(dev).view(torch.bfloat16)
               for n in ("q", "k", "v"))
    bounds = w.chunk_bounds(args.ring_overlap)
    k_loc, v_loc = k[:, :bounds[0][1]].contiguous(), v[:, :bounds[0][1]].contiguous()
    remote = [(k[:, lo:hi].contiguous(), v[:, lo:hi].contiguous()) for lo, hi in bounds[1:]]
    side = torch.cuda.Stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def serial():
        kr = torch.cat([a for a, _ in remote], dim=1)
        vr = torch.cat([b for _, b in remote], dim=1)
        o1, l1 = ops.attn_fwd(q, k_loc, v_loc, o_dtype=torch.float32)
        return ops.attn_fwd_update(q, kr, vr, o1, l1, lse=l1)

    def overlapped():
        return ops.ring_overlap_attention(q, k_loc, v_loc, remote, gather_stream=side)

    res = {}
    for name, fn in (("serial", serial), ("overlapped", overlapped)):
        for _ in range(3):
            fn()
        torch.cuda.synchronize()
        ts = []
        for _ in range(max(args.steps, 5)):
            flush.zero_()
            torch.cuda.synchronize()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        res[name] = statistics.median(ts)
    print(json.dumps({"mode": "ring_overlap_emulation", "workload": w.name, "ranks": args.ring_overlap,
                      "serial_ms": res["serial"], "overlapped_ms": res["overlapped"],
                      "attention_tflops_overlapped": w.attention_flops() / res["overlapped"] / 1e9}))


def run_hbm_kernels(args):
    """Diagnostic: each HBM-bound kernel alone at the workload's shapes (synthetic inputs, L2 flushed before every
    timed launch, CUDA events, median of the steps): prologue, LSE merge of the workload's chunk count (8 for a
    one-chunk workload), LayerNorm-modulate and RMSNorm over C = H*D, fp8 quantiser.  Achieved = algorithmic bytes /
    time."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import build, ops

    build.build()
    ops.load_library()
    ops.set_launch_overlap(not args.no_launch_overlap)
    w = inputs.WORKLOADS[args.workload]
    B, S, H, D = w.B, w.S, w.H, w.D
    C = w.chunks if w.chunks > 1 else 8
    pdt = torch.float32 if PARTIAL[w.name] == "f32" else torch.bfloat16
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + w.index)
    rnd = lambda *shape: torch.randn(*shape, device=dev, generator=g)  # noqa: E731
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        ts = []
        for _ in range(max(args.steps, 5)):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record()
            fn()
            e1.record()
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1) * 1e3)
        ops.poll_device_error()
        return statistics.median(ts)

    peak_tf, peak_gbs, src = peaks()
    res = {}

    def record(name, us, nbytes):
        gbs = nbytes / us / 1e3
        res[name] = {"us": us, "GB": nbytes / 1e9, "GB/s": gbs, "frac": gbs / peak_gbs}

    q, k = rnd(B, S, H, D).to(torch.bfloat16), rnd(B, S, H, D).to(torch.bfloat16)
    wq, wk = 1 + 0.1 * rnd(D), 1 + 0.1 * rnd(D)
    cos, sin = rnd(S, D // 2), rnd(S, D // 2)
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    record("qk_norm_rope", timed(lambda: ops.qk_norm_rope(q, k, wq, wk, cos, sin, w.eps, q_out=qo, k_out=ko)),
           8 * B * S * H * D + 4 * S * D + 8 * D)
    del k, ko
    parts = rnd(C, B, S, H, D).to(pdt)
    lse_parts = 3 + 2 * rnd(C, B, H, S)
    lse = torch.empty(B, H, S, device=dev)
    record(f"merge_lse C={C} {PARTIAL[w.name]}->bf16", timed(lambda: ops.attn_merge_lse(parts, lse_parts, o=qo, lse=lse)),
           C * B * S * H * D * parts.element_size() + 4 * C * B * H * S + 2 * B * S * H * D + 4 * B * H * S)
    del parts, lse_parts
    x, y = q.view(B, S, H * D), qo.view(B, S, H * D)
    Cc = H * D
    sc, sh, wn = 0.1 * rnd(B, Cc), 0.1 * rnd(B, Cc), 1 + 0.1 * rnd(Cc)
    record("layer_norm_modulate", timed(lambda: ops.layer_norm_modulate(x, sc, sh, w.eps, y=y)),
           4 * B * S * Cc + 8 * B * Cc)
    record("rms_norm (over C)", timed(lambda: ops.rms_norm(x, wn, w.eps, y=y)), 4 * B * S * Cc + 4 * Cc)
    codes = torch.empty((B * S, Cc), dtype=torch.uint8, device=dev)
    scales = torch.empty(B * S, dtype=torch.float32, device=dev)
    record("quant_fp8_rows", timed(lambda: ops.quant_fp8_rows(x.view(B * S, Cc), codes, scales)),
           3 * B * S * Cc + 4 * B * S)
    print(json.dumps({"mode": "hbm_kernels", "workload": w.name, "peak_GBps": peak_gbs, "peak_source": src,
                      "kernels": res}))


def run_qkv_fp8(args):
    """Diagnostic: per-token e4m3 quantisation of the tokens (B*S x H*D) and the fp8 GEMM with a
    [3*H*D, H*D] QKV weight, synthetic, timed with CUDA events (L2 flushed before each step)."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import build, ops

    build.build()
    ops.load_library()
    w = inputs.WORKLOADS[args.workload]
    M, K, N = w.B * w.S, w.H * w.D, 3 * w.H * w.D
    dev = torch.device("cuda")
    x = torch.from_numpy(inputs.bf16_normal(M * K, seed=7000 + w.index).reshape(M, K)).to(dev).view(torch.bfloat16)
    wt = torch.from_numpy(inputs.bf16_normal(N * K, seed=7100 + w.index, std=0.02).reshape(N, K)).to(dev)
    wq, ws = ops.quant_fp8_rows(wt.view(torch.bfloat16))
    xq = torch.empty((M, K), dtype=torch.uint8, device=dev)
    xs = torch.empty(M, dtype=torch.float32, device=dev)
    out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    tq, tg = [], []
    for i in range(args.warmup + max(args.steps, 5)):
        flush.zero_()
        e = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
        e[0].record()
        ops.quant_fp8_rows(x, xq, xs)
        e[1].record()
        ops.gemm_fp8(xq, xs, wq, ws, out=out)
        e[2].record()
        torch.cuda.synchronize()
        if i >= args.warmup:
            tq.append(e[0].elapsed_time(e[1]))
            tg.append(e[1].elapsed_time(e[2]))
    ops.poll_device_error()
    t_q, t_g = statistics.median(tq), statistics.median(tg)
    print(json.dumps({"mode": "qkv_fp8", "workload": w.name, "M": M, "N": N, "K": K,
                      "quant_ms": t_q, "quant_GBps": 3 * M * K / t_q / 1e6,
                      "gemm_ms": t_g, "gemm_TFLOPs": 2 * M * N * K / t_g / 1e9}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: about 2 s worth)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="qwen_image", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--chunks", type=int, default=0, help="KV chunks (0: the workload's own)")
    ap.add_argument("--attention-variant", type=int, choices=[0, 1, 2, 3, 4], default=0,
                    help="attention kernel for head dim 128: 0 default, 1 one CTA (P in TMEM), 2 CTA pairs with two "
                         "tiles per CTA, 3 CTA pairs with one tile per CTA and three S buffers, 4 one CTA with P in "
                         "shared memory")
    ap.add_argument("--no-launch-overlap", action="store_true",
                    help="launch without programmatic dependent launch (each kernel starts after the previous ends)")
    ap.add_argument("--merge", choices=["auto", "kernel", "update"], default="auto",
                    help="combine KV chunks by the merge kernel or in the attention epilogue (auto: the workload's)")
    ap.add_argument("--ref-rows", type=int, default=48, help="query rows per (b, h) in each reference step")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--ring-overlap", type=int, default=0, metavar="RANKS",
                    help="time the one-GPU ring-overlap emulation with RANKS key shards instead (diagnostic)")
    ap.add_argument("--hbm-kernels", action="store_true",
                    help="time each HBM-bound kernel alone at the workload's shapes instead (diagnostic)")
    ap.add_argument("--qkv-fp8", action="store_true",
                    help="time the W8A8 fp8 QKV projection of the workload's tokens instead (diagnostic)")
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per attention launch from an ncu capture of the current kernel")
    args = ap.parse_args()
    if args.impl == "ours":
        args.warmup = max(3, args.warmup)  # at least 3 untimed warm-up steps
    elif not args.steps:
        args.steps = 5
    if args.impl == "reference":
        run_reference(args)
    elif args.ring_overlap:
        run_ring_overlap(args)
    elif args.qkv_fp8:
        run_qkv_fp8(args)
    elif args.hbm_kernels:
        run_hbm_kernels(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
