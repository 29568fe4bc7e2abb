#!/usr/bin/env python3
"""Benchmark of the DiT attention hot path on GB300.

One step = the whole path on one batch of synthetic input, resident in HBM,
as one dit_attention call: QK-RMSNorm + interleaved RoPE on Q and K (when the
workload has it), flash attention over the workload's KV chunks, and the LSE
merge (by the merge kernel over stacked partials, or in the last chunk's
epilogue).  Default workload: Wan2.2 720p (B1 H40 D128 S75600 = 21x45x80
patches, K x 3, no prologue), KV in 8 chunks with bf16 partials merged by the
LSE-merge kernel.

The JSON line (rank 0) carries, beside the step throughput:
  roofline      the attention launches of the step, timed in a second region of
                the same steps (events around the attention launches only)
  hbm           the step's merge kernel (events around it in that region) and,
                timed alone at the workload's shapes, the QK-RMSNorm + RoPE
                prologue and the DiT block's LayerNorm-modulate, RMSNorm over
                C and fp8 quantiser on its tokens; algorithmic bytes / time
                against the measured HBM copy bandwidth
  fp8_gemm      the W8A8 QKV projection of those tokens (tcgen05 fp8 GEMM),
                timed alone, against 2x the measured bf16 peaks
  per_workload  the other full-size workloads (Qwen-Image, Qwen-Image-Edit,
                Wan2.2 480p), each its own step and attention regions
  e2e           the public host-buffer call (dit_attention_host) with the
                host<->device copies inside the timed region
Every timed region has its own nvidia-smi clock record, holding only the
samples taken while that region ran.

`--impl reference` times the fp64 CPU oracle (the only reference this method
has) on a bounded sample of the same workload.

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
FALLBACK = {"bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "hbm_gbs": 6800.0}
L2_FLUSH_BYTES = 512 << 20
REGION_S = 1.5           # target length of the regions whose step count bench.py chooses
SAMPLER_WARMUP_S = 0.6   # nvidia-smi is given this long to start before a timed region
PARTIAL = {"tiny": "f32", "qwen_image": "f32", "qwen_image_edit": "f32", "wan480": "f32", "wan720": "bf16"}
# How the KV chunks are combined: "update" folds each later chunk into the running (O, LSE) in its attention
# epilogue; "kernel" writes stacked per-chunk partials and runs the LSE-merge kernel (Wan720's workload
# specifies per-chunk bf16 partials merged by the merge kernel).
MERGE = {"tiny": "update", "qwen_image": "update", "qwen_image_edit": "update", "wan480": "kernel",
         "wan720": "kernel"}
PER_WORKLOAD = ("qwen_image", "qwen_image_edit", "wan480")
# DRAM bytes (read + write) per attention launch, from an ncu capture of the attention kernel whose code (source
# without comments, attn_source_digest) has this sha256 prefix; reported as roofline.traffic only while it matches.
ATTN_TRAFFIC = {"source_sha256_prefix": "4f9d9b792e932a0e", "by_workload": {"wan720": 1716.6e6},
                "capture": "stored ncu capture (dram__bytes_read.sum + dram__bytes_write.sum) of one Wan2.2-720p "
                           "chunk launch, bench.py --profile-kernel attention --workload wan720"}


def peaks():
    path = ROOT / "MEASURED_PEAKS.json"
    if path.exists():
        try:
            d = json.loads(path.read_text())
            out = {k: float(d[k]) for k in FALLBACK if d.get(k)}
            if len(out) == len(FALLBACK):
                return out, "measured"
        except (ValueError, OSError, TypeError):
            pass
    return dict(FALLBACK), "fallback"


class ClockSampler:
    """nvidia-smi samples (every 200 ms), each stamped with the host time it arrived; summary() keeps those that
    arrived inside a given window (the timed region, plus one sampling period for the sample in flight)."""

    FIELDS = ("uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    PERIOD_S = 0.2

    def __init__(self, uuid: str | None):
        self.uuid = uuid
        self.lines: list[tuple[float, str]] = []
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                                          "-lms", str(int(self.PERIOD_S * 1000))], stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.perf_counter(), line.strip()))

    def ready(self, timeout_s: float = SAMPLER_WARMUP_S):
        """Wait (bounded) for the first sample, so the region's first samples are not lost to start-up."""
        t0 = time.perf_counter()
        while self.proc and not self.lines and time.perf_counter() - t0 < timeout_s:
            time.sleep(0.02)

    def __exit__(self, *exc):
        if self.proc:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self, t0: float | None = None, t1: float | None = None):
        rows = []
        for t, line in self.lines:
            if not line or (t0 is not None and t < t0) or (t1 is not None and t > t1 + self.PERIOD_S):
                continue
            rows.append(line.split(", "))
        if self.uuid:
            mine = [r for r in rows if r and self.uuid in r[0]]
            rows = mine or rows
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            try:
                sm.append(float(r[1]))
                smax.append(float(r[2]))
            except (ValueError, IndexError):
                continue
            try:
                power.append(float(r[3]))
            except (ValueError, IndexError):
                pass
            for n, v in zip(names, r[5:9]):
                if v.strip().lower() == "active":
                    reasons.add(n)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        out = {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
               "samples": len(sm)}
        if power:
            out["power_w_median"] = statistics.median(power)
        return out


# ----------------------------------------------------------------------------- CPU oracle (reference arm)

class OracleInputs:
    """The workload's inputs as fp64 arrays for the oracle (converted once; the key side is reused by every
    sampled row)."""

    def __init__(self, inp, chunks: int):
        import oracle

        self.orc = oracle.get()
        self.inp = inp
        self.chunks = chunks
        w = inp.w
        self.c64, self.s64 = inp.cos.astype(np.float64), inp.sin.astype(np.float64)
        k = inputs.bf16_bits_to_f64(inp.k)
        if w.prologue:
            k = oracle.round_bf16(self.orc.qk_norm_rope(k, inp.wk.astype(np.float64), self.c64, self.s64, w.eps))
        self.k = k
        self.v = inputs.bf16_bits_to_f64(inp.v)

    def step(self, rows: np.ndarray):
        """The hot path on the oracle for a sample of query rows (all heads, all keys): prologue of those rows,
        attention over every KV chunk, merge."""
        import oracle

        w = self.inp.w
        q = inputs.bf16_bits_to_f64(self.inp.q[:, rows])
        if w.prologue:
            q = oracle.round_bf16(self.orc.qk_norm_rope(q, self.inp.wq.astype(np.float64), self.c64[rows],
                                                        self.s64[rows], w.eps))
        parts = [self.orc.attention(q, self.k, self.v, w.scale, lo, hi) for lo, hi in w.chunk_bounds(self.chunks)]
        return self.orc.merge_lse(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))


def cpu_sample_rows(w, n: int) -> np.ndarray:
    return np.linspace(0, w.S - 1, n).round().astype(np.int64)


def cpu_baseline(inp, chunks: int, budget_s: float = 15.0):
    """Time the oracle on growing row samples until about budget_s of CPU work has been measured."""
    import oracle

    w = inp.w
    ref = OracleInputs(inp, chunks)
    n, total_t, total_f = 8, 0.0, 0.0
    while True:
        rows = cpu_sample_rows(w, min(n, w.S))
        t0 = time.perf_counter()
        ref.step(rows)
        dt = time.perf_counter() - t0
        total_t += dt
        total_f += 4.0 * w.B * w.H * len(rows) * w.S * w.D
        if total_t >= budget_s or n >= w.S:
            break
        n = min(w.S, max(2 * n, int(n * (budget_s - total_t) / max(dt, 1e-3))))
    return {"value": total_f / total_t / 1e12, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{w.name}: attention over {chunks} KV chunks + merge (and the prologue, where the workload "
                      f"has one) for evenly spaced query rows, all {w.H} heads, all {w.S} keys; row counts growing "
                      f"to {len(rows)}; {total_t:.1f} s of fp64 C/OpenMP work in total (the key-side fp64 "
                      f"conversion, done once, is not timed)"}


def run_reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    import oracle

    inp = inputs.make_inputs(args.workload)
    w = inp.w
    chunks = args.chunks or w.chunks
    ref = OracleInputs(inp, chunks)
    rows = cpu_sample_rows(w, args.ref_rows)
    for _ in range(args.warmup):
        ref.step(rows)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        ref.step(rows)
    dt = time.perf_counter() - t0
    flops = 4.0 * w.B * w.H * len(rows) * w.S * w.D * args.steps
    value = flops / dt / 1e12
    sample = (f"{w.name}: {len(rows)} evenly spaced query rows per (b, h) against all {w.S} keys; "
              f"{chunks} KV chunks and merge (and the prologue, where the workload has one) on the fp64 oracle")
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


def merge_text(merge: str, chunks: int) -> str:
    if chunks <= 1:
        return "none (one KV chunk)"
    return "update (fused in each later chunk's epilogue)" if merge == "update" else "kernel (LSE-merge kernel)"


def config_of(w, chunks, args):
    return {"workload": w.description, "name": w.name, "B": w.B, "H": w.H, "D": w.D, "Sq": w.S, "Skv": w.S,
            "kv_chunks": chunks, "partial_o": PARTIAL[w.name], "merge": merge_text(merge_mode(w, args), chunks),
            "prologue": w.prologue, "causal": False,
            "launch_overlap": not getattr(args, "no_launch_overlap", False),
            "scale": "1/sqrt(D)", "l2": "flushed before every timed step (512 MiB write)",
            "parallelism": "replicas" if args.gpus > 1 else "single GPU"}


# ----------------------------------------------------------------------------- GPU arm

def attn_source_digest() -> str:
    """sha256 prefix of the attention kernel's source with comments and blank lines removed (comment edits keep
    a stored capture valid; any code change invalidates it)."""
    import hashlib
    import re

    text = (ROOT / "diffusion_transformer_attention_dit_gb300" / "csrc" / "attn_fwd.cu").read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    code = "\n".join(ln.rstrip() for ln in text.splitlines() if ln.strip())
    return hashlib.sha256(code.encode()).hexdigest()[:16]


def attn_traffic(name: str):
    """ncu DRAM bytes per attention launch, or None if the kernel code changed since the capture."""
    if ATTN_TRAFFIC["source_sha256_prefix"] != attn_source_digest():
        return None
    return ATTN_TRAFFIC["by_workload"].get(name)


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


def merge_bytes(C, B, S, H, D, s_in, s_out):
    """Algorithmic bytes of one merge: C partial O and LSE slabs in, one O and LSE out."""
    return C * B * S * H * D * s_in + 4 * C * B * H * S + B * S * H * D * s_out + 4 * B * H * S


def prologue_bytes(B, S, H, D):
    """Algorithmic bytes of one prologue: q, k read and q', k' written (bf16), cos/sin tables, two weights."""
    return 8 * B * S * H * D + 4 * S * D + 8 * D


class Device:
    """Device-side state of one workload: inputs, outputs, workspace, the L2 flush buffer."""

    def __init__(self, inp, chunks, merge, dev):
        import torch

        from diffusion_transformer_attention_dit_gb300 import ops

        w = inp.w
        self.w, self.inp, self.chunks, self.merge, self.dev = w, inp, chunks, merge, dev
        self.pdt = torch.float32 if PARTIAL[w.name] == "f32" else torch.bfloat16
        bf = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).to(dev).view(torch.bfloat16)  # noqa
        self.q, self.k, self.v = bf(inp.q), bf(inp.k), bf(inp.v)
        self.tabs = [torch.from_numpy(a).to(dev) for a in (inp.wq, inp.wk, inp.cos, inp.sin)]
        B, S, H, D = w.B, w.S, w.H, w.D
        self.o = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
        self.lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        self.flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.ws = torch.empty(max(1, ops.attention_workspace_bytes(B, S, H, D, chunks, w.prologue, self.pdt, merge)),
                              dtype=torch.uint8, device=dev)
        self.merge_kernel = chunks > 1 and merge == "kernel"
        self.launches = (1 if w.prologue else 0) + chunks + (1 if self.merge_kernel else 0)

    def step(self, attn_events=None):
        from diffusion_transformer_attention_dit_gb300 import ops

        ops.dit_attention(self.q, self.k, self.v, *self.tabs, eps=self.w.eps, chunks=self.chunks,
                          partial_dtype=self.pdt, prologue=self.w.prologue, merge=self.merge, o=self.o, lse=self.lse,
                          workspace=self.ws, attn_events=attn_events)


def made_events(n, stream):
    """Events created and recorded once before a timed region, so none is created inside it."""
    import torch

    evs = [torch.cuda.Event(enable_timing=True) for _ in range(n)]
    for e in evs:
        e.record(stream)
    return evs


def steps_for(dev_state, seconds: float, cap: int = 20000) -> int:
    """Steps that fill about `seconds` of timed work (one flushed step is measured first)."""
    import torch

    stream = torch.cuda.current_stream()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    dev_state.flush.zero_()
    e0.record(stream)
    dev_state.step()
    e1.record(stream)
    torch.cuda.synchronize()
    return int(min(cap, max(10, seconds * 1e3 / max(e0.elapsed_time(e1), 1e-3))))


def time_workload(ds, steps, uuid, world=1):
    """The step region (events around whole steps only), then the attention region (events right before the first
    and after the last attention launch of each step, and after the merge kernel when there is one).  Returns the
    summed seconds and each region's clock record."""
    import torch
    import torch.distributed as dist

    from diffusion_transformer_attention_dit_gb300 import ops

    stream = torch.cuda.current_stream()
    res = {}
    # Timed region: whole steps only.  Events between the kernels of a step stall the stream and cut the launch
    # overlap between them, so the step region carries none.
    step_ev = made_events(2 * steps, stream)
    with ClockSampler(uuid) as clocks:
        clocks.ready()
        if world > 1:
            dist.barrier()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(steps):
            ds.flush.zero_()
            step_ev[2 * i].record(stream)
            ds.step()
            step_ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
        if world > 1:
            dist.barrier()
    ops.poll_device_error()
    res["t_steps"] = sum(step_ev[2 * i].elapsed_time(step_ev[2 * i + 1]) for i in range(steps)) / 1e3
    res["clocks_steps"] = clocks.summary(wall0, wall1)
    res["wall_steps"] = wall1 - wall0
    # Attention region: dit_attention records its events on this stream right before the first and after the last
    # attention launch; one more event after the call closes the merge kernel.
    attn_steps = steps
    n_ev = 3 if ds.merge_kernel else 2
    ev = made_events(n_ev * attn_steps, stream)
    with ClockSampler(uuid) as clocks:
        clocks.ready()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(attn_steps):
            ds.flush.zero_()
            e = ev[n_ev * i:n_ev * (i + 1)]
            ds.step((e[0], e[1]))
            if ds.merge_kernel:
                e[2].record(stream)
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
    ops.poll_device_error()
    res["attn_steps"] = attn_steps
    res["t_attn"] = sum(ev[n_ev * i].elapsed_time(ev[n_ev * i + 1]) for i in range(attn_steps)) / 1e3
    if ds.merge_kernel:
        res["t_merge"] = sum(ev[n_ev * i + 1].elapsed_time(ev[n_ev * i + 2]) for i in range(attn_steps)) / 1e3
    res["clocks_attn"] = clocks.summary(wall0, wall1)
    return res


def time_alone(run, flush, uuid, seconds: float = REGION_S):
    """One kernel launched alone, back to back for about `seconds` with L2 flushed before every launch; median
    seconds per launch, the launch count and the clock record."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import ops

    stream = torch.cuda.current_stream()
    for _ in range(3):
        run()
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    run()
    e1.record(stream)
    torch.cuda.synchronize()
    n = int(min(20000, max(20, seconds * 1e3 / (e0.elapsed_time(e1) + 0.1))))
    ev = made_events(2 * n, stream)
    with ClockSampler(uuid) as clocks:
        clocks.ready()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(n):
            flush.zero_()
            ev[2 * i].record(stream)
            run()
            ev[2 * i + 1].record(stream)
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
    ops.poll_device_error()
    ts = [ev[2 * i].elapsed_time(ev[2 * i + 1]) / 1e3 for i in range(n)]
    return statistics.median(ts), n, clocks.summary(wall0, wall1)


def time_prologue_alone(ds, uuid, seconds: float = REGION_S):
    """The prologue kernel alone at the workload's shapes (L2 flushed before every launch), for about `seconds`."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import ops

    qo, ko = torch.empty_like(ds.q), torch.empty_like(ds.k)
    out = time_alone(lambda: ops.qk_norm_rope(ds.q, ds.k, *ds.tabs, ds.w.eps, q_out=qo, k_out=ko), ds.flush, uuid,
                     seconds)
    del qo, ko
    return out


def block_kernel_records(ds, uuid, pk):
    """The DiT block's other kernels on this workload's tokens, each alone (L2 flushed before every launch, a
    ~REGION_S region with its clock record): LayerNorm-modulate, RMSNorm over C and the fp8 quantiser on the
    tokens as [B*S, C = H*D] rows (x = the workload's q), and the fp8 QKV projection GEMM they feed
    ([B*S, C] x [3C, C] codes).  Returns (hbm records, the GEMM record)."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import ops

    w = ds.w
    B, S, C = w.B, w.S, w.H * w.D
    M = B * S
    dev = ds.q.device
    g = torch.Generator(device=dev)
    g.manual_seed(4242 + w.index)
    x = ds.q.view(B, S, C)
    sc = 0.1 * torch.randn(B, C, device=dev, generator=g)
    sh = 0.1 * torch.randn(B, C, device=dev, generator=g)
    wn = 1 + 0.1 * torch.randn(C, device=dev, generator=g)
    y = torch.empty_like(x)
    codes = torch.empty((M, C), dtype=torch.uint8, device=dev)
    scale = torch.empty(M, dtype=torch.float32, device=dev)
    hbm = {}
    how = (f"the kernel alone on this workload's tokens as [{M}, {C}] bf16 rows (x = the workload's q), L2 "
           "flushed before every launch, median")
    t, n, clk = time_alone(lambda: ops.layer_norm_modulate(x, sc, sh, w.eps, y=y), ds.flush, uuid)
    hbm["layer_norm_modulate"] = hbm_record("row_pair_kernel (LayerNorm-modulate)", t, 4 * M * C + 8 * B * C,
                                            pk["hbm_gbs"], n, clk, how + "; fp32 scale / shift per batch entry")
    t, n, clk = time_alone(lambda: ops.rms_norm(x, wn, w.eps, y=y), ds.flush, uuid)
    hbm["rms_norm"] = hbm_record("row_kernel (RMSNorm over C)", t, 4 * M * C + 4 * C, pk["hbm_gbs"], n, clk, how)
    t, n, clk = time_alone(lambda: ops.quant_fp8_rows(x.view(M, C), codes, scale), ds.flush, uuid)
    hbm["quant_fp8_rows"] = hbm_record("quant_fp8_rows_kernel", t, 3 * M * C + 4 * M, pk["hbm_gbs"], n, clk,
                                       how + "; e4m3 codes and a per-row scale out")
    del y
    wt = (0.02 * torch.randn(3 * C, C, device=dev, generator=g)).to(torch.bfloat16)
    wq, ws = ops.quant_fp8_rows(wt)
    del wt
    out = torch.empty((M, 3 * C), dtype=torch.bfloat16, device=dev)
    t, n, clk = time_alone(lambda: ops.gemm_fp8(codes, scale, wq, ws, out=out), ds.flush, uuid)
    flops = 2.0 * M * 3 * C * C
    tf = flops / t / 1e12
    peak, peak_s = 2 * pk["bf16_tflops"], 2 * pk["bf16_tflops_sustained"]
    gemm = {"kernel": "gemm_fp8_kernel (CTA pairs)", "M": M, "N": 3 * C, "K": C, "flops": flops, "us": t * 1e6,
            "TFLOP/s": tf, "peak": peak, "frac": tf / peak, "peak_sustained": peak_s, "frac_sustained": tf / peak_s,
            "peak_kind": "2x the measured bf16 burst / sustained figures (the nominal fp8 : bf16 dense ratio)",
            "launches": n, "timing": "the W8A8 QKV projection of these tokens alone ([M, K] x [N, K] e4m3 codes, "
                                     "per-row / per-channel scales, bf16 out), L2 flushed before every launch, "
                                     "median", "clocks": clk}
    del out, codes, scale, wq, ws
    torch.cuda.empty_cache()
    return hbm, gemm


def hbm_record(name, t_s, nbytes, peak_gbs, launches, clocks, how):
    gbs = nbytes / t_s / 1e9
    return {"kernel": name, "bytes": nbytes, "us": t_s * 1e6, "GB/s": gbs, "peak": peak_gbs, "frac": gbs / peak_gbs,
            "launches": launches, "timing": how, "clocks": clocks}


def e2e_measure(inp, chunks, merge, steps, warmup, dev, flush):
    """The public host-buffer entry point (dit_attention_host) on pinned host inputs, copies inside the timed
    region; returns (seconds summed over the steps, h2d bytes, d2h bytes)."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import ops

    w = inp.w
    B, S, H, D = w.B, w.S, w.H, w.D
    pdt = torch.float32 if PARTIAL[w.name] == "f32" else torch.bfloat16
    pin = {n: torch.from_numpy(np.ascontiguousarray(getattr(inp, n)).view(np.int16)).pin_memory()
           for n in ("q", "k", "v")}
    hq, hk, hv = (pin[n].view(torch.bfloat16).view(B, S, H, D) for n in ("q", "k", "v"))
    small = [torch.from_numpy(a).pin_memory() for a in (inp.wq, inp.wk, inp.cos, inp.sin)] if w.prologue else []
    o_host = torch.empty((B, S, H, D), dtype=torch.bfloat16).pin_memory()
    lse_host = torch.empty((B, H, S), dtype=torch.float32).pin_memory()
    h2d = sum(t.numel() * t.element_size() for t in list(pin.values()) + small)
    d2h = o_host.numel() * 2 + lse_host.numel() * 4
    ws = torch.empty(ops.attention_host_workspace_bytes(B, S, H, D, chunks, w.prologue, pdt, merge=merge),
                     dtype=torch.uint8, device=dev)
    tabs = small if w.prologue else [None] * 4
    stream = torch.cuda.current_stream()
    # the host link's rate right now (it is shared with the machine's other GPUs): one pinned copy of q
    probe = torch.empty_like(pin["q"], device=dev)
    probe.copy_(pin["q"], non_blocking=True)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    probe.copy_(pin["q"], non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_gbps = probe.numel() * 2 / e0.elapsed_time(e1) / 1e6
    del probe

    def e2e_step():
        ops.dit_attention_host(hq, hk, hv, *tabs, eps=w.eps, chunks=chunks, partial_dtype=pdt, prologue=w.prologue,
                               merge=merge, o=o_host, lse=lse_host, workspace=ws)

    for _ in range(max(1, warmup)):
        e2e_step()
    torch.cuda.synchronize()
    ts, host = [], []
    for _ in range(steps):
        flush.zero_()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        t0 = time.perf_counter()
        e2e_step()
        host.append(time.perf_counter() - t0)  # how long the call took to queue the step's work
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1) / 1e3)
    ops.poll_device_error()
    del ws
    return ts, h2d, d2h, h2d_gbps, host


def per_workload_record(name, args, dev, uuid, pk, src):
    """One of the other full-size workloads: its step and attention regions, with their clocks."""
    import torch

    inp = inputs.make_inputs(name)
    w = inp.w
    chunks = w.chunks
    merge = MERGE[name]
    ds = Device(inp, chunks, merge, dev)
    for _ in range(args.warmup):
        ds.step()
    steps = steps_for(ds, REGION_S)
    r = time_workload(ds, steps, uuid)
    flops = w.attention_flops()
    attn = flops * r["attn_steps"] / r["t_attn"] / 1e12
    rec = {"workload": w.description, "B": w.B, "H": w.H, "D": w.D, "S": w.S, "kv_chunks": chunks,
           "merge": merge_text(merge, chunks), "partial_o": PARTIAL[name], "prologue": w.prologue,
           "steps": steps, "ms_per_step": r["t_steps"] / steps * 1e3,
           "step_tflops": flops * steps / r["t_steps"] / 1e12,
           "attention_tflops": attn, "attention_frac": attn / pk["bf16_tflops"],
           "attention_frac_sustained": attn / pk["bf16_tflops_sustained"], "peak_source": src,
           "clocks": r["clocks_steps"], "clocks_attention": r["clocks_attn"]}
    del ds
    torch.cuda.empty_cache()
    return rec


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
    dev = torch.device("cuda", torch.cuda.current_device())
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        pass
    pk, src = peaks()

    inp = inputs.make_inputs(args.workload)
    w = inp.w
    chunks = args.chunks or w.chunks
    merge = merge_mode(w, args)
    ds = Device(inp, chunks, merge, dev)
    for _ in range(args.warmup):
        ds.step()
    ops.poll_device_error()
    if not args.steps:
        args.steps = steps_for(ds, 2.0)
    r = time_workload(ds, args.steps, uuid, world)
    flops_step = w.attention_flops()
    t_max, value = aggregate(r["t_steps"], flops_step, args.steps, world, dev)
    B, S, H, D = w.B, w.S, w.H, w.D

    hbm = {}
    if r.get("t_merge") is not None:
        s_in = 4 if PARTIAL[w.name] == "f32" else 2
        hbm["merge_lse"] = hbm_record(
            "merge_lse_bulk_kernel", r["t_merge"] / r["attn_steps"], merge_bytes(chunks, B, S, H, D, s_in, 2),
            pk["hbm_gbs"], r["attn_steps"], r["clocks_attn"],
            f"the step's merge kernel ({chunks} {PARTIAL[w.name]} partials -> bf16), events around it in the "
            "attention region of the same steps, mean per launch")
    if not args.no_hbm:
        t_pro, n_pro, clk_pro = time_prologue_alone(ds, uuid)
        hbm["qk_norm_rope"] = hbm_record(
            "qk_norm_rope_kernel", t_pro, prologue_bytes(B, S, H, D), pk["hbm_gbs"], n_pro, clk_pro,
            f"the prologue kernel alone on this workload's q, k, weights and rotary tables (the step "
            f"{'runs it' if w.prologue else 'has none'}), L2 flushed before every launch, median")
    fp8_gemm = None
    if not args.no_hbm and not args.no_block_kernels:
        more, fp8_gemm = block_kernel_records(ds, uuid, pk)
        hbm.update(more)

    e2e = None
    if not args.no_e2e:
        e2e_steps = max(3, min(args.steps, 20))
        ts_e2e, h2d, d2h, h2d_gbps, host = e2e_measure(inp, chunks, merge, e2e_steps, args.warmup, dev, ds.flush)
        t_e2e = sum(ts_e2e)
        _, e2e_value = aggregate(t_e2e, flops_step, e2e_steps, world, dev)
        e2e = {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "steps": e2e_steps, "ms_per_step": t_e2e / e2e_steps * 1e3,
               # the spread of the steps (the host link is shared with the machine's other GPUs)
               "ms_per_step_min": min(ts_e2e) * 1e3, "ms_per_step_median": statistics.median(ts_e2e) * 1e3,
               "ms_per_step_max": max(ts_e2e) * 1e3,
               "ms_each": [round(t * 1e3, 1) for t in ts_e2e],
               "host_to_device_GBps": h2d_gbps,
               "host_call_ms_median": statistics.median(host) * 1e3, "host_call_ms_max": max(host) * 1e3,
               "api": "dit_attention_host (" + ("query ranges, stacked partials + merge kernel per range, each "
                                                "range's O copied back while the next computes" if
                                                (merge == "kernel" or chunks == 1) else
                                                "value rows pipelined per KV chunk, update-form merge") + ")"}
    launches = ds.launches * args.steps
    del ds
    torch.cuda.empty_cache()

    per = {}
    if rank == 0 and world == 1 and not args.no_per_workload:
        for name in PER_WORKLOAD:
            if name != w.name:
                per[name] = per_workload_record(name, args, dev, uuid, pk, src)

    if rank == 0:
        achieved = flops_step * r["attn_steps"] / r["t_attn"] / 1e12
        traffic = args.traffic if args.traffic is not None else attn_traffic(w.name)
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": t_max / args.steps * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
            "config": config_of(w, chunks, args),
            "roofline": {"bound": "tensor", "kernel": "attn_fwd_kernel", "achieved": achieved,
                         "peak": pk["bf16_tflops"], "unit": "TFLOP/s", "frac": achieved / pk["bf16_tflops"],
                         "peak_kind": "burst (cuBLAS bf16 GEMM, best of 10)",
                         "peak_sustained": pk["bf16_tflops_sustained"],
                         "frac_sustained": achieved / pk["bf16_tflops_sustained"], "peak_source": src,
                         "traffic": traffic,
                         "traffic_source": (ATTN_TRAFFIC["capture"] if traffic is not None and args.traffic is None
                                            else "given on the command line" if traffic is not None else
                                            "none for this attention source"),
                         "timing": f"{r['attn_steps']} further steps with events right before the first and after "
                                   "the last attention launch (the step region carries no events between kernels)",
                         "clocks": r["clocks_attn"]},
            "hbm": hbm,
            "fp8_gemm": fp8_gemm,
            "per_workload": per,
            "e2e": e2e,
            "gpu_launches": launches,
            "clocks": r["clocks_steps"],
            "wall_s_timed_region": r["wall_steps"],
        }
        if world == 1 and not args.no_cpu_baseline:
            line["cpu_baseline"] = cpu_baseline(inp, chunks, args.cpu_budget)
        print(json.dumps(line))
    if world > 1:
        dist.destroy_process_group()


def run_ring_overlap(args):
    """Diagnostic: one rank's ring overlap (dit_attention_ring_overlap: local attention || device copies gathering
    the remote key shards, then the attention over them merged in its epilogue) against the same work run back to
    back on one stream."""
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
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    B, S, H, D = q.shape
    s_rem = sum(b.shape[1] for b, _ in remote)
    kr = torch.empty((B, s_rem, H, D), dtype=torch.bfloat16, device=dev)
    vr = torch.empty_like(kr)
    acc = torch.empty((B, S, H, D), dtype=torch.float32, device=dev)
    o = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
    lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
    ws = torch.empty(ops.ring_overlap_workspace_bytes(B, S, H, D, s_rem, torch.float32), dtype=torch.uint8,
                     device=dev)

    def serial():  # the same work on one stream: gather copies, local attention, merged attention
        off = 0
        for kk, vv in remote:
            kr[:, off:off + kk.shape[1]].copy_(kk)
            vr[:, off:off + vv.shape[1]].copy_(vv)
            off += kk.shape[1]
        ops.attn_fwd(q, k_loc, v_loc, o=acc, lse=lse)
        return ops.attn_fwd_update(q, kr, vr, acc, lse, o=o, lse=lse)

    def overlapped():  # dit_attention_ring_overlap: the gather on its own stream beside the local attention
        return ops.ring_overlap_attention(q, k_loc, v_loc, remote, o=o, lse=lse, workspace=ws)

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
    timed launch, CUDA events, median over about REGION_S seconds of launches, each kernel with its own clock
    record): prologue, LSE merge of the workload's chunk count (8 for a one-chunk workload), LayerNorm-modulate
    and RMSNorm over C = H*D, fp8 quantiser.  Achieved = algorithmic bytes / time."""
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
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        pass
    g = torch.Generator(device=dev)
    g.manual_seed(1234 + w.index)
    rnd = lambda *shape: torch.randn(*shape, device=dev, generator=g)  # noqa: E731
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def timed(fn):
        for _ in range(max(args.warmup, 3)):
            fn()
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        n = int(min(20000, max(max(args.steps, 5), REGION_S * 1e3 / (e0.elapsed_time(e1) + 0.1))))
        ev = made_events(2 * n, stream)
        with ClockSampler(uuid) as clocks:
            clocks.ready()
            torch.cuda.synchronize()
            wall0 = time.perf_counter()
            for i in range(n):
                flush.zero_()
                ev[2 * i].record(stream)
                fn()
                ev[2 * i + 1].record(stream)
            torch.cuda.synchronize()
            wall1 = time.perf_counter()
        ops.poll_device_error()
        return statistics.median(ev[2 * i].elapsed_time(ev[2 * i + 1]) * 1e3 for i in range(n)), n, \
            clocks.summary(wall0, wall1)

    pk, src = peaks()
    res = {}

    def record(name, timing, nbytes):
        us, n, clk = timing
        gbs = nbytes / us / 1e3
        res[name] = {"us": us, "GB": nbytes / 1e9, "GB/s": gbs, "frac": gbs / pk["hbm_gbs"], "launches": n,
                     "clocks": clk}

    q, k = rnd(B, S, H, D).to(torch.bfloat16), rnd(B, S, H, D).to(torch.bfloat16)
    wq, wk = 1 + 0.1 * rnd(D), 1 + 0.1 * rnd(D)
    cos, sin = rnd(S, D // 2), rnd(S, D // 2)
    qo, ko = torch.empty_like(q), torch.empty_like(k)
    record("qk_norm_rope", timed(lambda: ops.qk_norm_rope(q, k, wq, wk, cos, sin, w.eps, q_out=qo, k_out=ko)),
           prologue_bytes(B, S, H, D))
    del k, ko
    parts = rnd(C, B, S, H, D).to(pdt)
    lse_parts = 3 + 2 * rnd(C, B, H, S)
    lse = torch.empty(B, H, S, device=dev)
    record(f"merge_lse C={C} {PARTIAL[w.name]}->bf16",
           timed(lambda: ops.attn_merge_lse(parts, lse_parts, o=qo, lse=lse)),
           merge_bytes(C, B, S, H, D, parts.element_size(), 2))
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
    print(json.dumps({"mode": "hbm_kernels", "workload": w.name, "peak_GBps": pk["hbm_gbs"], "peak_source": src,
                      "kernels": res}))


def run_profile_kernel(args):
    """Diagnostic for ncu captures: exactly three launches of one kernel at the workload's shapes (synthetic
    inputs; --profile-heads shrinks H to keep the device footprint of a multi-pass capture at a few GB).  The
    attention runs the second of the workload's KV chunks, as a bench step does."""
    import torch

    from diffusion_transformer_attention_dit_gb300 import build, ops

    build.build()
    ops.load_library()
    w = inputs.WORKLOADS[args.workload]
    B, S, D = w.B, w.S, w.D
    H = args.profile_heads or w.H
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(4321 + w.index)
    rnd = lambda *shape: torch.randn(*shape, device=dev, generator=g)  # noqa: E731
    kind = args.profile_kernel
    if kind in ("prologue", "attention"):
        q, k = rnd(B, S, H, D).to(torch.bfloat16), (w.k_scale * rnd(B, S, H, D)).to(torch.bfloat16)
    if kind == "prologue":
        wq, wk, cos, sin = 1 + 0.1 * rnd(D), 1 + 0.1 * rnd(D), rnd(S, D // 2), rnd(S, D // 2)
        qo, ko = torch.empty_like(q), torch.empty_like(k)
        run = lambda: ops.qk_norm_rope(q, k, wq, wk, cos, sin, w.eps, q_out=qo, k_out=ko)  # noqa: E731
    elif kind == "attention":
        v = rnd(B, S, H, D).to(torch.bfloat16)
        lo, hi = w.chunk_bounds(max(w.chunks, 2))[1]
        o = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev)
        lse = torch.empty((B, H, S), dtype=torch.float32, device=dev)
        run = lambda: ops.attn_fwd(q, k, v, None, lo, hi, o=o, lse=lse)  # noqa: E731
    elif kind == "merge":
        C = max(w.chunks, 2)
        parts = rnd(C, B, S, H, D).to(torch.float32 if PARTIAL[w.name] == "f32" else torch.bfloat16)
        lp = 3 + 2 * rnd(C, B, H, S)
        o, lse = torch.empty((B, S, H, D), dtype=torch.bfloat16, device=dev), torch.empty((B, H, S), device=dev)
        run = lambda: ops.attn_merge_lse(parts, lp, o=o, lse=lse)  # noqa: E731
    else:
        x = rnd(B, S, H * D).to(torch.bfloat16)
        y = torch.empty_like(x)
        if kind == "layer_norm_modulate":
            sc, sh = 0.1 * rnd(B, H * D), 0.1 * rnd(B, H * D)
            run = lambda: ops.layer_norm_modulate(x, sc, sh, w.eps, y=y)  # noqa: E731
        elif kind == "rms_norm":
            wn = 1 + 0.1 * rnd(H * D)
            run = lambda: ops.rms_norm(x, wn, w.eps, y=y)  # noqa: E731
        else:
            codes = torch.empty((B * S, H * D), dtype=torch.uint8, device=dev)
            scales = torch.empty(B * S, dtype=torch.float32, device=dev)
            run = lambda: ops.quant_fp8_rows(x.view(B * S, H * D), codes, scales)  # noqa: E731
    for _ in range(3):
        run()
    ops.poll_device_error()
    print(json.dumps({"mode": "profile_kernel", "kernel": kind, "workload": w.name, "H": H, "launches": 3}))


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
    uuid = None
    try:
        uuid = str(torch.cuda.get_device_properties(dev).uuid)
    except Exception:  # noqa: BLE001
        pass
    # a region of about REGION_S seconds, so the clock record holds samples under load
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record()
    ops.quant_fp8_rows(x, xq, xs)
    ops.gemm_fp8(xq, xs, wq, ws, out=out)
    e1.record()
    torch.cuda.synchronize()
    steps = int(min(20000, max(args.steps, 20, REGION_S * 1e3 / (e0.elapsed_time(e1) + 0.05))))
    ev = made_events(3 * (args.warmup + steps), torch.cuda.current_stream())
    with ClockSampler(uuid) as clocks:
        clocks.ready()
        torch.cuda.synchronize()
        wall0 = time.perf_counter()
        for i in range(args.warmup + steps):
            flush.zero_()
            ev[3 * i].record()
            ops.quant_fp8_rows(x, xq, xs)
            ev[3 * i + 1].record()
            ops.gemm_fp8(xq, xs, wq, ws, out=out)
            ev[3 * i + 2].record()
        torch.cuda.synchronize()
        wall1 = time.perf_counter()
    ops.poll_device_error()
    timed = range(args.warmup, args.warmup + steps)
    t_q = statistics.median(ev[3 * i].elapsed_time(ev[3 * i + 1]) for i in timed)
    t_g = statistics.median(ev[3 * i + 1].elapsed_time(ev[3 * i + 2]) for i in timed)
    pk, src = peaks()
    fp8_peak = 2 * pk["bf16_tflops"]  # the nominal fp8 : bf16 dense ratio applied to the measured bf16 burst
    print(json.dumps({"mode": "qkv_fp8", "workload": w.name, "M": M, "N": N, "K": K, "steps": steps,
                      "quant_ms": t_q, "quant_GBps": 3 * M * K / t_q / 1e6,
                      "gemm_ms": t_g, "gemm_TFLOPs": 2 * M * N * K / t_g / 1e9,
                      "gemm_frac_of_fp8_peak": 2 * M * N * K / t_g / 1e9 / fp8_peak,
                      "fp8_peak_TFLOPs": fp8_peak, "peak_source": src,
                      "clocks": clocks.summary(wall0, wall1)}))


def main():
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=0, help="timed steps (0: about 2 s worth)")
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="wan720", choices=sorted(inputs.WORKLOADS))
    ap.add_argument("--chunks", type=int, default=0, help="KV chunks (0: the workload's own)")
    ap.add_argument("--no-launch-overlap", action="store_true",
                    help="launch without programmatic dependent launch (each kernel starts after the previous ends)")
    ap.add_argument("--merge", choices=["auto", "kernel", "update"], default="auto",
                    help="combine KV chunks by the merge kernel or in the attention epilogue (auto: the workload's)")
    ap.add_argument("--ref-rows", type=int, default=16, help="query rows per (b, h) in each reference step")
    ap.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-workload", action="store_true", help="skip the per_workload record")
    ap.add_argument("--no-hbm", action="store_true", help="skip the kernels timed alone (prologue, block kernels, fp8 GEMM)")
    ap.add_argument("--no-block-kernels", action="store_true",
                    help="skip the LayerNorm-modulate / RMSNorm / quantiser entries of the hbm record and the fp8 GEMM")
    ap.add_argument("--no-e2e", action="store_true", help="skip the end-to-end (host buffers) measurement")
    ap.add_argument("--ring-overlap", type=int, default=0, metavar="RANKS",
                    help="time the one-GPU ring-overlap emulation with RANKS key shards instead (diagnostic)")
    ap.add_argument("--hbm-kernels", action="store_true",
                    help="time each HBM-bound kernel alone at the workload's shapes instead (diagnostic)")
    ap.add_argument("--qkv-fp8", action="store_true",
                    help="time the W8A8 fp8 QKV projection of the workload's tokens instead (diagnostic)")
    ap.add_argument("--profile-kernel", default=None,
                    choices=["prologue", "attention", "merge", "layer_norm_modulate", "rms_norm", "quant_fp8"],
                    help="run exactly three launches of one kernel at the workload's shapes (for ncu captures)")
    ap.add_argument("--profile-heads", type=int, default=0, help="heads for --profile-kernel (0: the workload's)")
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
    elif args.profile_kernel:
        run_profile_kernel(args)
    elif args.hbm_kernels:
        run_hbm_kernels(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
