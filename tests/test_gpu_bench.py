"""bench.py's JSON line on the GPU: one short run of the whole line on the tiny workload (the per-workload and
prologue-alone records left out to keep it short), checked for every field the line promises."""

import json
import os
import subprocess
import sys
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent


def test_bench_line_has_every_field():
    env = dict(os.environ, RANK="0", WORLD_SIZE="1")
    r = subprocess.run([sys.executable, str(ROOT / "bench.py"), "--workload", "tiny", "--steps", "3", "--warmup", "3",
                        "--no-per-workload", "--cpu-budget", "0.5"], capture_output=True, text=True, env=env,
                       cwd=ROOT, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    line = json.loads(r.stdout.strip().splitlines()[-1])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step", "higher_is_better", "scaling",
                "vs_baseline", "dtype", "data", "config", "roofline", "hbm", "e2e", "gpu_launches", "clocks",
                "cpu_baseline"):
        assert key in line, key
    assert line["unit"] == "TFLOP/s" and line["value"] > 0 and line["steps"] == 3 and line["warmup"] == 3
    assert line["config"]["name"] == "tiny" and line["config"]["kv_chunks"] == 4
    roof = line["roofline"]
    assert roof["bound"] == "tensor" and roof["achieved"] > 0 and roof["peak"] > 0
    assert abs(roof["frac"] - roof["achieved"] / roof["peak"]) < 1e-9
    for k in ("qk_norm_rope", "layer_norm_modulate", "rms_norm", "quant_fp8_rows"):
        assert k in line["hbm"] and line["hbm"][k]["GB/s"] > 0 and "clocks" in line["hbm"][k], k
    gemm = line["fp8_gemm"]
    assert gemm["TFLOP/s"] > 0 and abs(gemm["frac"] - gemm["TFLOP/s"] / gemm["peak"]) < 1e-9
    assert (gemm["M"], gemm["N"], gemm["K"]) == (256, 384, 128)  # tiny: 256 tokens, C = H * D = 128
    e2e = line["e2e"]
    assert e2e["value"] > 0 and e2e["h2d_bytes_per_step"] > 0 and e2e["d2h_bytes_per_step"] > 0
    assert "dit_attention_host" in e2e["api"]
    # the tiny workload: prologue + 4 chunks (update form: no merge launch) per step
    assert line["gpu_launches"] == 5 * 3
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
