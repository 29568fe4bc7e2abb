"""First use from several host threads at once.

Each launcher does a one-time setup per device the first time it runs there:
it raises the kernel's shared-memory limit, and the fp8 GEMM also caches how
many CTA pairs can be resident. This test runs a fresh process in which four
threads make their first calls of the GEMM, the attention, the prologue, the
merge and LayerNorm-modulate at the same moment, each on its own stream.
ctypes releases the GIL, so the setups really race. Every thread must succeed
and produce the same bits as a later call made alone."""

import os
import subprocess
import sys
import textwrap
from pathlib import Path

import pytest

pytestmark = pytest.mark.gpu
ROOT = Path(__file__).resolve().parent.parent

CHILD = textwrap.dedent("""
    import threading
    import numpy as np
    import torch
    from diffusion_transformer_attention_dit_gb300 import ops

    ops.load_library()
    dev = torch.device("cuda")
    g = torch.Generator(device=dev)
    g.manual_seed(11)
    rng = np.random.default_rng(11)
    # fp8 operands as seeded bytes (NaN codes replaced), so no library kernel runs before the threads start
    M, N, K = 700, 1032, 512
    a = rng.integers(0, 256, (M, K), dtype=np.uint8); a[(a & 0x7F) == 0x7F] = 0x38
    b = rng.integers(0, 256, (N, K), dtype=np.uint8); b[(b & 0x7F) == 0x7F] = 0x38
    a, b = torch.from_numpy(a).to(dev), torch.from_numpy(b).to(dev)
    sa = torch.rand(M, device=dev, generator=g) * 1e-2
    sb = torch.rand(N, device=dev, generator=g) * 1e-3
    B, S, H, D = 1, 1000, 4, 128
    q, k, v = (torch.randn(B, S, H, D, device=dev, generator=g).to(torch.bfloat16) for _ in range(3))
    wq, wk = 1 + 0.1 * torch.randn(D, device=dev, generator=g), 1 + 0.1 * torch.randn(D, device=dev, generator=g)
    cos, sin = torch.randn(S, D // 2, device=dev, generator=g), torch.randn(S, D // 2, device=dev, generator=g)
    parts = torch.randn(3, B, S, H, D, device=dev, generator=g).to(torch.bfloat16)
    lparts = torch.randn(3, B, H, S, device=dev, generator=g)
    x = torch.randn(2, 300, 5120, device=dev, generator=g).to(torch.bfloat16)
    sc, sh = 0.1 * torch.randn(2, 5120, device=dev, generator=g), 0.1 * torch.randn(2, 5120, device=dev, generator=g)
    torch.cuda.synchronize()

    def work(stream):
        with torch.cuda.stream(stream):
            return (ops.gemm_fp8(a, sa, b, sb, stream=stream),
                    ops.attn_fwd(q, k, v, stream=stream)[0],
                    torch.cat([t.flatten() for t in ops.qk_norm_rope(q, k, wq, wk, cos, sin, stream=stream)]),
                    ops.attn_merge_lse(parts, lparts, stream=stream)[0],
                    ops.layer_norm_modulate(x, sc, sh, stream=stream))

    n = 4
    start = threading.Barrier(n)
    results, errors = [None] * n, []

    def run(i):
        s = torch.cuda.Stream()
        try:
            start.wait()
            results[i] = work(s)
            s.synchronize()
        except Exception as e:  # noqa: BLE001
            errors.append(repr(e))

    threads = [threading.Thread(target=run, args=(i,)) for i in range(n)]
    for t in threads: t.start()
    for t in threads: t.join()
    assert not errors, errors
    ops.poll_device_error()
    ref = work(torch.cuda.current_stream())
    torch.cuda.synchronize()
    for i in range(n):
        for got, want in zip(results[i], ref):
            assert torch.equal(got, want), i
    print("ok")
""")


def test_first_launches_from_four_threads_at_once():
    r = subprocess.run([sys.executable, "-c", CHILD], capture_output=True, text=True, cwd=ROOT, timeout=600,
                       env=dict(os.environ, PYTHONPATH=str(ROOT)))
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), (r.stdout[-2000:], r.stderr[-3000:])
