"""Full-size DiT workloads, run exactly as bench.py times them (prologue, KV
chunks, LSE merge), checked against the fp64 oracle on sampled query rows of
every (b, h) -- each sampled row against all keys -- and, on every element,
against the GPU single-pass attention."""

import math

import numpy as np
import pytest

import oracle
from diffusion_transformer_attention_dit_gb300 import build, inputs, ops
from parity import check_bf16_rounding, check_lse, check_o, dev_bf16, dev_f32, host_f64, sample_rows

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

PARTIAL = {"qwen_image": torch.float32, "qwen_image_edit": torch.float32, "wan480": torch.float32,
           "wan720": torch.bfloat16}


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load_library()


def _device_compare(a: torch.Tensor, b: torch.Tensor):
    a = a.float().flatten()
    b = b.float().flatten()
    err = (a - b).abs().max().item()
    cos = (torch.dot(a.double(), b.double()) / (a.double().norm() * b.double().norm())).item()
    return err, cos


@pytest.mark.parametrize("name,chunks,merge", [
    ("qwen_image", 1, "kernel"), ("qwen_image_edit", 1, "kernel"), ("wan480", 1, "kernel"),  # as bench.py runs them
    ("wan720", 8, "kernel"),
    # the two-chunk forms (a local and a remote part, as in the Wan2.2 ring-overlap split), both merges
    ("qwen_image", 2, "update"), ("qwen_image", 2, "kernel"), ("qwen_image_edit", 2, "update")])
def test_workload_parity(name, chunks, merge):
    orc = oracle.get()
    inp = inputs.make_inputs(name)
    w = inp.w
    dq, dk, dv = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    tabs = (dev_f32(inp.wq), dev_f32(inp.wk), dev_f32(inp.cos), dev_f32(inp.sin))
    o, lse = ops.dit_attention(dq, dk, dv, *tabs, eps=w.eps, chunks=chunks, partial_dtype=PARTIAL[name],
                               prologue=w.prologue, merge=merge)
    if w.prologue:
        pq, pk = ops.qk_norm_rope(dq, dk, *tabs, eps=w.eps)
    else:
        pq, pk = dq, dk
    o1, l1 = ops.attn_fwd(pq, pk, dv)
    ops.poll_device_error()

    # every element: merged chunks vs single pass
    err, cos = _device_compare(o, o1)
    assert err <= 2e-2 and cos >= 0.9999, (err, cos)
    assert (lse - l1).abs().max().item() <= 1e-3

    rows = sample_rows(w.S, 64, seed=w.index)
    rows_t = torch.from_numpy(rows).cuda()
    got_o = host_f64(o.index_select(1, rows_t))           # [B, R, H, D]
    got_l = host_f64(lse.index_select(2, rows_t))         # [B, H, R]
    got_pq = host_f64(pq.index_select(1, rows_t)) if w.prologue else None
    c64, s64 = inp.cos.astype(np.float64), inp.sin.astype(np.float64)
    ref_o = np.empty_like(got_o)
    ref_l = np.empty_like(got_l)
    for h in range(w.H):
        qh = inputs.bf16_bits_to_f64(inp.q[:, :, h:h + 1, :])
        kh = inputs.bf16_bits_to_f64(inp.k[:, :, h:h + 1, :])
        vh = inputs.bf16_bits_to_f64(inp.v[:, :, h:h + 1, :])
        if w.prologue:
            qh = orc.qk_norm_rope(qh[:, rows], inp.wq.astype(np.float64), c64[rows], s64[rows], w.eps)
            kh = orc.qk_norm_rope(kh, inp.wk.astype(np.float64), c64, s64, w.eps)
            check_bf16_rounding(got_pq[:, :, h:h + 1, :], qh, f"{name} prologue head {h}")
            # the prologue hands bf16 Q/K to attention
            qh, kh = oracle.round_bf16(qh), oracle.round_bf16(kh)
            rsel = None
        else:
            rsel = rows
        oh, lh = orc.attention(qh, kh, vh, w.scale, rows=rsel)
        ref_o[:, :, h:h + 1, :] = oh
        ref_l[:, h:h + 1, :] = lh
    check_o(got_o, ref_o, what=f"{name} merged vs oracle (sampled rows)")
    check_lse(got_l, ref_l, what=f"{name} merged vs oracle (sampled rows)")


def test_qwen_image_every_element():
    """Qwen-Image (B1 H24 S4312, prologue, one pass, as bench.py runs it): every element of O and LSE against the
    oracle (its prologue in fp64, rounded to bf16 as the kernel hands Q and K to the attention)."""
    orc = oracle.get()
    inp = inputs.make_inputs("qwen_image")
    w = inp.w
    dq, dk, dv = dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v)
    tabs = (dev_f32(inp.wq), dev_f32(inp.wk), dev_f32(inp.cos), dev_f32(inp.sin))
    o, lse = ops.dit_attention(dq, dk, dv, *tabs, eps=w.eps, chunks=1, prologue=True)
    ops.poll_device_error()
    c64, s64 = inp.cos.astype(np.float64), inp.sin.astype(np.float64)
    q = oracle.round_bf16(orc.qk_norm_rope(inputs.bf16_bits_to_f64(inp.q), inp.wq.astype(np.float64), c64, s64,
                                           w.eps))
    k = oracle.round_bf16(orc.qk_norm_rope(inputs.bf16_bits_to_f64(inp.k), inp.wk.astype(np.float64), c64, s64,
                                           w.eps))
    ro, rl = orc.attention(q, k, inputs.bf16_bits_to_f64(inp.v), w.scale)
    check_o(host_f64(o), ro, what="qwen_image every element")
    check_lse(host_f64(lse), rl, what="qwen_image every element")
