"""GPU parity of each kernel against the fp64 oracle on small seeded inputs that
span several tiles and ragged tails (all elements compared)."""

import math

import numpy as np
import pytest

import oracle
from diffusion_transformer_attention_dit_gb300 import build, inputs, ops
from parity import (check_bf16_rounding, check_lse, check_o, dev_bf16, dev_f32, host_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu


def vmax(v_bits) -> float:
    return float(np.abs(inputs.bf16_bits_to_f64(v_bits)).max())


@pytest.fixture(scope="module", autouse=True)
def _lib():
    build.build()
    ops.load_library()
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"


@pytest.fixture(scope="module")
def orc():
    return oracle.get()


# ---------------------------------------------------------------- prologue

@pytest.mark.parametrize("B,S,H,D", [(1, 256, 2, 64), (2, 37, 3, 128), (1, 129, 40, 128), (3, 5, 1, 64)])
def test_qk_norm_rope_parity(orc, B, S, H, D):
    q, k, _, wq, wk, cos, sin = inputs.small_case(B, S, H, D, seed=100 + S)
    qo, ko = ops.qk_norm_rope(dev_bf16(q), dev_bf16(k), dev_f32(wq), dev_f32(wk), dev_f32(cos), dev_f32(sin), 1e-6)
    for got, x, w in [(qo, q, wq), (ko, k, wk)]:
        ref = orc.qk_norm_rope(inputs.bf16_bits_to_f64(x), w.astype(np.float64), cos.astype(np.float64),
                               sin.astype(np.float64), 1e-6)
        check_bf16_rounding(host_f64(got), ref, "prologue")


def test_qk_norm_rope_in_place(orc):
    q, k, _, wq, wk, cos, sin = inputs.small_case(1, 64, 4, 128, seed=7)
    tq, tk = dev_bf16(q), dev_bf16(k)
    ref_q, ref_k = ops.qk_norm_rope(tq, tk, dev_f32(wq), dev_f32(wk), dev_f32(cos), dev_f32(sin))
    ops.qk_norm_rope(tq, tk, dev_f32(wq), dev_f32(wk), dev_f32(cos), dev_f32(sin), q_out=tq, k_out=tk)
    assert torch.equal(tq, ref_q) and torch.equal(tk, ref_k)


# ---------------------------------------------------------------- attention

SHAPES = [
    # B, H, Sq, Skv, D
    (1, 2, 256, 256, 64),
    (1, 2, 256, 256, 128),
    (2, 3, 200, 333, 128),
    (1, 1, 1, 1, 128),
    (1, 2, 1, 700, 64),
    (1, 1, 517, 3, 128),
    (2, 2, 300, 129, 64),
]


@pytest.mark.parametrize("B,H,Sq,Skv,D", SHAPES)
@pytest.mark.parametrize("o_dtype", ["bf16", "f32"])
def test_attn_fwd_full_parity(orc, B, H, Sq, Skv, D, o_dtype):
    q, k, v, *_ = inputs.small_case(B, Sq, H, D, seed=Sq * 7 + Skv, Skv=Skv)
    dt = torch.bfloat16 if o_dtype == "bf16" else torch.float32
    scale = 1.0 / math.sqrt(D)
    o, lse = ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v), scale, o_dtype=dt)
    ro, rl = orc.attention(inputs.bf16_bits_to_f64(q), inputs.bf16_bits_to_f64(k), inputs.bf16_bits_to_f64(v), scale)
    check_o(host_f64(o), ro, f32=o_dtype == "f32", what=f"attn {B, H, Sq, Skv, D}", vmax=vmax(v))
    check_lse(host_f64(lse), rl, what=f"attn {B, H, Sq, Skv, D}")


@pytest.mark.parametrize("lo,hi", [(0, 64), (64, 128), (5, 6), (100, 333), (0, 333), (129, 300)])
def test_attn_fwd_chunk_parity(orc, lo, hi):
    B, H, Sq, Skv, D = 2, 2, 150, 333, 128
    q, k, v, *_ = inputs.small_case(B, Sq, H, D, seed=31, Skv=Skv, k_std=2.0)
    o, lse = ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v), 0.1, lo, hi, o_dtype=torch.float32)
    ro, rl = orc.attention(inputs.bf16_bits_to_f64(q), inputs.bf16_bits_to_f64(k), inputs.bf16_bits_to_f64(v), 0.1,
                           lo, hi)
    check_o(host_f64(o), ro, f32=True, what=f"chunk [{lo},{hi})", vmax=vmax(v[:, lo:hi]))
    check_lse(host_f64(lse), rl, what=f"chunk [{lo},{hi})")


def test_attn_fwd_strided_views(orc):
    """q/k/v as views into a packed [B, S, 3, H, D] QKV buffer and O into a wider buffer."""
    B, S, H, D = 1, 190, 3, 64
    bits = inputs.bf16_normal(B * S * 3 * H * D, seed=44).reshape(B, S, 3, H, D)
    qkv = dev_bf16(bits)
    q, k, v = qkv[:, :, 0], qkv[:, :, 1], qkv[:, :, 2]
    o_buf = torch.zeros((B, S, H, 2 * D), dtype=torch.bfloat16, device="cuda")
    o = o_buf[..., :D]
    _, lse = ops.attn_fwd(q, k, v, 0.125, o=o)
    f = inputs.bf16_bits_to_f64(bits)
    ro, rl = orc.attention(f[:, :, 0], f[:, :, 1], f[:, :, 2], 0.125)
    check_o(host_f64(o), ro, what="strided")
    check_lse(host_f64(lse), rl, what="strided")
    assert torch.count_nonzero(o_buf[..., D:]) == 0, "kernel wrote outside the O view"


def test_attn_fwd_deterministic():
    q, k, v, *_ = inputs.small_case(1, 300, 4, 128, seed=9)
    args = [dev_bf16(q), dev_bf16(k), dev_bf16(v)]
    o1, l1 = ops.attn_fwd(*args)
    o2, l2 = ops.attn_fwd(*args)
    assert torch.equal(o1, o2) and torch.equal(l1, l2)


def test_attn_fwd_sharp_softmax_rescale(orc):
    """Large logits (K x 8) make the running max grow between blocks: exercises the O rescale path."""
    B, H, S, D = 1, 2, 640, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=77, k_std=8.0)
    o, lse = ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v), 1 / math.sqrt(D), o_dtype=torch.float32)
    ro, rl = orc.attention(inputs.bf16_bits_to_f64(q), inputs.bf16_bits_to_f64(k), inputs.bf16_bits_to_f64(v),
                           1 / math.sqrt(D))
    check_o(host_f64(o), ro, f32=True, what="sharp", vmax=vmax(v))
    check_lse(host_f64(lse), rl, what="sharp")


def test_attn_fwd_rescale_with_growing_scores(orc):
    """Keys whose scores rise by about 20 (base-2 units) from one 128-key block to the next: every row's running
    max is raised, and O rescaled, on every block."""
    B, H, S, D = 1, 2, 640, 128
    rng = np.random.default_rng(12)
    q = np.ones((B, S, H, D), np.float32) + 0.05 * rng.standard_normal((B, S, H, D)).astype(np.float32)
    ramp = (np.arange(S) // 128).astype(np.float32)[None, :, None, None] * 1.25
    k = ramp * np.ones((B, S, H, D), np.float32) + 0.05 * rng.standard_normal((B, S, H, D)).astype(np.float32)
    v = rng.standard_normal((B, S, H, D)).astype(np.float32)
    qb, kb, vb = (inputs.f32_to_bf16_bits(x) for x in (q, k, v))
    scale = 1 / math.sqrt(D)
    o, lse = ops.attn_fwd(dev_bf16(qb), dev_bf16(kb), dev_bf16(vb), scale, o_dtype=torch.float32)
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (qb, kb, vb)), scale)
    check_o(host_f64(o), ro, f32=True, what="growing scores", vmax=vmax(vb))
    check_lse(host_f64(lse), rl, what="growing scores")


# ---------------------------------------------------------------- merge

@pytest.mark.parametrize("C", [1, 2, 3, 8, 20])  # 20 parts take the register (non-bulk) path
@pytest.mark.parametrize("in_dt,out_dt", [("bf16", "bf16"), ("f32", "f32"), ("f32", "bf16"), ("bf16", "f32")])
def test_merge_parity(orc, C, in_dt, out_dt):
    B, Sq, H, D = 2, 77, 3, 128
    rng = np.random.default_rng(C)
    dts = {"bf16": torch.bfloat16, "f32": torch.float32}
    o_parts = torch.from_numpy(rng.normal(0, 1, (C, B, Sq, H, D)).astype(np.float32)).cuda().to(dts[in_dt])
    lse_np = rng.normal(3, 2, (C, B, H, Sq)).astype(np.float32)
    lse_np[0, 0, 0, :5] = -np.inf          # an empty block for a few rows
    if C > 1:
        lse_np[:, 1, 2, 7] = -np.inf       # every block empty for one row
    lse_parts = torch.from_numpy(lse_np).cuda()
    o, lse = ops.attn_merge_lse(o_parts, lse_parts, out_dtype=dts[out_dt])
    ro, rl = orc.merge_lse(host_f64(o_parts), lse_np.astype(np.float64))
    got_o, got_l = host_f64(o), host_f64(lse)
    finite = np.isfinite(rl)
    assert np.array_equal(finite, np.isfinite(got_l))
    np.testing.assert_allclose(got_l[finite], rl[finite], rtol=0, atol=2e-6 * (1 + np.abs(rl[finite]).max()))
    if out_dt == "f32":
        np.testing.assert_allclose(got_o, ro, rtol=1e-5, atol=1e-5)
    else:
        check_bf16_rounding(got_o, ro, "merge")
    if C > 1:
        assert np.all(got_o[1, 7, 2] == 0)


@pytest.mark.parametrize("C,partial", [(2, "f32"), (4, "bf16"), (4, "f32"), (7, "f32")])
def test_chunked_merged_equals_full(orc, C, partial):
    """chunk-mode attention over C key blocks merged by LSE == single-pass attention (and the oracle)."""
    B, H, S, D = 1, 3, 500, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=C * 11, k_std=3.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    dt = torch.float32 if partial == "f32" else torch.bfloat16
    edges = [(i * S) // C for i in range(C + 1)]
    o_parts = torch.empty((C, B, S, H, D), dtype=dt, device="cuda")
    lse_parts = torch.empty((C, B, H, S), dtype=torch.float32, device="cuda")
    for c in range(C):
        ops.attn_fwd(tq, tk, tv, None, edges[c], edges[c + 1], o=o_parts[c], lse=lse_parts[c])
    om, lm = ops.attn_merge_lse(o_parts, lse_parts, out_dtype=torch.bfloat16)
    of, lf = ops.attn_fwd(tq, tk, tv)
    ro, rl = orc.attention(inputs.bf16_bits_to_f64(q), inputs.bf16_bits_to_f64(k), inputs.bf16_bits_to_f64(v),
                           1 / math.sqrt(D))
    check_o(host_f64(om), ro, what="merged vs oracle")
    check_lse(host_f64(lm), rl, what="merged vs oracle")
    check_o(host_f64(om), host_f64(of), what="merged vs single pass")
    check_lse(host_f64(lm), host_f64(lf), what="merged vs single pass")
    # a ring loop that never merges returns one block's own output: make sure we do not
    for c in range(C):
        assert (host_f64(om) - host_f64(o_parts[c])).__abs__().max() > 0.05


@pytest.mark.parametrize("edges,partial", [
    ([0, 1, 64, 65, 300, 500], "f32"),              # unequal chunks, two of one key
    ([0, 1, 64, 65, 300, 500], "bf16"),
    ([0, 500], "f32"),                              # C = 1: the merge of one part is that part
    ([0, 63, 127, 128, 250, 251, 380, 499, 500], "f32"),  # C = 8, ragged against the 128-key blocks
])
def test_merged_unequal_chunks_equal_single_pass(orc, edges, partial):
    """Unequal key chunks (including chunks of one key, C = 1 and C = 8) merged by LSE: every element against the
    single pass on the GPU and against the oracle."""
    B, H, S, D = 2, 3, 500, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=len(edges) * 13, k_std=2.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    dt = torch.float32 if partial == "f32" else torch.bfloat16
    C = len(edges) - 1
    o_parts = torch.empty((C, B, S, H, D), dtype=dt, device="cuda")
    lse_parts = torch.empty((C, B, H, S), dtype=torch.float32, device="cuda")
    for c in range(C):
        ops.attn_fwd(tq, tk, tv, None, edges[c], edges[c + 1], o=o_parts[c], lse=lse_parts[c])
    om, lm = ops.attn_merge_lse(o_parts, lse_parts, out_dtype=torch.bfloat16)
    of, lf = ops.attn_fwd(tq, tk, tv)
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D))
    check_o(host_f64(om), ro, what=f"merged {edges} vs oracle")
    check_lse(host_f64(lm), rl, what=f"merged {edges} vs oracle")
    check_o(host_f64(om), host_f64(of), what=f"merged {edges} vs single pass")
    check_lse(host_f64(lm), host_f64(lf), what=f"merged {edges} vs single pass")


@pytest.mark.parametrize("S", [1, 63, 64, 127, 129, 200, 4312])
@pytest.mark.parametrize("D", [64, 128])
def test_attn_fwd_tail_lengths(orc, S, D):
    """Sequence lengths around the 128-row tiles and 128-key blocks (and the Qwen-Image length), every element
    against the oracle."""
    B, H = 1, 2
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=S * 3 + D)
    o, lse = ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v))
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D))
    check_o(host_f64(o), ro, what=f"S {S} D {D}")
    check_lse(host_f64(lse), rl, what=f"S {S} D {D}")


def test_fp32_partials_merge_closer_to_the_oracle_than_bf16(orc):
    """Ring attention that merges bf16-rounded block outputs loses accuracy (the reason this library offers fp32
    partials).  On the Wan2.2-720p-style sharp softmax (K drawn x 3, 8 KV chunks, stacked partials + merge kernel,
    fp32 output so the final rounding does not hide the difference) both are within the bf16 bar, and the fp32
    partials are measurably closer to the oracle: the RMS error with bf16 partials is 1.84x that with fp32
    partials on these inputs (the kernel is bitwise deterministic, so the ratio repeats exactly); the bar is
    1.5x.  Both share the rounding of P to bf16 before PV; the bf16 partials add one rounding of every chunk's
    O before the merge."""
    B, H, S, D, C = 1, 4, 2048, 128, 8
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=720, k_std=3.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D))
    rms = {}
    for name, pdt in (("f32", torch.float32), ("bf16", torch.bfloat16)):
        o, lse = ops.dit_attention(tq, tk, tv, None, None, None, None, chunks=C, partial_dtype=pdt,
                                   out_dtype=torch.float32, prologue=False, merge="kernel")
        ops.poll_device_error()
        got = host_f64(o)
        check_o(got, ro, what=f"{name} partials merged")  # the bf16-output bar holds for both
        check_lse(host_f64(lse), rl, what=f"{name} partials merged")
        rms[name] = float(np.sqrt(((got - ro) ** 2).mean()))
    print(f"merged-vs-oracle RMS error: fp32 partials {rms['f32']:.3e}, bf16 partials {rms['bf16']:.3e}, "
          f"ratio {rms['bf16'] / rms['f32']:.2f}")
    assert rms["bf16"] >= 1.5 * rms["f32"], rms


# ---------------------------------------------------------------- update form (merge in the epilogue)

UPDATE_SHAPES = [
    # B, H, Sq, Skv, D, split
    (1, 2, 256, 256, 128, 128),
    (2, 3, 200, 333, 128, 129),
    (1, 2, 517, 300, 64, 37),
    (1, 1, 1, 2, 128, 1),
    (2, 2, 300, 700, 64, 650),
]


@pytest.mark.parametrize("B,H,Sq,Skv,D,split", UPDATE_SHAPES)
@pytest.mark.parametrize("acc_dt,out_dt", [("f32", "bf16"), ("f32", "f32"), ("bf16", "bf16"), ("bf16", "f32")])
def test_attn_update_parity(orc, B, H, Sq, Skv, D, split, acc_dt, out_dt):
    """Chunk [0, split) as the running result, then [split, Skv) merged into it in the epilogue == full attention."""
    dts = {"bf16": torch.bfloat16, "f32": torch.float32}
    q, k, v, *_ = inputs.small_case(B, Sq, H, D, seed=Sq + 5 * Skv + split, Skv=Skv, k_std=2.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    acc, lse_acc = ops.attn_fwd(tq, tk, tv, None, 0, split, o_dtype=dts[acc_dt])
    o, lse = ops.attn_fwd_update(tq, tk, tv, acc, lse_acc, None, split, Skv, o_dtype=dts[out_dt])
    f = [inputs.bf16_bits_to_f64(x) for x in (q, k, v)]
    ro, rl = orc.attention(*f, 1 / math.sqrt(D))
    strict = acc_dt == "f32" and out_dt == "f32"
    check_o(host_f64(o), ro, f32=strict, what=f"update {B, H, Sq, Skv, D, split}", vmax=vmax(v))
    check_lse(host_f64(lse), rl, what=f"update {B, H, Sq, Skv, D, split}")
    assert torch.equal(lse_acc, ops.attn_fwd(tq, tk, tv, None, 0, split, o_dtype=dts[acc_dt])[1]), \
        "the running LSE must not be written when it is not the output"


@pytest.mark.parametrize("C", [3, 4, 7])
def test_attn_update_chain_in_place(orc, C):
    """C chunks folded into an fp32 running result in place, the last straight into bf16: == merge kernel == oracle."""
    B, H, S, D = 1, 3, 500, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=C * 13, k_std=3.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    edges = [(i * S) // C for i in range(C + 1)]
    acc, lse = ops.attn_fwd(tq, tk, tv, None, edges[0], edges[1], o_dtype=torch.float32)
    for c in range(1, C - 1):
        ops.attn_fwd_update(tq, tk, tv, acc, lse, None, edges[c], edges[c + 1], o=acc, lse=lse)
    o = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
    ops.attn_fwd_update(tq, tk, tv, acc, lse, None, edges[-2], edges[-1], o=o, lse=lse)
    f = [inputs.bf16_bits_to_f64(x) for x in (q, k, v)]
    ro, rl = orc.attention(*f, 1 / math.sqrt(D))
    check_o(host_f64(o), ro, what=f"update chain C={C}")
    check_lse(host_f64(lse), rl, what=f"update chain C={C}")
    om, lm = ops.dit_attention(tq, tk, tv, None, None, None, None, chunks=C, prologue=False, merge="kernel")
    check_o(host_f64(o), host_f64(om), what="update chain vs merge kernel")
    check_lse(host_f64(lse), host_f64(lm), what="update chain vs merge kernel")
    ou, lu = ops.dit_attention(tq, tk, tv, None, None, None, None, chunks=C, prologue=False, merge="update")
    assert torch.equal(ou, o) and torch.equal(lu, lse)


def test_attn_update_causal_and_empty_rows(orc):
    """Causal ranges in both orders: rows that see nothing in one part take the other part unchanged, and rows
    that see nothing in either give O = 0, LSE = -inf."""
    B, H, S, D = 1, 2, 600, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=62)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    f = [inputs.bf16_bits_to_f64(x) for x in (q, k, v)]
    ro, rl = orc.attention(*f, 1 / math.sqrt(D), causal=True)
    for first, second in [((0, 260), (260, 600)), ((260, 600), (0, 260))]:
        acc, lse_acc = ops.attn_fwd(tq, tk, tv, None, *first, o_dtype=torch.float32, causal=True)
        o, lse = ops.attn_fwd_update(tq, tk, tv, acc, lse_acc, None, *second, o_dtype=torch.float32, causal=True)
        check_o(host_f64(o), ro, f32=True, what=f"causal update {first} {second}", vmax=vmax(v))
        check_lse(host_f64(lse), rl, what=f"causal update {first} {second}")
    # rows < 400 see no key of [400, 600): both parts empty for them
    acc, lse_acc = ops.attn_fwd(tq, tk, tv, None, 400, 500, o_dtype=torch.float32, causal=True)
    o, lse = ops.attn_fwd_update(tq, tk, tv, acc, lse_acc, None, 500, 600, o_dtype=torch.float32, causal=True)
    got_o, got_l = host_f64(o), host_f64(lse)
    assert np.all(got_o[:, :400] == 0) and np.all(np.isneginf(got_l[:, :, :400]))
    ro2, rl2 = orc.attention(*f, 1 / math.sqrt(D), 400, 600, causal=True)
    check_o(got_o[:, 400:], ro2[:, 400:], f32=True, what="causal update tail", vmax=vmax(v))
    check_lse(got_l[:, :, 400:], rl2[:, :, 400:], what="causal update tail")


def test_attn_update_strided_running_result(orc):
    """The running result as an fp32 view into a wider buffer; nothing outside the views is written."""
    B, S, H, D = 1, 190, 3, 64
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=45)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    acc_buf = torch.zeros((B, S, H, 2 * D), dtype=torch.float32, device="cuda")
    acc = acc_buf[..., :D]
    _, lse_acc = ops.attn_fwd(tq, tk, tv, None, 0, 90, o=acc)
    o_buf = torch.zeros((B, S, H, 2 * D), dtype=torch.bfloat16, device="cuda")
    o, lse = ops.attn_fwd_update(tq, tk, tv, acc, lse_acc, None, 90, S, o=o_buf[..., :D])
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D))
    check_o(host_f64(o), ro, what="update strided")
    check_lse(host_f64(lse), rl, what="update strided")
    assert torch.count_nonzero(o_buf[..., D:]) == 0 and torch.count_nonzero(acc_buf[..., D:]) == 0


def test_launch_overlap_gives_identical_results():
    """Programmatic dependent launch changes only when a kernel starts: the back-to-back chain prologue ->
    chunk attention -> update -> merge gives bit-identical results with it on and off."""
    inp = inputs.make_inputs("tiny")
    w = inp.w
    args = [dev_bf16(inp.q), dev_bf16(inp.k), dev_bf16(inp.v), dev_f32(inp.wq), dev_f32(inp.wk), dev_f32(inp.cos),
            dev_f32(inp.sin)]
    res = {}
    for on in (False, True):
        ops.set_launch_overlap(on)
        try:
            res[on] = [ops.dit_attention(*args, eps=w.eps, chunks=4, merge=m) for m in ("update", "kernel")]
            torch.cuda.synchronize()
        finally:
            ops.set_launch_overlap(True)
    for (o0, l0), (o1, l1) in zip(res[False], res[True]):
        assert torch.equal(o0, o1) and torch.equal(l0, l1)


def test_poll_device_error_clean():
    q, k, v, *_ = inputs.small_case(1, 128, 1, 64, seed=3)
    ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v))
    ops.poll_device_error()


def test_full_hot_path_tiny(orc):
    """Prologue + 4 KV chunks + merge on the tiny workload, bf16 and fp32 outputs."""
    inp = inputs.make_inputs("tiny")
    w = inp.w
    dq = dev_bf16(inp.q)
    dk = dev_bf16(inp.k)
    dv = dev_bf16(inp.v)
    args = (dev_f32(inp.wq), dev_f32(inp.wk), dev_f32(inp.cos), dev_f32(inp.sin))
    f = {n: inputs.bf16_bits_to_f64(getattr(inp, n)) for n in ("q", "k", "v")}
    # the prologue hands bf16 Q/K to attention, so the oracle chain rounds there too
    rq = oracle.round_bf16(orc.qk_norm_rope(f["q"], inp.wq.astype(np.float64), inp.cos.astype(np.float64),
                                            inp.sin.astype(np.float64), w.eps))
    rk = oracle.round_bf16(orc.qk_norm_rope(f["k"], inp.wk.astype(np.float64), inp.cos.astype(np.float64),
                                            inp.sin.astype(np.float64), w.eps))
    parts = [orc.attention(rq, rk, f["v"], w.scale, lo, hi) for lo, hi in w.chunk_bounds()]
    ro, rl = orc.merge_lse(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    for out_dt, part_dt in [(torch.bfloat16, torch.bfloat16), (torch.float32, torch.float32)]:
        o, lse = ops.dit_attention(dq, dk, dv, *args, eps=w.eps, chunks=w.chunks, partial_dtype=part_dt,
                                   out_dtype=out_dt)
        check_o(host_f64(o), ro, f32=out_dt == torch.float32, what="tiny hot path", vmax=vmax(inp.v))
        check_lse(host_f64(lse), rl, what="tiny hot path")


def test_bounded_wait_times_out_and_context_survives():
    """A wait on a barrier nothing completes gives up (~2 s) and is reported; later launches still work."""
    import time

    ops.poll_device_error()  # clear
    t0 = time.time()
    ops.selftest_wait_timeout()
    with pytest.raises(ops.DitError) as e:
        ops.poll_device_error()
    assert e.value.status == ops.DIT_ERR_TIMEOUT
    assert time.time() - t0 < 30
    ops.poll_device_error()  # cleared by the previous poll
    q, k, v, *_ = inputs.small_case(1, 128, 1, 64, seed=5)
    o, _ = ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v))
    assert torch.isfinite(o.float()).all()


# ---------------------------------------------------------------- causal variant

@pytest.mark.parametrize("B,H,Sq,Skv,D", [(1, 2, 256, 256, 64), (2, 3, 200, 333, 128), (1, 1, 517, 300, 128),
                                          (1, 2, 700, 700, 128), (1, 1, 1, 1, 64)])
def test_attn_fwd_causal_parity(orc, B, H, Sq, Skv, D):
    q, k, v, *_ = inputs.small_case(B, Sq, H, D, seed=Sq + 3 * Skv, Skv=Skv, k_std=2.0)
    o, lse = ops.attn_fwd(dev_bf16(q), dev_bf16(k), dev_bf16(v), o_dtype=torch.float32, causal=True)
    f = [inputs.bf16_bits_to_f64(x) for x in (q, k, v)]
    ro, rl = orc.attention(*f, 1 / math.sqrt(D), causal=True)
    check_o(host_f64(o), ro, f32=True, what=f"causal {B, H, Sq, Skv, D}", vmax=vmax(v))
    check_lse(host_f64(lse), rl, what=f"causal {B, H, Sq, Skv, D}")


def test_attn_fwd_causal_chunks_merge(orc):
    """Causal key chunks: rows before a chunk see nothing (O = 0, LSE = -inf); merged chunks = full causal."""
    B, H, S, D = 1, 2, 600, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=61)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    bounds = [(0, 150), (150, 389), (389, 600)]
    o_parts = torch.empty((3, B, S, H, D), dtype=torch.float32, device="cuda")
    lse_parts = torch.empty((3, B, H, S), dtype=torch.float32, device="cuda")
    f = [inputs.bf16_bits_to_f64(x) for x in (q, k, v)]
    for c, (lo, hi) in enumerate(bounds):
        ops.attn_fwd(tq, tk, tv, None, lo, hi, o=o_parts[c], lse=lse_parts[c], causal=True)
        ro, rl = orc.attention(*f, 1 / math.sqrt(D), lo, hi, causal=True)
        got_l = host_f64(lse_parts[c])
        assert np.array_equal(np.isinf(got_l), np.isinf(rl))
        assert np.all(host_f64(o_parts[c])[:, :lo] == 0)
        fin = np.isfinite(rl)
        assert np.abs(got_l[fin] - rl[fin]).max() <= 1e-3
        check_o(host_f64(o_parts[c])[:, lo:], ro[:, lo:], f32=True, what=f"causal chunk {lo, hi}", vmax=vmax(v))
    om, lm = ops.attn_merge_lse(o_parts, lse_parts, out_dtype=torch.float32)
    ro, rl = orc.attention(*f, 1 / math.sqrt(D), causal=True)
    check_o(host_f64(om), ro, f32=True, what="causal merged", vmax=vmax(v))
    check_lse(host_f64(lm), rl, what="causal merged")


# ---------------------------------------------------------------- LayerNorm-modulate / RMSNorm over C

# odd L: a row pair of the two-row kernel straddles two batch entries; an odd row
# count leaves a last pair of one row; (3, 1001, 1024) and (2, 2049, 5120) give
# every CTA several pairs; C = 7168 is the widest row of the two-row kernel,
# C = 8192 the one-row kernel's
@pytest.mark.parametrize("B,L,C", [(2, 37, 3072), (1, 130, 5120), (3, 5, 8), (1, 7, 8192), (2, 300, 128),
                                   (3, 3, 7168), (3, 1001, 1024), (2, 2049, 5120), (2, 65, 4096), (1, 33, 6144),
                                   (4, 1, 512), (1, 1, 256)])  # every pair straddles; one row
def test_layer_norm_modulate_parity(orc, B, L, C):
    rng = np.random.default_rng(C + L)
    x = inputs.bf16_normal(B * L * C, seed=C + 7, std=2.0, mean=0.3).reshape(B, L, C)
    scale = rng.normal(0, 0.3, (B, C)).astype(np.float32)
    shift = rng.normal(0, 0.3, (B, C)).astype(np.float32)
    y = ops.layer_norm_modulate(dev_bf16(x), dev_f32(scale), dev_f32(shift), 1e-6)
    ref = orc.layer_norm_modulate(inputs.bf16_bits_to_f64(x), scale.astype(np.float64), shift.astype(np.float64), 1e-6)
    check_bf16_rounding(host_f64(y), ref, "ln modulate", atol=2e-5)
    y0 = ops.layer_norm_modulate(dev_bf16(x), None, None, 1e-6)
    ref0 = orc.layer_norm_modulate(inputs.bf16_bits_to_f64(x), None, None, 1e-6)
    check_bf16_rounding(host_f64(y0), ref0, "plain ln", atol=2e-5)


@pytest.mark.parametrize("rows,C", [(37, 5120), (300, 3072), (1, 8)])
def test_rms_norm_over_channels_parity(orc, rows, C):
    x = inputs.bf16_normal(rows * C, seed=rows + C).reshape(rows, C)
    w = inputs.f32_normal(C, seed=C, std=0.1, mean=1.0)
    tx = dev_bf16(x)
    y = ops.rms_norm(tx, dev_f32(w), 1e-6)
    ref = orc.rms_norm(inputs.bf16_bits_to_f64(x), w.astype(np.float64), 1e-6)
    check_bf16_rounding(host_f64(y), ref, "rms over C")
    ops.rms_norm(tx, dev_f32(w), 1e-6, y=tx)  # in place
    assert torch.equal(tx, y)


# ---------------------------------------------------------------- ring-overlap emulation

def test_ring_overlap_equals_full_attention(orc):
    """Local FA || gather of 3 remote chunks on a side stream, FA over the gathered keys, LSE merge == full."""
    B, H, S, D = 1, 4, 1000, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=91, k_std=2.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    bounds = [(0, 250), (250, 500), (500, 800), (800, 1000)]  # rank 0 local, ranks 1-3 remote
    remote = [(tk[:, lo:hi].contiguous(), tv[:, lo:hi].contiguous()) for lo, hi in bounds[1:]]
    o, lse = ops.ring_overlap_attention(tq, tk[:, :250].contiguous(), tv[:, :250].contiguous(), remote)
    torch.cuda.synchronize()
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D))
    check_o(host_f64(o), ro, what="ring overlap")
    check_lse(host_f64(lse), rl, what="ring overlap")


@pytest.mark.parametrize("B,H,D,local,remote_lens,pdt", [
    (2, 3, 128, 300, [129, 1, 400], "f32"),   # batch of 2 (strided gather), ragged shards, a one-key shard
    (1, 2, 64, 64, [64, 64, 64, 64, 64, 64, 64], "bf16"),
    (1, 4, 128, 517, [], "f32"),              # a ring of one rank: plain attention
])
def test_ring_overlap_equals_its_entry_points(orc, B, H, D, local, remote_lens, pdt):
    """dit_attention_ring_overlap == dit_attn_fwd over the local shard then dit_attn_fwd_update over the
    concatenated remote shards, bit for bit; and == the oracle's attention over all keys."""
    dts = {"bf16": torch.bfloat16, "f32": torch.float32}
    S = local + sum(remote_lens)
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=S + B, k_std=2.0)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    edges = [local]
    for n in remote_lens:
        edges.append(edges[-1] + n)
    remote = [(tk[:, a:b].contiguous(), tv[:, a:b].contiguous()) for a, b in zip(edges[:-1], edges[1:])]
    kl, vl = tk[:, :local].contiguous(), tv[:, :local].contiguous()
    o, lse = ops.ring_overlap_attention(tq, kl, vl, remote, partial_dtype=dts[pdt])
    if remote_lens:
        acc, rl = ops.attn_fwd(tq, kl, vl, o_dtype=dts[pdt])
        ro, rl = ops.attn_fwd_update(tq, tk[:, local:].contiguous(), tv[:, local:].contiguous(), acc, rl, lse=rl)
    else:
        ro, rl = ops.attn_fwd(tq, kl, vl)
    torch.cuda.synchronize()
    ops.poll_device_error()
    assert torch.equal(o, ro) and torch.equal(lse, rl)
    fo, fl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D))
    check_o(host_f64(o), fo, what="ring overlap", vmax=vmax(v))
    check_lse(host_f64(lse), fl, what="ring overlap")


# ---------------------------------------------------------------- W8A8 fp8

@pytest.mark.parametrize("M,K", [(7, 3072), (300, 128), (1, 16), (64, 8192)])
def test_quant_fp8_rows_bit_exact(orc, M, K):
    x = inputs.bf16_normal(M * K, seed=M * 13 + K, std=3.0).reshape(M, K)
    x[0, :] = 0 if M > 1 else x[0, :]
    codes, scale = ops.quant_fp8_rows(dev_bf16(x))
    rc, rs = orc.quant_fp8_rows(inputs.bf16_bits_to_f64(x))
    assert np.array_equal(scale.cpu().numpy(), rs)
    assert np.array_equal(codes.cpu().numpy(), rc)


def test_quant_fp8_division_matches_ieee_on_every_input():
    """The quantiser's Markstein division gives the e4m3 code of IEEE division for every bf16 row maximum and every
    bf16 element it can meet: about 2.1e9 pairs, evaluated on the device.  The fp32 quotient itself may differ (it is
    not an output); it does in about 0.1 % of the pairs, never by enough to change a code."""
    fp32_diff, code_diff = ops.selftest_fp8_quotients()
    assert code_diff == 0, (fp32_diff, code_diff)
    assert fp32_diff < 2.1e9 * 0.01, fp32_diff


def test_quant_fp8_rows_tiny_and_signed_zero_rows(orc):
    """Rows whose scale falls below the fast path's range (max magnitude ~1e-30) divide exactly too; -0 keeps its
    sign (code 0x80); an all-zero row gets scale 1."""
    rng = np.random.default_rng(5)
    K = 256
    x = rng.normal(0, 1, (4, K)).astype(np.float32)
    x[1] *= 1e-30
    x[2] = 0.0
    x[2, :7] = -0.0
    x[3, 3] = -0.0
    bits = inputs.f32_to_bf16_bits(x)
    codes, scale = ops.quant_fp8_rows(dev_bf16(bits))
    ref_codes, ref_scale = orc.quant_fp8_rows(inputs.bf16_bits_to_f64(bits).astype(np.float32))
    assert np.array_equal(codes.cpu().numpy().view(np.uint8), ref_codes)
    assert np.array_equal(scale.cpu().numpy(), ref_scale)
    assert codes.cpu().numpy().view(np.uint8)[2, 0] == 0x80 and scale.cpu().numpy()[2] == 1.0


def _fp8_operands(orc, M, N, K, seed, a_std=2.0, b_std=0.05):
    """Seeded bf16 activations and weights quantised by the oracle (host); codes and scales go to the GPU."""
    xa = inputs.bf16_normal(M * K, seed=seed, std=a_std).reshape(M, K)
    xb = inputs.bf16_normal(N * K, seed=seed + 1, std=b_std).reshape(N, K)
    a, sa = orc.quant_fp8_rows(inputs.bf16_bits_to_f64(xa))
    b, sb = orc.quant_fp8_rows(inputs.bf16_bits_to_f64(xb))
    dev = [torch.from_numpy(np.ascontiguousarray(t)).cuda() for t in (a, sa, b, sb)]
    return (a, sa, b, sb), dev


@pytest.mark.parametrize("M,N,K", [(256, 512, 256), (300, 264, 208), (1, 8, 16), (520, 768, 1024),
                                   (4100, 1288, 256)])  # the last: 102 tiles of 256 x 256, so CTA pairs take two,
# ragged N; M = 1 and 300 leave the second CTA of a pair rows wholly past M
def test_gemm_fp8_parity(orc, M, N, K):
    (a, sa, b, sb), (da, dsa, db, dsb) = _fp8_operands(orc, M, N, K, seed=M + 3 * N + K)
    out = ops.gemm_fp8(da, dsa, db, dsb)
    ref = orc.gemm_fp8(a, sa, b, sb)
    # fp32 accumulation of exact e4m3 products, two fp32 scale multiplies, one bf16 rounding
    check_bf16_rounding(host_f64(out), ref, "fp8 gemm", atol=1e-5 * np.abs(ref).max())


def test_gemm_fp8_strided_output(orc):
    M, N, K = 130, 72, 64
    (a, sa, b, sb), (da, dsa, db, dsb) = _fp8_operands(orc, M, N, K, seed=5, a_std=1.0, b_std=1.0)
    buf = torch.zeros((M, N + 40), dtype=torch.bfloat16, device="cuda")
    ops.gemm_fp8(da, dsa, db, dsb, out=buf[:, :N])
    ref = orc.gemm_fp8(a, sa, b, sb)
    check_bf16_rounding(host_f64(buf[:, :N]), ref, "fp8 gemm strided", atol=1e-5 * np.abs(ref).max())
    assert torch.count_nonzero(buf[:, N:]) == 0


@pytest.mark.parametrize("M,N,K", [(17248, 9216, 3072), (32760, 15360, 5120)])
def test_gemm_fp8_qkv_projection_full_size(orc, M, N, K):
    """The QKV projections of Qwen-Image-Edit (17248 tokens x 9216 x 3072) and Wan2.2 480p (32760 x 15360 x
    5120) in the launch bench.py times: every CTA pair runs 32-33 (Edit) or 101-102 (Wan480) tiles of 256 x
    256, and the last tile row holds 96 or 248 tokens; sampled output rows against the oracle."""
    # any e4m3 codes are valid GEMM operands: seeded random bytes (NaN codes replaced) and scales
    rng = np.random.default_rng(97 + K)
    a = rng.integers(0, 256, (M, K), dtype=np.uint8)
    b = rng.integers(0, 256, (N, K), dtype=np.uint8)
    a[(a & 0x7F) == 0x7F] = 0x38
    b[(b & 0x7F) == 0x7F] = 0x38
    sa = rng.uniform(1e-3, 1e-2, M).astype(np.float32)
    sb = rng.uniform(1e-4, 1e-3, N).astype(np.float32)
    da, dsa, db, dsb = (torch.from_numpy(t).cuda() for t in (a, sa, b, sb))
    out = ops.gemm_fp8(da, dsa, db, dsb)
    from parity import sample_rows
    rows = sample_rows(M, 40, seed=3)
    ref = orc.gemm_fp8(np.ascontiguousarray(a[rows]), np.ascontiguousarray(sa[rows]), b, sb)
    got = host_f64(out[torch.from_numpy(rows).cuda()])
    check_bf16_rounding(got, ref, "fp8 gemm full size", atol=1e-5 * np.abs(ref).max())


def test_w8a8_projection_accuracy():
    """W8A8 (per-token activations, per-channel weights, e4m3) against the exact product of the bf16 inputs.

    Each e4m3 code carries a relative rounding error of at most 2^-4 (3 mantissa bits), so the product of two
    codes errs by about 5 % rms per term and the projection by a few percent in norm; the pages report a
    single-layer fp8 cosine of 0.9993."""
    M, N, K = 512, 1024, 3072
    x = inputs.bf16_normal(M * K, seed=811).reshape(M, K)
    w = inputs.bf16_normal(N * K, seed=812, std=0.02).reshape(N, K)
    a, sa = ops.quant_fp8_rows(dev_bf16(x))
    b, sb = ops.quant_fp8_rows(dev_bf16(w))
    out = host_f64(ops.gemm_fp8(a, sa, b, sb))
    ref = inputs.bf16_bits_to_f64(x) @ inputs.bf16_bits_to_f64(w).T
    rel = np.linalg.norm(out - ref) / np.linalg.norm(ref)
    cos = float((out * ref).sum() / (np.linalg.norm(out) * np.linalg.norm(ref)))
    print(f"w8a8 relative error {rel:.4f}, cosine {cos:.6f}")
    assert rel < 0.06 and cos > 0.998


# ---------------------------------------------------------------- the hot path from host buffers

@pytest.mark.parametrize("B,S,H,D,chunks,prologue,pdt,odt,pinned,merge", [
    (1, 256, 2, 64, 4, True, "f32", "bf16", True, "update"),     # the tiny workload's shape
    (2, 300, 3, 128, 3, True, "f32", "f32", True, "update"),     # B = 2: value rows of a chunk are strided copies
    (2, 333, 2, 128, 2, False, "bf16", "bf16", False, "update"),  # no prologue, pageable host memory
    (1, 129, 4, 64, 1, True, "f32", "bf16", True, "update"),     # one chunk: no running result
    (1, 256, 2, 64, 4, True, "f32", "f32", True, "kernel"),      # stacked partials, one query range
    (2, 333, 2, 128, 3, False, "bf16", "bf16", True, "kernel"),   # no prologue: keys travel with their chunk
    (1, 6000, 64, 64, 3, False, "bf16", "bf16", True, "kernel"),  # two query ranges (a ragged one)
    (4, 2100, 152, 64, 3, True, "f32", "bf16", True, "kernel"),   # eight query ranges, B = 4, prologue
    (1, 8000, 64, 128, 1, False, "bf16", "f32", True, "kernel"),  # one chunk over three query ranges
    (1, 16384, 152, 64, 2, False, "bf16", "bf16", True, "kernel"),  # six tapered query ranges (3/8 ... 1/16)
    (2, 1000, 3, 128, 2, False, "f32", "bf16", False, "kernel"),  # pageable host memory
])
def test_attention_host_matches_device_path(orc, B, S, H, D, chunks, prologue, pdt, odt, pinned, merge):
    """The host-buffer path against the one-call device path on device copies of the same inputs (same chunks,
    merge form and partial dtype): bit-identical, including the query-range form whose range edges fall on the
    attention's 256-row CTA tiles.  Without the prologue, also against the oracle (sampled rows when large)."""
    dts = {"bf16": torch.bfloat16, "f32": torch.float32}
    q, k, v, wq, wk, cos, sin = inputs.small_case(B, S, H, D, seed=S + chunks)
    host = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16)  # noqa
    hq, hk, hv = host(q), host(k), host(v)
    hw = [torch.from_numpy(np.ascontiguousarray(t)) for t in (wq, wk, cos, sin)]
    if pinned:
        hq, hk, hv = hq.pin_memory(), hk.pin_memory(), hv.pin_memory()
        hw = [t.pin_memory() for t in hw]
    o, lse = ops.dit_attention_host(hq, hk, hv, *hw, eps=1e-6, chunks=chunks, partial_dtype=dts[pdt],
                                    out_dtype=dts[odt], prologue=prologue, merge=merge)
    torch.cuda.synchronize()  # (hq, hk, hv, hw stay referenced until here)
    ops.poll_device_error()
    od, ld = ops.dit_attention(dev_bf16(q), dev_bf16(k), dev_bf16(v), *(dev_f32(t) for t in (wq, wk, cos, sin)),
                               eps=1e-6, chunks=chunks, partial_dtype=dts[pdt], out_dtype=dts[odt],
                               prologue=prologue, merge=merge)
    assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())
    if not prologue:
        from parity import sample_rows
        rows = None if S <= 1000 else sample_rows(S, 12, seed=S)
        fq, fk, fv = (inputs.bf16_bits_to_f64(x) for x in (q, k, v))
        ro, rl = orc.attention(fq, fk, fv, 1 / math.sqrt(D), rows=rows)
        go, gl = o.double().numpy(), lse.double().numpy()
        if rows is not None:
            go, gl = go[:, rows], gl[:, :, rows]
        check_o(go, ro, f32=odt == "f32", what=f"host path ({merge})", vmax=vmax(v))
        check_lse(gl, rl, what=f"host path ({merge})")


@pytest.mark.parametrize("merge", ["update", "kernel"])
def test_attention_host_back_to_back_calls_share_a_workspace(merge):
    """Two calls on one stream with one workspace and different inputs: the second call's copies wait for the
    first call's kernels (the workspace is reused), so each result matches its own inputs."""
    B, S, H, D = 1, 400, 2, 128
    outs = []
    ws = torch.empty(ops.attention_host_workspace_bytes(B, S, H, D, 2, merge=merge), dtype=torch.uint8,
                     device="cuda")
    cases = [inputs.small_case(B, S, H, D, seed=s) for s in (1, 2)]
    host = lambda bits: torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).pin_memory()  # noqa
    keep = []  # the host inputs must outlive the asynchronous copies
    for q, k, v, wq, wk, cos, sin in cases:
        args = [host(q), host(k), host(v)] + [torch.from_numpy(np.ascontiguousarray(t)).pin_memory()
                                              for t in (wq, wk, cos, sin)]
        keep.append(args)
        outs.append(ops.dit_attention_host(*args, chunks=2, workspace=ws, merge=merge))
    torch.cuda.synchronize()
    for (o, lse), (q, k, v, wq, wk, cos, sin) in zip(outs, cases):
        od, ld = ops.dit_attention(dev_bf16(q), dev_bf16(k), dev_bf16(v),
                                   *(dev_f32(t) for t in (wq, wk, cos, sin)), chunks=2, merge=merge)
        assert torch.equal(o, od.cpu()) and torch.equal(lse, ld.cpu())


@pytest.mark.parametrize("merge,chunks,prologue,pdt", [
    ("update", 2, True, "f32"), ("update", 3, False, "bf16"), ("update", 5, True, "bf16"),
    ("kernel", 3, True, "f32"), ("kernel", 4, False, "bf16"), ("kernel", 1, True, "f32"),
])
def test_dit_attention_equals_its_entry_points(merge, chunks, prologue, pdt):
    """The one-call path (later chunks start beside the previous chunk's last wave and wait for it only where they
    need its results) is bit-identical to the same entry points called one by one, each waiting at its start."""
    dts = {"bf16": torch.bfloat16, "f32": torch.float32}
    B, S, H, D = 2, 1000, 4, 128
    q, k, v, wq, wk, cos, sin = inputs.small_case(B, S, H, D, seed=chunks * 7 + len(merge))
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    tw = [dev_f32(t) for t in (wq, wk, cos, sin)]
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    o, lse = ops.dit_attention(tq, tk, tv, *tw, eps=1e-6, chunks=chunks, partial_dtype=dts[pdt], prologue=prologue,
                               merge=merge, attn_events=(e0, e1))
    aq, ak = ops.qk_norm_rope(tq, tk, *tw, 1e-6) if prologue else (tq, tk)
    edges = [(i * S) // chunks for i in range(chunks + 1)]
    if chunks == 1:
        ro, rl = ops.attn_fwd(aq, ak, tv, None, 0, S)
    elif merge == "update":
        acc, rl = ops.attn_fwd(aq, ak, tv, None, edges[0], edges[1], o_dtype=dts[pdt])
        for c in range(1, chunks - 1):
            ops.attn_fwd_update(aq, ak, tv, acc, rl, None, edges[c], edges[c + 1], o=acc, lse=rl)
        ro = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
        ops.attn_fwd_update(aq, ak, tv, acc, rl, None, edges[-2], edges[-1], o=ro, lse=rl)
    else:
        parts = torch.empty((chunks, B, S, H, D), dtype=dts[pdt], device="cuda")
        lparts = torch.empty((chunks, B, H, S), dtype=torch.float32, device="cuda")
        for c in range(chunks):
            ops.attn_fwd(aq, ak, tv, None, edges[c], edges[c + 1], o=parts[c], lse=lparts[c])
        ro, rl = ops.attn_merge_lse(parts, lparts)
    torch.cuda.synchronize()
    ops.poll_device_error()
    assert torch.equal(o, ro) and torch.equal(lse, rl)
    assert e0.elapsed_time(e1) > 0.0


def test_dit_attention_back_to_back_steps_share_a_workspace():
    """Steps issued back to back on one stream with one workspace and different inputs (the next step's prologue
    rewrites the workspace the previous step's last chunk reads): each result matches its own inputs."""
    B, S, H, D = 1, 900, 3, 128
    cases = [inputs.small_case(B, S, H, D, seed=s) for s in (3, 4, 5)]
    dev = [[dev_bf16(q), dev_bf16(k), dev_bf16(v)] + [dev_f32(t) for t in (wq, wk, cos, sin)]
           for q, k, v, wq, wk, cos, sin in cases]
    for merge in ("update", "kernel"):
        ws = torch.empty(ops.attention_workspace_bytes(B, S, H, D, 3, True, torch.float32, merge),
                         dtype=torch.uint8, device="cuda")
        outs = [ops.dit_attention(*args, chunks=3, merge=merge, workspace=ws) for args in dev]
        torch.cuda.synchronize()
        for (o, lse), args in zip(outs, dev):
            ro, rl = ops.dit_attention(*args, chunks=3, merge=merge)
            torch.cuda.synchronize()
            assert torch.equal(o, ro) and torch.equal(lse, rl)


# ---------------------------------------------------------------- sizes at the edges

def test_attn_long_sequence_sampled_rows(orc):
    """131072 queries and keys (one head): 512 CTAs along the rows and 1024 key blocks per CTA, so every ring
    and S/P barrier goes through hundreds of phases; sampled rows (first, last, ragged tail, random) vs the
    oracle over all keys, plain and update forms."""
    from parity import sample_rows
    B, H, S, D = 1, 1, 131072, 128
    q, k, v, *_ = inputs.small_case(B, S, H, D, seed=2024)
    tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
    o, lse = ops.attn_fwd(tq, tk, tv)
    acc, lse_acc = ops.attn_fwd(tq, tk, tv, None, 0, 70001, o_dtype=torch.float32)
    o2, l2 = ops.attn_fwd_update(tq, tk, tv, acc, lse_acc, None, 70001, S)
    ops.poll_device_error()
    rows = sample_rows(S, 16, seed=5)
    rt = torch.from_numpy(rows).cuda()
    ro, rl = orc.attention(*(inputs.bf16_bits_to_f64(x) for x in (q, k, v)), 1 / math.sqrt(D), rows=rows)
    for got_o, got_l, what in [(o, lse, "long"), (o2, l2, "long, update form")]:
        check_o(host_f64(got_o.index_select(1, rt)), ro, what=what)
        check_lse(host_f64(got_l.index_select(2, rt)), rl, what=what)


def test_empty_inputs_launch_nothing():
    """Zero-sized work through the binding returns empty results without a launch or an error."""
    e = torch.empty((1, 0, 2, 128), dtype=torch.bfloat16, device="cuda")
    o, lse = ops.attn_fwd(e, e, e)
    assert o.shape == (1, 0, 2, 128) and lse.shape == (1, 2, 0)
    o, lse = ops.attn_merge_lse(torch.empty((2, 1, 0, 2, 128), device="cuda"),
                                torch.empty((2, 1, 2, 0), device="cuda"))
    assert o.numel() == 0 and lse.numel() == 0
    w = torch.ones(128, device="cuda")
    tab = torch.empty((0, 64), device="cuda")
    qo, ko = ops.qk_norm_rope(e, e, w, w, tab, tab)
    assert qo.numel() == 0 and ko.numel() == 0
    x = torch.empty((0, 5120), dtype=torch.bfloat16, device="cuda")
    assert ops.rms_norm(x, torch.ones(5120, device="cuda")).numel() == 0
    codes, scale = ops.quant_fp8_rows(x)
    assert codes.numel() == 0 and scale.numel() == 0
    ops.poll_device_error()
