"""Checks that pin the fp64 oracle to something other than itself.

Each `pin_*` function takes an `oracle.Oracle` and raises AssertionError when
the oracle disagrees with a closed form, an invariant, a hand-derived golden
fixture, or an independent library routine (torch's fp64 rms_norm and
scaled_dot_product_attention, numpy complex multiplication).  The same
functions run against deliberately broken copies of the oracle in
test_oracle_mutants.py, which shows that a plausible slip in any oracle
function fails at least one pin.
"""

from __future__ import annotations

import json
import math
from pathlib import Path

import numpy as np
import torch

from diffusion_transformer_attention_dit_gb300 import inputs

GOLDEN = Path(__file__).resolve().parent / "golden"


def _golden(name):
    return json.loads((GOLDEN / name).read_text())


def _close(a, b, rtol=1e-11, atol=1e-12, what=""):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    assert a.shape == b.shape, (what, a.shape, b.shape)
    err = np.abs(a - b)
    bound = atol + rtol * np.abs(b)
    assert np.all(err <= bound), f"{what}: max err {err.max():.3e}"


def _rng(seed):
    return np.random.default_rng(seed)


# ---------------------------------------------------------------- RMSNorm

def pin_rms_constant(orc):
    """x == c everywhere gives y = c * w / sqrt(c^2 + eps)."""
    rng = _rng(1)
    w = rng.normal(1.0, 0.1, 16)
    for c, eps in [(0.5, 1e-6), (-2.0, 0.5), (3.0, 4.0)]:
        x = np.full((3, 16), c)
        y = orc.rms_norm(x, w, eps)
        _close(y, np.broadcast_to(c * w / math.sqrt(c * c + eps), y.shape), what="rms const")


def pin_rms_torch(orc):
    """Agrees with torch.nn.functional.rms_norm in float64."""
    rng = _rng(2)
    for D, eps in [(64, 1e-6), (128, 1e-5), (7, 0.3)]:
        x = rng.normal(0, 2, (5, D))
        w = rng.normal(1, 0.1, D)
        ref = torch.nn.functional.rms_norm(torch.from_numpy(x), (D,), weight=torch.from_numpy(w), eps=eps).numpy()
        _close(orc.rms_norm(x, w, eps), ref, rtol=1e-12, what="rms vs torch")


def pin_rms_golden(orc):
    g = _golden("rms_norm_3_4.json")
    for case in g["cases"]:
        y = orc.rms_norm(np.array([case["x"]]), np.array(case["w"]), case["eps"])
        _close(y[0], case["y"], rtol=1e-14, what="rms golden")


def pin_rms_unit_rms(orc):
    """With eps = 0 and unit weights the output has mean square exactly 1 and is scale invariant."""
    rng = _rng(3)
    x = rng.normal(0, 1, (4, 32))
    y = orc.rms_norm(x, np.ones(32), 0.0)
    _close((y * y).mean(axis=1), np.ones(4), what="unit rms")
    _close(orc.rms_norm(7.5 * x, np.ones(32), 0.0), y, what="scale invariance")


# ---------------------------------------------------------------- LayerNorm + modulation

def pin_ln_modulate_torch(orc):
    """Agrees with torch fp64 layer_norm using weight 1 + scale and bias shift, per sample."""
    rng = _rng(23)
    B, L, C = 3, 5, 24
    x = rng.normal(0.5, 2, (B, L, C))
    scale = rng.normal(0, 0.3, (B, C))
    shift = rng.normal(0, 0.3, (B, C))
    y = orc.layer_norm_modulate(x, scale, shift, 1e-6)
    for b in range(B):
        ref = torch.nn.functional.layer_norm(torch.from_numpy(x[b]), (C,), weight=torch.from_numpy(1 + scale[b]),
                                             bias=torch.from_numpy(shift[b]), eps=1e-6).numpy()
        _close(y[b], ref, rtol=1e-11, atol=1e-12, what="ln modulate vs torch")
    plain = orc.layer_norm_modulate(x, None, None, 1e-6)
    ref = torch.nn.functional.layer_norm(torch.from_numpy(x), (C,), eps=1e-6).numpy()
    _close(plain, ref, rtol=1e-11, atol=1e-12, what="plain ln vs torch")


def pin_ln_modulate_closed_forms(orc):
    """A constant row normalises to 0 (y = shift); x = (1, 3) has mean 2, variance 1."""
    y = orc.layer_norm_modulate(np.full((1, 2, 4), 7.0), np.full((1, 4), 0.5), np.array([[1.0, -2.0, 0.0, 3.0]]), 1e-6)
    _close(y, np.broadcast_to([1.0, -2.0, 0.0, 3.0], y.shape), what="constant row")
    y = orc.layer_norm_modulate(np.array([[[1.0, 3.0]]]), np.array([[1.0, 0.0]]), np.array([[0.0, 10.0]]), 0.0)
    _close(y.ravel(), [-2.0, 11.0], what="two-element row")


# ---------------------------------------------------------------- RoPE

def _angles_tables(theta):
    return np.cos(theta), np.sin(theta)


def pin_rope_identity_at_zero(orc):
    rng = _rng(4)
    x = rng.normal(0, 1, (2, 3, 4, 16))
    c, s = np.ones((3, 8)), np.zeros((3, 8))
    _close(orc.rope_interleaved(x, c, s), x, what="rope identity")


def pin_rope_complex(orc):
    """Pair (x_2i, x_2i+1) read as x_2i + i x_2i+1 is multiplied by exp(i theta)."""
    rng = _rng(5)
    B, S, H, D = 2, 5, 3, 12
    x = rng.normal(0, 1, (B, S, H, D))
    theta = rng.uniform(-4, 4, (S, D // 2))
    c, s = _angles_tables(theta)
    z = (x[..., 0::2] + 1j * x[..., 1::2]) * np.exp(1j * theta)[None, :, None, :]
    ref = np.empty_like(x)
    ref[..., 0::2] = z.real
    ref[..., 1::2] = z.imag
    _close(orc.rope_interleaved(x, c, s), ref, what="rope complex")


def pin_rope_golden(orc):
    g = _golden("rope_quarter_turn.json")
    x = np.array(g["x"]).reshape(1, 1, 1, 4)
    y = orc.rope_interleaved(x, np.array([g["cos"]]), np.array([g["sin"]]))
    _close(y.ravel(), g["y"], what="rope golden")


def pin_rope_norm_and_inverse(orc):
    """Each pair keeps its length; rotating by -theta undoes the rotation."""
    rng = _rng(6)
    x = rng.normal(0, 1, (1, 6, 2, 8))
    theta = rng.uniform(-3, 3, (6, 4))
    c, s = _angles_tables(theta)
    y = orc.rope_interleaved(x, c, s)
    n_x = x[..., 0::2] ** 2 + x[..., 1::2] ** 2
    n_y = y[..., 0::2] ** 2 + y[..., 1::2] ** 2
    _close(n_y, n_x, what="pair norm")
    _close(orc.rope_interleaved(y, c, -s), x, what="inverse rotation")


def pin_rope_relative(orc):
    """<R(p) q, R(p') k> depends only on p - p': shifting every position on every axis leaves scores unchanged."""
    rng = _rng(7)
    D, S = 16, 9
    q = rng.normal(0, 1, (1, S, 1, D))
    k = rng.normal(0, 1, (1, S, 1, D))
    pos = rng.integers(0, 50, (S, 3))
    dims = (4, 6, 6)
    c0, s0 = inputs.rope_tables(pos, dims)
    c1, s1 = inputs.rope_tables(pos, dims, offset=(11, -3, 5))
    sc0 = np.einsum("sd,td->st", orc.rope_interleaved(q, c0, s0)[0, :, 0], orc.rope_interleaved(k, c0, s0)[0, :, 0])
    sc1 = np.einsum("sd,td->st", orc.rope_interleaved(q, c1, s1)[0, :, 0], orc.rope_interleaved(k, c1, s1)[0, :, 0])
    # tables are fp32-rounded, so agreement is to fp32 precision
    _close(sc1, sc0, rtol=1e-5, atol=1e-5, what="relative position")


def pin_prologue_chain(orc):
    """qk_norm_rope = rotation of torch's fp64 rms_norm output (complex form)."""
    rng = _rng(8)
    B, S, H, D = 2, 7, 3, 16
    x = rng.normal(0, 1, (B, S, H, D))
    w = rng.normal(1, 0.1, D)
    theta = rng.uniform(-2, 2, (S, D // 2))
    c, s = _angles_tables(theta)
    n = torch.nn.functional.rms_norm(torch.from_numpy(x), (D,), weight=torch.from_numpy(w), eps=1e-6).numpy()
    z = (n[..., 0::2] + 1j * n[..., 1::2]) * np.exp(1j * theta)[None, :, None, :]
    ref = np.empty_like(x)
    ref[..., 0::2] = z.real
    ref[..., 1::2] = z.imag
    _close(orc.qk_norm_rope(x, w, c, s, 1e-6), ref, rtol=1e-11, atol=1e-12, what="prologue chain")


def pin_round_bf16(orc):
    """The op-boundary rounding matches torch's float32 -> bfloat16 conversion and exact tie cases."""
    import oracle

    rng = _rng(20)
    x = rng.normal(0, 3, 10000).astype(np.float32)
    ref = torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    _close(oracle.round_bf16(x.astype(np.float64)), ref, rtol=0, atol=0, what="round_bf16 vs torch")
    ties = np.array([1 + 2.0 ** -8, 1 + 3 * 2.0 ** -8, -(2 + 2.0 ** -7), 1 + 2.0 ** -9])
    _close(oracle.round_bf16(ties), [1.0, 1 + 2.0 ** -6, -2.0, 1.0], rtol=0, atol=0, what="round_bf16 ties")


# ---------------------------------------------------------------- attention

def _sdpa(q, k, v, scale):
    """torch fp64 scaled_dot_product_attention on BSHD arrays; returns (o BSHD, lse [B,H,Sq])."""
    tq, tk, tv = (torch.from_numpy(np.ascontiguousarray(a)).permute(0, 2, 1, 3) for a in (q, k, v))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=scale)
    lse = torch.logsumexp(scale * (tq @ tk.transpose(-1, -2)), dim=-1)
    return o.permute(0, 2, 1, 3).numpy(), lse.numpy()


def pin_attn_sdpa(orc):
    rng = _rng(9)
    B, H, Sq, Skv, D = 2, 3, 5, 11, 8
    q = rng.normal(0, 1, (B, Sq, H, D))
    k = rng.normal(0, 1, (B, Skv, H, D))
    v = rng.normal(0, 1, (B, Skv, H, D))
    for scale, lo, hi in [(0.37, 0, Skv), (1.3, 2, 9)]:
        o, lse = orc.attention(q, k, v, scale, lo, hi)
        ro, rl = _sdpa(q, k[:, lo:hi], v[:, lo:hi], scale)
        _close(o, ro, rtol=1e-10, atol=1e-12, what="attn vs sdpa")
        _close(lse, rl, rtol=1e-12, what="lse vs logsumexp")


def pin_attn_zero_q(orc):
    """q = 0: every key gets weight 1/n, so o = mean_j v_j and lse = ln n."""
    rng = _rng(10)
    k = rng.normal(0, 1, (1, 9, 2, 8))
    v = rng.normal(0, 1, (1, 9, 2, 8))
    q = np.zeros((1, 4, 2, 8))
    o, lse = orc.attention(q, k, v, 0.5, 1, 7)
    _close(o, np.broadcast_to(v[:, 1:7].mean(axis=1, keepdims=True), o.shape), what="zero q")
    _close(lse, np.full(lse.shape, math.log(6)), what="zero q lse")


def pin_attn_const_v(orc):
    rng = _rng(11)
    q = rng.normal(0, 2, (1, 6, 2, 8))
    k = rng.normal(0, 2, (1, 10, 2, 8))
    u = rng.normal(0, 1, (1, 1, 2, 8))
    v = np.broadcast_to(u, (1, 10, 2, 8)).copy()
    o, _ = orc.attention(q, k, v, 0.4)
    _close(o, np.broadcast_to(u, o.shape), what="constant v")


def pin_attn_single_key(orc):
    """One key j: o = v_j and lse = scale * q.k_j."""
    rng = _rng(12)
    q = rng.normal(0, 1, (2, 3, 2, 8))
    k = rng.normal(0, 1, (2, 5, 2, 8))
    v = rng.normal(0, 1, (2, 5, 2, 8))
    o, lse = orc.attention(q, k, v, 0.7, 3, 4)
    _close(o, np.broadcast_to(v[:, 3:4], o.shape), what="single key o")
    ref = 0.7 * np.einsum("bqhd,bhd->bhq", q, k[:, 3])
    _close(lse, ref, what="single key lse")


def pin_attn_golden(orc):
    g = _golden("attention_two_keys.json")
    q = np.array(g["q"]).reshape(1, 1, 1, 1)
    k = np.array(g["k"]).reshape(1, 2, 1, 1)
    v = np.array(g["v"]).reshape(1, 2, 1, 1)
    o, lse = orc.attention(q, k, v, 1.0)
    _close(o.ravel(), [g["o"]], rtol=1e-14, what="attn golden o")
    _close(lse.ravel(), [g["lse"]], rtol=1e-14, what="attn golden lse")


def pin_attn_permutation(orc):
    rng = _rng(13)
    q = rng.normal(0, 1, (1, 5, 2, 8))
    k = rng.normal(0, 1, (1, 12, 2, 8))
    v = rng.normal(0, 1, (1, 12, 2, 8))
    perm = rng.permutation(12)
    o0, l0 = orc.attention(q, k, v, 0.35)
    o1, l1 = orc.attention(q, k[:, perm], v[:, perm], 0.35)
    _close(o1, o0, what="kv permutation o")
    _close(l1, l0, what="kv permutation lse")


def pin_attn_probs(orc):
    """Softmax rows are non-negative, sum to 1, and o = P v."""
    rng = _rng(14)
    q = rng.normal(0, 1, (2, 4, 3, 8))
    k = rng.normal(0, 1, (2, 9, 3, 8))
    v = rng.normal(0, 1, (2, 9, 3, 8))
    p = orc.attention_probs(q, k, 0.6, 1, 8)
    assert np.all(p >= 0)
    _close(p.sum(axis=-1), np.ones(p.shape[:-1]), what="rows sum to one")
    o, _ = orc.attention(q, k, v, 0.6, 1, 8)
    ref = np.einsum("bhij,bjhd->bihd", p, v[:, 1:8])
    _close(o, ref, what="o = P v")


def pin_attn_rows(orc):
    """A row subset reproduces the same rows of the full result."""
    rng = _rng(15)
    q = rng.normal(0, 1, (2, 10, 2, 8))
    k = rng.normal(0, 1, (2, 6, 2, 8))
    v = rng.normal(0, 1, (2, 6, 2, 8))
    rows = np.array([9, 0, 4])
    o, lse = orc.attention(q, k, v, 0.5)
    os_, ls = orc.attention(q, k, v, 0.5, rows=rows)
    _close(os_, o[:, rows], what="rows o")
    _close(ls, lse[:, :, rows], what="rows lse")


def pin_attn_causal_sdpa(orc):
    """causal: torch fp64 scaled_dot_product_attention(is_causal=True), square and rectangular."""
    rng = _rng(21)
    for B, H, Sq, Skv in [(2, 3, 9, 9), (1, 2, 6, 11), (1, 1, 12, 5)]:
        q = rng.normal(0, 1, (B, Sq, H, 8))
        k = rng.normal(0, 1, (B, Skv, H, 8))
        v = rng.normal(0, 1, (B, Skv, H, 8))
        o, lse = orc.attention(q, k, v, 0.45, causal=True)
        tq, tk, tv = (torch.from_numpy(a).permute(0, 2, 1, 3) for a in (q, k, v))
        ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, scale=0.45, is_causal=True)
        mask = torch.ones(Sq, Skv, dtype=torch.bool).tril()
        sc = (0.45 * (tq @ tk.transpose(-1, -2))).masked_fill(~mask, float("-inf"))
        _close(o, ref.permute(0, 2, 1, 3).numpy(), rtol=1e-10, atol=1e-12, what="causal vs sdpa")
        _close(lse, torch.logsumexp(sc, dim=-1).numpy(), rtol=1e-12, what="causal lse")


def pin_attn_causal_first_row_and_chunks(orc):
    """Row 0 sees only key 0; a chunk starting after a row gives it o = 0, lse = -inf; chunks merge to causal."""
    rng = _rng(22)
    q = rng.normal(0, 1, (1, 10, 2, 8))
    k = rng.normal(0, 1, (1, 10, 2, 8))
    v = rng.normal(0, 1, (1, 10, 2, 8))
    o, lse = orc.attention(q, k, v, 0.3, causal=True)
    _close(o[:, 0], v[:, 0], what="causal row 0")
    _close(lse[:, :, 0], 0.3 * np.einsum("bhd,bhd->bh", q[:, 0], k[:, 0]), what="causal row 0 lse")
    oc, lc = orc.attention(q, k, v, 0.3, 4, 10, causal=True)
    assert np.all(oc[:, :4] == 0) and np.all(lc[:, :, :4] == -np.inf)
    parts = [orc.attention(q, k, v, 0.3, lo, hi, causal=True) for lo, hi in [(0, 4), (4, 7), (7, 10)]]
    om, lm = orc.merge_lse(np.stack([p[0] for p in parts]), np.stack([p[1] for p in parts]))
    _close(om, o, rtol=1e-10, atol=1e-12, what="causal chunks merged")
    _close(lm, lse, rtol=1e-12, what="causal chunks merged lse")


# ---------------------------------------------------------------- fp8 e4m3 (W8A8)

def pin_e4m3_codec(orc):
    """Spec values, decode/encode round trip of every finite code, and torch's float8_e4m3fn cast."""
    assert orc.e4m3_decode(0x38) == 1.0 and orc.e4m3_decode(0x7E) == 448.0 and orc.e4m3_decode(0xFE) == -448.0
    assert orc.e4m3_decode(0x01) == 2.0 ** -9 and orc.e4m3_decode(0x08) == 2.0 ** -6
    assert math.isnan(orc.e4m3_decode(0x7F))
    for c in range(256):
        if c & 0x7F != 0x7F and c != 0x80:
            assert orc.e4m3_encode(orc.e4m3_decode(c)) == c, hex(c)
    assert orc.e4m3_encode(1000.0) == 0x7E and orc.e4m3_encode(-1000.0) == 0xFE  # saturating
    rng = _rng(24)
    # every midpoint between neighbouring finite codes is a tie: it must go to the even code
    vals = np.array([orc.e4m3_decode(c) for c in range(0x7F)])
    mids = (vals[:-1] + vals[1:]) / 2
    xs = np.concatenate([rng.normal(0, 50, 4000), rng.normal(0, 0.01, 1000), mids, -mids]).astype(np.float32)
    ref = torch.from_numpy(xs).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ours = np.array([orc.e4m3_encode(float(x)) for x in xs], dtype=np.uint8)
    assert np.array_equal(ours, ref)


def pin_quant_rows(orc):
    """Per-row scale = absmax / 448; the row's largest magnitude maps to +-448; codes decode near x / scale."""
    rng = _rng(25)
    x = rng.normal(0, 3, (6, 40))
    x[3] = 0.0
    codes, scale = orc.quant_fp8_rows(x)
    absmax = np.abs(x.astype(np.float32)).max(axis=1)
    assert scale[3] == 1.0 and np.all(codes[3] == 0)
    for m in (0, 1, 2, 4, 5):
        assert scale[m] == np.float32(absmax[m]) / np.float32(448.0)
        dec = np.array([orc.e4m3_decode(c) for c in codes[m]])
        assert np.abs(dec).max() == 448.0
        q = (x[m].astype(np.float32) / scale[m]).astype(np.float64)
        assert np.all(np.abs(dec - q) <= np.maximum(np.abs(q) * 2.0 ** -4, 2.0 ** -10))


def pin_gemm_fp8(orc):
    """The scaled fp8 GEMM equals numpy's matmul of the decoded codes times both scales."""
    rng = _rng(26)
    a = rng.integers(0, 256, (5, 48)).astype(np.uint8)
    b = rng.integers(0, 256, (7, 48)).astype(np.uint8)
    a[a & 0x7F == 0x7F] = 0
    b[b & 0x7F == 0x7F] = 0
    sa = rng.uniform(0.1, 2, 5).astype(np.float32)
    sb = rng.uniform(0.1, 2, 7).astype(np.float32)
    lut = np.array([orc.e4m3_decode(c) for c in range(256)])
    lut[np.isnan(lut)] = 0
    ref = (lut[a] @ lut[b].T) * sa.astype(np.float64)[:, None] * sb.astype(np.float64)[None, :]
    _close(orc.gemm_fp8(a, sa, b, sb), ref, rtol=1e-12, atol=1e-12, what="fp8 gemm")


# ---------------------------------------------------------------- merge

def _parts(orc, q, k, v, scale, bounds):
    os_, ls = [], []
    for lo, hi in bounds:
        o, l = orc.attention(q, k, v, scale, lo, hi)
        os_.append(o)
        ls.append(l)
    return np.stack(os_), np.stack(ls)


def pin_merge_golden(orc):
    g = _golden("merge_two_blocks.json")
    o_parts = np.array(g["o_parts"]).reshape(2, 1, 1, 1, 2)
    l_parts = np.array(g["lse_parts"]).reshape(2, 1, 1, 1)
    o, lse = orc.merge_lse(o_parts, l_parts)
    _close(o.ravel(), g["o"], rtol=1e-14, atol=1e-14, what="merge golden o")
    _close(lse.ravel(), [g["lse"]], rtol=1e-14, what="merge golden lse")


def pin_merge_identity_and_duplicate(orc):
    rng = _rng(16)
    o1 = rng.normal(0, 1, (1, 2, 4, 3, 8))
    l1 = rng.normal(0, 3, (1, 2, 3, 4))
    o, lse = orc.merge_lse(o1, l1)
    _close(o, o1[0], what="C=1 identity o")
    _close(lse, l1[0], what="C=1 identity lse")
    o, lse = orc.merge_lse(np.concatenate([o1, o1]), np.concatenate([l1, l1]))
    _close(o, o1[0], what="duplicate o")
    _close(lse, l1[0] + math.log(2), what="duplicate lse")


def pin_merge_equals_full(orc):
    """Attention over disjoint key blocks, merged, equals attention over all keys."""
    rng = _rng(17)
    q = rng.normal(0, 1, (2, 7, 3, 8))
    k = rng.normal(0, 2, (2, 23, 3, 8))
    v = rng.normal(0, 1, (2, 23, 3, 8))
    o, lse = orc.attention(q, k, v, 0.5)
    for bounds in [[(0, 23)], [(0, 5), (5, 23)], [(0, 1), (1, 9), (9, 10), (10, 23)]]:
        op, lp = _parts(orc, q, k, v, 0.5, bounds)
        om, lm = orc.merge_lse(op, lp)
        _close(om, o, rtol=1e-10, atol=1e-12, what="merged == full o")
        _close(lm, lse, rtol=1e-12, what="merged == full lse")
        if len(bounds) > 1:
            # the signature of a ring loop that never merges: output equal to one block's own attention
            for c in range(len(bounds)):
                assert np.abs(om - op[c]).max() > 1e-3, "merged output equals a single block's output"


def pin_merge_associative(orc):
    rng = _rng(18)
    op = rng.normal(0, 1, (3, 1, 5, 2, 4))
    lp = rng.normal(0, 2, (3, 1, 2, 5))
    o3, l3 = orc.merge_lse(op, lp)
    o2, l2 = orc.merge_lse(op[:2], lp[:2])
    oa, la = orc.merge_lse(np.stack([o2, op[2]]), np.stack([l2, lp[2]]))
    _close(oa, o3, what="associative o")
    _close(la, l3, what="associative lse")


def pin_merge_neg_inf(orc):
    """A block with lse = -inf carries no weight; all -inf gives o = 0, lse = -inf."""
    rng = _rng(19)
    op = rng.normal(0, 1, (2, 1, 3, 1, 4))
    lp = np.array([[[[0.3, -np.inf, -np.inf]]], [[[-np.inf, 1.1, -np.inf]]]])
    o, lse = orc.merge_lse(op, lp)
    _close(o[0, 0, 0], op[0, 0, 0, 0], what="-inf weight 0 (a)")
    _close(o[0, 1, 0], op[1, 0, 1, 0], what="-inf weight 0 (b)")
    _close(lse[0, 0, :2], [0.3, 1.1], what="-inf lse")
    assert np.all(o[0, 2] == 0) and lse[0, 0, 2] == -np.inf


ALL_PINS = [v for k, v in sorted(globals().items()) if k.startswith("pin_")]
