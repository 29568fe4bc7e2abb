"""Seeded synthetic inputs for the DiT attention core.

This module is the one place both the CUDA path and the fp64 oracle get their
inputs from.  It holds none of the method's arithmetic: it draws normal
variates, rounds them to bf16 bit patterns, enumerates token positions and
tabulates the rotary angles (cos/sin of position x frequency) that both sides
receive as plain inputs -- the fused rotary operator on the Wan2.2 page
("NPU Wan2.2-I2V model inference optimisation practice", section "NPU
rotary_mul operator adaptation") likewise takes precomputed cos/sin tensors.

Workloads (shapes of the DiT models the pages discuss; all tensors synthetic):

  tiny             B1 H2  D64  S256, 1-D positions, KV in 4 chunks
  qwen_image       B1 H24 D128 S4312 = 256 text + 78x52 image tokens, one pass
  qwen_image_edit  B2 H24 D128 S8624 = 512 text + 2 x 78x52 (target+reference), one pass
  wan480           B1 H40 D128 S32760 = 21x30x52 video patches, one pass
  wan720           B1 H40 D128 S75600 = 21x45x80, K x 3, no prologue, 8 chunks

Only the tiny and the 720p workloads are stated with a KV chunking; the
others are single-pass attention (chunked runs of them take an explicit
chunk count).

Seeds: 1000*workload_index + 100*batch_index + tensor_id with tensor ids
q=0, k=1, v=2, wq=3, wk=4.  Large tensors are drawn in fixed 4 Mi-element
blocks, each from its own PCG64 stream keyed by (seed, block), so the bits do
not depend on how many threads draw them.
"""

from __future__ import annotations

import concurrent.futures as _cf
import dataclasses
import math
import os

import numpy as np

TENSOR_IDS = {"q": 0, "k": 1, "v": 2, "wq": 3, "wk": 4}
_BLOCK = 1 << 22


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic DiT attention workload."""

    index: int
    name: str
    B: int
    H: int
    D: int
    S: int
    text_tokens: int            # leading text tokens (0 for pure video)
    grids: tuple                # tuple of (frames, height, width) latent grids
    axis_dims: tuple            # rotary dims per axis (sums to D); 1 axis => 1-D positions
    chunks: int                 # KV chunks for the chunk-mode + LSE-merge pass
    prologue: bool              # QK-RMSNorm + RoPE applied before attention
    k_scale: float = 1.0        # K drawn as k_scale * N(0,1)
    eps: float = 1e-6
    rope_base: float = 10000.0
    description: str = ""

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def attention_flops(self) -> float:
        """4*B*H*Sq*Skv*D: two GEMMs (QK^T and PV) of 2 flops per MAC."""
        return 4.0 * self.B * self.H * self.S * self.S * self.D

    def chunk_bounds(self, chunks: int | None = None):
        c = self.chunks if chunks is None else chunks
        edges = [(i * self.S) // c for i in range(c + 1)]
        return [(edges[i], edges[i + 1]) for i in range(c)]


WORKLOADS = {
    w.name: w
    for w in [
        Workload(1, "tiny", 1, 2, 64, 256, 0, ((1, 1, 256),), (64,), 4, True,
                 description="tiny oracle case B1 H2 D64 S256, 1-D RoPE, 4 KV chunks"),
        Workload(2, "qwen_image", 1, 24, 128, 4312, 256, ((1, 78, 52),), (16, 56, 56), 1, True,
                 description="Qwen-Image joint attention B1 H24 D128 S4312 (256 text + 78x52 image)"),
        Workload(3, "qwen_image_edit", 2, 24, 128, 8624, 512, ((1, 78, 52), (1, 78, 52)), (16, 56, 56), 1,
                 True, description="Qwen-Image-Edit B2 (CFG pair) H24 D128 S8624 (512 text + 2x78x52)"),
        Workload(4, "wan480", 1, 40, 128, 32760, 0, ((21, 30, 52),), (44, 42, 42), 1, True,
                 description="Wan2.2 480p video attention B1 H40 D128 S32760 (21x30x52)"),
        Workload(5, "wan720", 1, 40, 128, 75600, 0, ((21, 45, 80),), (44, 42, 42), 8, False, k_scale=3.0,
                 description="Wan2.2 720p video attention B1 H40 D128 S75600 (21x45x80), K x3, 8 KV chunks"),
    ]
}


def seed_for(workload: Workload, tensor: str, batch: int = 0) -> int:
    return 1000 * workload.index + 100 * batch + TENSOR_IDS[tensor]


# ----------------------------------------------------------------------------
# bf16 bit patterns
# ----------------------------------------------------------------------------

def f32_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bf16 (round to nearest even); returns int16 bit patterns.

    Inputs are finite normal draws, so the NaN/Inf branch of a general
    converter is not needed.
    """
    u = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16).view(np.int16)


def bf16_bits_to_f32(bits: np.ndarray) -> np.ndarray:
    u = np.ascontiguousarray(bits).view(np.uint16).astype(np.uint32) << np.uint32(16)
    return u.view(np.float32)


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    return bf16_bits_to_f32(bits).astype(np.float64)


def _fill_block(out: np.ndarray, seed: int, block: int, std: float, mean: float):
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, block])))
    x = rng.standard_normal(out.shape[0], dtype=np.float32)
    if std != 1.0:
        x *= np.float32(std)
    if mean != 0.0:
        x += np.float32(mean)
    out[:] = f32_to_bf16_bits(x)


def bf16_normal(n: int, seed: int, std: float = 1.0, mean: float = 0.0, threads: int | None = None) -> np.ndarray:
    """n bf16 draws of mean + std*N(0,1) (the normal draw and the affine map in fp32)."""
    out = np.empty(n, dtype=np.int16)
    nblk = (n + _BLOCK - 1) // _BLOCK
    if nblk <= 1:
        _fill_block(out, seed, 0, std, mean)
        return out
    threads = threads or min(16, os.cpu_count() or 1)
    with _cf.ThreadPoolExecutor(threads) as ex:
        futs = [ex.submit(_fill_block, out[i * _BLOCK:(i + 1) * _BLOCK], seed, i, std, mean) for i in range(nblk)]
        for f in futs:
            f.result()
    return out


def f32_normal(n: int, seed: int, std: float = 1.0, mean: float = 1.0) -> np.ndarray:
    rng = np.random.Generator(np.random.PCG64(np.random.SeedSequence([seed, 0])))
    x = rng.standard_normal(n, dtype=np.float32)
    return (x * np.float32(std) + np.float32(mean)).astype(np.float32)


# ----------------------------------------------------------------------------
# positions and rotary tables
# ----------------------------------------------------------------------------

def positions(w: Workload) -> np.ndarray:
    """Integer token positions [S, n_axes].

    Text tokens come first and token i sits at (i, i, i); then each latent
    grid is enumerated row-major over (frame, h, w), grid g taking frame index
    g (target latent frame 0, reference latent frame 1).  One-axis workloads
    use 0..S-1.
    """
    n_axes = len(w.axis_dims)
    if n_axes == 1:
        return np.arange(w.S, dtype=np.int64)[:, None]
    parts = []
    if w.text_tokens:
        t = np.arange(w.text_tokens, dtype=np.int64)
        parts.append(np.stack([t, t, t], axis=1))
    for g, (f, hh, ww) in enumerate(w.grids):
        fi, hi, wi = np.meshgrid(np.arange(f), np.arange(hh), np.arange(ww), indexing="ij")
        fi = fi + (g if len(w.grids) > 1 else 0)
        parts.append(np.stack([fi.ravel(), hi.ravel(), wi.ravel()], axis=1).astype(np.int64))
    pos = np.concatenate(parts, axis=0)
    assert pos.shape == (w.S, 3), (pos.shape, w.S)
    return pos


def rope_tables(pos: np.ndarray, axis_dims, base: float = 10000.0, offset=None):
    """cos/sin tables [S, D/2] (float32) for interleaved rotary pairs.

    Axis a owns a contiguous run of axis_dims[a]/2 pairs; its local pair j at
    integer position p has angle p * base**(-2j/axis_dims[a]).  The angle is
    evaluated in fp64 and its cos/sin rounded once to fp32; both the kernel and
    the oracle receive those fp32 values.  `offset` shifts every position on
    each axis (used by the relative-position checks).
    """
    pos = np.asarray(pos, dtype=np.float64)
    if offset is not None:
        pos = pos + np.asarray(offset, dtype=np.float64)[None, :]
    angles = []
    for a, d_a in enumerate(axis_dims):
        j = np.arange(d_a // 2, dtype=np.float64)
        inv = base ** (-2.0 * j / d_a)
        angles.append(pos[:, a:a + 1] * inv[None, :])
    ang = np.concatenate(angles, axis=1)
    return np.cos(ang).astype(np.float32), np.sin(ang).astype(np.float32)


# ----------------------------------------------------------------------------
# whole workloads
# ----------------------------------------------------------------------------

@dataclasses.dataclass
class Inputs:
    """Host-side inputs of one workload: bf16 tensors as int16 bit patterns, BSHD."""

    w: Workload
    q: np.ndarray
    k: np.ndarray
    v: np.ndarray
    wq: np.ndarray
    wk: np.ndarray
    cos: np.ndarray
    sin: np.ndarray


def _bshd(w: Workload, tensor: str, std: float = 1.0) -> np.ndarray:
    per = w.S * w.H * w.D
    out = np.empty(w.B * per, dtype=np.int16)
    for b in range(w.B):
        out[b * per:(b + 1) * per] = bf16_normal(per, seed_for(w, tensor, b), std=std)
    return out.reshape(w.B, w.S, w.H, w.D)


def make_inputs(name: str) -> Inputs:
    w = WORKLOADS[name]
    q = _bshd(w, "q")
    k = _bshd(w, "k", std=w.k_scale)
    v = _bshd(w, "v")
    wq = f32_normal(w.D, seed_for(w, "wq"), std=0.1, mean=1.0)
    wk = f32_normal(w.D, seed_for(w, "wk"), std=0.1, mean=1.0)
    cos, sin = rope_tables(positions(w), w.axis_dims, w.rope_base)
    return Inputs(w, q, k, v, wq, wk, cos, sin)


def small_case(B: int, S: int, H: int, D: int, seed: int, Skv: int | None = None, k_std: float = 1.0):
    """Small seeded q/k/v (bf16 bits, BSHD) plus weights and 1-D rotary tables for tests."""
    Skv = S if Skv is None else Skv
    q = bf16_normal(B * S * H * D, seed).reshape(B, S, H, D)
    k = bf16_normal(B * Skv * H * D, seed + 1, std=k_std).reshape(B, Skv, H, D)
    v = bf16_normal(B * Skv * H * D, seed + 2).reshape(B, Skv, H, D)
    wq = f32_normal(D, seed + 3, std=0.1, mean=1.0)
    wk = f32_normal(D, seed + 4, std=0.1, mean=1.0)
    cos, sin = rope_tables(np.arange(max(S, Skv))[:, None], (D,))
    return q, k, v, wq, wk, cos, sin
