"""Shared helpers for the GPU parity tests: host<->device moves and the tolerances.

Tolerances (written here once, used by every parity test):
  bf16 O vs fp64 oracle      max abs <= 2e-2 and cosine >= 0.9999
  LSE vs fp64 oracle         abs <= 1e-3
  fp32 O vs fp64 oracle      max abs <= 2^-8 * max_j |v_j| and cosine >= 0.99999.
                             The kernel rounds the softmax weights P to bf16
                             before the PV product (relative error <= 2^-9 per
                             weight, normaliser l kept in fp32), so
                             |dO| <= 2^-9 * sum_j p_j |v_j| / l <= 2^-9 * max|v|;
                             the bound doubles that for fp32 accumulation.  With
                             few keys the weights are O(1) and this bound is
                             reached; with many keys the error averages down.
  prologue (bf16 out)        within one bf16 ulp of the fp64 value: fp32
                             arithmetic (~1e-6 relative) plus one rounding.
  merge vs oracle merge of the same partials
                             fp32 out: 1e-5 relative to the row scale;
                             bf16 out: one bf16 ulp.
"""

from __future__ import annotations

import math

import numpy as np
import torch

from diffusion_transformer_attention_dit_gb300 import inputs

O_BF16_MAX_ABS = 2e-2
O_COS_MIN = 0.9999
LSE_MAX_ABS = 1e-3
O_F32_REL_VMAX = 2.0 ** -8
O_F32_COS_MIN = 0.99999


def dev_bf16(bits: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).cuda().view(torch.bfloat16)


def dev_f32(x: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).cuda()


def host_f64(t: torch.Tensor) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(np.float64)


def bf16_ulp(x: np.ndarray) -> np.ndarray:
    """Spacing of bf16 numbers at |x| (8 significant bits)."""
    ax = np.maximum(np.abs(x), 2.0 ** -126)
    return 2.0 ** (np.floor(np.log2(ax)) - 7)


def cosine(a: np.ndarray, b: np.ndarray) -> float:
    a = a.ravel()
    b = b.ravel()
    return float(np.dot(a, b) / (np.linalg.norm(a) * np.linalg.norm(b)))


def check_o(got: np.ndarray, ref: np.ndarray, f32: bool = False, what: str = "", vmax: float | None = None):
    """bf16 O: max abs <= 2e-2, cosine >= 0.9999.  fp32 O: max abs <= 2^-8 * vmax, cosine >= 0.99999."""
    err = np.abs(got - ref).max()
    cos = cosine(got, ref)
    if f32:
        assert vmax is not None, "fp32 parity needs max |v| over the keys"
        bound, cmin = O_F32_REL_VMAX * vmax, O_F32_COS_MIN
    else:
        bound, cmin = O_BF16_MAX_ABS, O_COS_MIN
    assert err <= bound, f"{what}: O max abs err {err:.3e} > {bound:.3e}"
    assert cos >= cmin, f"{what}: O cosine {cos:.7f} < {cmin}"
    return err, cos


def check_lse(got: np.ndarray, ref: np.ndarray, what: str = ""):
    err = np.abs(got - ref).max()
    assert err <= LSE_MAX_ABS, f"{what}: LSE max abs err {err:.3e} > {LSE_MAX_ABS}"
    return err


def check_bf16_rounding(got: np.ndarray, ref: np.ndarray, what: str = "", atol: float = 1e-6):
    """|got - ref| <= one bf16 ulp of ref, plus `atol` for values cancelled down to near zero in fp32."""
    err = np.abs(got - ref)
    bad = err > bf16_ulp(ref) + atol
    assert not bad.any(), f"{what}: {bad.sum()} values off by more than one bf16 ulp (max err {err.max():.3e})"


def sample_rows(S: int, n: int = 64, seed: int = 0) -> np.ndarray:
    """First row, last row, rows of the last (ragged) 128-row tile, then seeded random rows."""
    tail0 = (S // 128) * 128 if S % 128 else S - 128
    fixed = {0, S - 1, max(tail0, 0), max(S - 2, 0)}
    rng = np.random.default_rng(seed)
    rest = rng.choice(S, size=min(S, n) , replace=False)
    rows = list(fixed) + [int(r) for r in rest if r not in fixed]
    return np.array(sorted(rows[:n]), dtype=np.int64)


def tensors(bits: dict) -> dict:
    return {k: dev_bf16(v) for k, v in bits.items()}


def workload_inputs(name: str):
    return inputs.make_inputs(name)


def scale_of(D: int) -> float:
    return 1.0 / math.sqrt(D)
