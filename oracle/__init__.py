"""fp64 CPU oracle for the DiT attention core -- TEST INFRASTRUCTURE ONLY.

Only `tests/`, `__graft_entry__.smoke()` and `bench.py`'s CPU-baseline leg
load this package.  The product path (the C-ABI library and its Python
binding) never imports it and shares no code with it.

`Oracle` wraps the plain-C library built from `oracle.c` (gcc, OpenMP, fp64,
no fast-math, no FMA contraction).  All arrays are numpy float64; bf16 inputs
arrive as their exact fp64 values.
"""

from __future__ import annotations

import ctypes
import subprocess
from pathlib import Path

import numpy as np

HERE = Path(__file__).resolve().parent
SOURCE = HERE / "oracle.c"
LIBRARY = HERE / "liboracle.so"

_D = ctypes.POINTER(ctypes.c_double)
_I64 = ctypes.c_int64


def build(source: Path = SOURCE, output: Path = LIBRARY, extra_flags=()) -> Path:
    """Compile the oracle with gcc into a shared library (idempotent on mtime)."""
    source, output = Path(source), Path(output)
    if output.exists() and output.stat().st_mtime >= source.stat().st_mtime and not extra_flags:
        return output
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
           *extra_flags, str(source), "-o", str(output), "-lm"]
    subprocess.run(cmd, check=True)
    return output


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_D)


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


class Oracle:
    """ctypes view of one compiled oracle library."""

    def __init__(self, path: Path | str = LIBRARY):
        self.path = Path(path)
        lib = ctypes.CDLL(str(self.path))
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_rms_norm.argtypes = [_D, _D, _I64, _I64, ctypes.c_double, _D]
        lib.oracle_layer_norm_modulate.argtypes = [_D, _D, _D, _I64, _I64, _I64, ctypes.c_double, _D]
        lib.oracle_layer_norm_modulate.restype = None
        _U8 = ctypes.POINTER(ctypes.c_ubyte)
        _F = ctypes.POINTER(ctypes.c_float)
        lib.oracle_e4m3_decode.argtypes = [ctypes.c_int]
        lib.oracle_e4m3_decode.restype = ctypes.c_double
        lib.oracle_e4m3_encode.argtypes = [ctypes.c_double]
        lib.oracle_e4m3_encode.restype = ctypes.c_int
        lib.oracle_quant_fp8_rows.argtypes = [_D, _I64, _I64, _U8, _F]
        lib.oracle_quant_fp8_rows.restype = None
        lib.oracle_gemm_fp8.argtypes = [_U8, _F, _U8, _F, _I64, _I64, _I64, _D]
        lib.oracle_gemm_fp8.restype = None
        lib.oracle_rope_interleaved.argtypes = [_D, _D, _D, _I64, _I64, _I64, _I64, _D]
        lib.oracle_qk_norm_rope.argtypes = [_D, _D, _D, _D, _I64, _I64, _I64, _I64, ctypes.c_double, _D]
        lib.oracle_attention.argtypes = [_D, _D, _D, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
                                         _I64, _I64, ctypes.POINTER(ctypes.c_int64), _I64, _D, _D]
        lib.oracle_attention_masked.argtypes = [_D, _D, _D, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
                                                _I64, _I64, ctypes.c_int, ctypes.POINTER(ctypes.c_int64), _I64, _D,
                                                _D]
        lib.oracle_attention_probs.argtypes = [_D, _D, _I64, _I64, _I64, _I64, _I64, ctypes.c_double,
                                               _I64, _I64, _D]
        lib.oracle_merge_lse.argtypes = [_D, _D, _I64, _I64, _I64, _I64, _I64, _D, _D]
        for name in ("oracle_rms_norm", "oracle_rope_interleaved", "oracle_qk_norm_rope",
                     "oracle_attention", "oracle_attention_masked", "oracle_attention_probs", "oracle_merge_lse"):
            getattr(lib, name).restype = None
        self.lib = lib

    def num_threads(self) -> int:
        return int(self.lib.oracle_num_threads())

    def rms_norm(self, x, w, eps: float) -> np.ndarray:
        x = _f64(x)
        w = _f64(w)
        D = x.shape[-1]
        y = np.empty_like(x)
        self.lib.oracle_rms_norm(_ptr(x), _ptr(w), x.size // D, D, eps, _ptr(y))
        return y

    def layer_norm_modulate(self, x, scale, shift, eps: float) -> np.ndarray:
        """x [B, L, C]; scale, shift [B, C] or None -> LN(x) * (1 + scale) + shift."""
        x = _f64(x)
        B, L, C = x.shape
        sc = None if scale is None else _f64(scale)
        sh = None if shift is None else _f64(shift)
        y = np.empty_like(x)
        self.lib.oracle_layer_norm_modulate(_ptr(x), None if sc is None else _ptr(sc), None if sh is None else _ptr(sh),
                                            B, L, C, eps, _ptr(y))
        return y

    def e4m3_decode(self, code: int) -> float:
        return float(self.lib.oracle_e4m3_decode(int(code)))

    def e4m3_encode(self, x: float) -> int:
        return int(self.lib.oracle_e4m3_encode(float(x)))

    def quant_fp8_rows(self, x):
        """x [M, K] -> (codes uint8 [M, K], scale float32 [M]) by per-row absmax / 448."""
        x = _f64(x)
        M, K = x.shape
        codes = np.empty((M, K), dtype=np.uint8)
        scale = np.empty(M, dtype=np.float32)
        self.lib.oracle_quant_fp8_rows(_ptr(x), M, K, codes.ctypes.data_as(ctypes.POINTER(ctypes.c_ubyte)),
                                       scale.ctypes.data_as(ctypes.POINTER(ctypes.c_float)))
        return codes, scale

    def gemm_fp8(self, a, a_scale, b, b_scale) -> np.ndarray:
        """a [M, K], b [N, K] e4m3 codes; a_scale [M], b_scale [N] -> fp64 [M, N]."""
        a = np.ascontiguousarray(a, dtype=np.uint8)
        b = np.ascontiguousarray(b, dtype=np.uint8)
        sa = np.ascontiguousarray(a_scale, dtype=np.float32)
        sb = np.ascontiguousarray(b_scale, dtype=np.float32)
        M, K = a.shape
        N = b.shape[0]
        out = np.empty((M, N))
        u8 = ctypes.POINTER(ctypes.c_ubyte)
        f = ctypes.POINTER(ctypes.c_float)
        self.lib.oracle_gemm_fp8(a.ctypes.data_as(u8), sa.ctypes.data_as(f), b.ctypes.data_as(u8),
                                 sb.ctypes.data_as(f), M, N, K, _ptr(out))
        return out

    def rope_interleaved(self, x, cos, sin) -> np.ndarray:
        """x [B, S, H, D]; cos/sin [>=S, D/2]."""
        x = _f64(x)
        B, S, H, D = x.shape
        cos = _f64(cos[:S])
        sin = _f64(sin[:S])
        y = np.empty_like(x)
        self.lib.oracle_rope_interleaved(_ptr(x), _ptr(cos), _ptr(sin), B, S, H, D, _ptr(y))
        return y

    def qk_norm_rope(self, x, w, cos, sin, eps: float) -> np.ndarray:
        x = _f64(x)
        B, S, H, D = x.shape
        w = _f64(w)
        cos = _f64(cos[:S])
        sin = _f64(sin[:S])
        y = np.empty_like(x)
        self.lib.oracle_qk_norm_rope(_ptr(x), _ptr(w), _ptr(cos), _ptr(sin), B, S, H, D, eps, _ptr(y))
        return y

    def attention(self, q, k, v, scale: float, kv_begin: int = 0, kv_end: int | None = None, rows=None,
                  causal: bool = False):
        """q [B, Sq, H, D], k/v [B, Skv, H, D] -> (o [B, nrows, H, D], lse [B, H, nrows]).

        causal: query i sees only keys j <= i (top-left aligned)."""
        q, k, v = _f64(q), _f64(k), _f64(v)
        B, Sq, H, D = q.shape
        Skv = k.shape[1]
        kv_end = Skv if kv_end is None else kv_end
        if rows is None:
            nrows, rows_p = Sq, None
        else:
            rows = np.ascontiguousarray(rows, dtype=np.int64)
            nrows, rows_p = rows.size, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))
        o = np.empty((B, nrows, H, D))
        lse = np.empty((B, H, nrows))
        self.lib.oracle_attention_masked(_ptr(q), _ptr(k), _ptr(v), B, H, Sq, Skv, D, scale, kv_begin, kv_end,
                                         int(bool(causal)), rows_p, nrows, _ptr(o), _ptr(lse))
        return o, lse

    def attention_probs(self, q, k, scale: float, kv_begin: int = 0, kv_end: int | None = None) -> np.ndarray:
        q, k = _f64(q), _f64(k)
        B, Sq, H, D = q.shape
        Skv = k.shape[1]
        kv_end = Skv if kv_end is None else kv_end
        p = np.empty((B, H, Sq, kv_end - kv_begin))
        self.lib.oracle_attention_probs(_ptr(q), _ptr(k), B, H, Sq, Skv, D, scale, kv_begin, kv_end, _ptr(p))
        return p

    def merge_lse(self, o_parts, lse_parts):
        """o_parts [C, B, Sq, H, D], lse_parts [C, B, H, Sq] -> (o [B, Sq, H, D], lse [B, H, Sq])."""
        o_parts, lse_parts = _f64(o_parts), _f64(lse_parts)
        C, B, Sq, H, D = o_parts.shape
        o = np.empty((B, Sq, H, D))
        lse = np.empty((B, H, Sq))
        self.lib.oracle_merge_lse(_ptr(o_parts), _ptr(lse_parts), C, B, H, Sq, D, _ptr(o), _ptr(lse))
        return o, lse


def round_bf16(x) -> np.ndarray:
    """Round values to bfloat16 (to fp32 first, then to nearest-even bf16), returned as fp64.

    The path hands bf16 tensors from one operator to the next: the RMSNorm of
    "Cosmos Ascend NPU multi-card parallel optimisation notes", section 3.2.2,
    returns its result in the input dtype (`.type_as(x)`), and the fused
    attention of "NPU Wan2.2-I2V model inference optimisation practice" consumes
    those bf16 Q/K tensors.  Composing the oracle's fp64 operators, a test
    rounds at that boundary with this function.
    """
    f = np.ascontiguousarray(x, dtype=np.float64).astype(np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    r = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return r.astype(np.uint32).view(np.float32).astype(np.float64)


_DEFAULT: Oracle | None = None


def get() -> Oracle:
    """The oracle built from `oracle.c` (compiled on first use)."""
    global _DEFAULT
    if _DEFAULT is None:
        build()
        _DEFAULT = Oracle(LIBRARY)
    return _DEFAULT


def num_threads() -> int:
    return get().num_threads()

