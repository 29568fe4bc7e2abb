"""Python binding of the C ABI in include/ditattn.h (argument marshalling only).

Every computation runs in the CUDA kernels of libditattn.so.  PyTorch supplies
device memory and the current stream; nothing here computes on the host and
there is no fallback: if the library is missing or the tensors are not on a
CUDA device, the call raises.
"""

from __future__ import annotations

import ctypes
import math
from pathlib import Path

import torch

LIBRARY = Path(__file__).resolve().parent / "libditattn.so"

DIT_OK, DIT_ERR_INVALID_ARG, DIT_ERR_UNSUPPORTED, DIT_ERR_CUDA, DIT_ERR_TIMEOUT = range(5)
DIT_BF16, DIT_F32 = 0, 1
EXPORTED = ("dit_qk_norm_rope", "dit_attn_fwd", "dit_attn_merge_lse", "dit_poll_device_error",
            "dit_status_string", "dit_last_error_detail", "dit_selftest_wait_timeout", "dit_attn_fwd_causal",
            "dit_layer_norm_modulate", "dit_rms_norm", "dit_quant_fp8_rows", "dit_gemm_fp8", "dit_attn_fwd_update",
            "dit_set_launch_overlap", "dit_attention_host", "dit_attention_host_workspace",
            "dit_attention", "dit_attention_workspace", "dit_attention_noalloc", "dit_selftest_fp8_quotients",
            "dit_attention_ring_overlap", "dit_attention_ring_overlap_workspace")

_lib = None


class DitError(RuntimeError):
    def __init__(self, status: int, name: str, detail: str):
        super().__init__(f"{name}: {detail}" if detail else name)
        self.status = status


def load_library(path: Path | str = LIBRARY) -> ctypes.CDLL:
    """Load libditattn.so (raises if it has not been built)."""
    global _lib
    if _lib is not None and path == LIBRARY:
        return _lib
    path = Path(path)
    if not path.exists():
        raise RuntimeError(f"{path} is not built: run `python -m diffusion_transformer_attention_dit_gb300.build` "
                           "(there is no CPU fallback)")
    lib = ctypes.CDLL(str(path))
    vp, i32, i64p, f32 = ctypes.c_void_p, ctypes.c_int, ctypes.POINTER(ctypes.c_int64), ctypes.c_float
    lib.dit_qk_norm_rope.argtypes = [vp, vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, vp]
    lib.dit_attn_fwd.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i64p, i64p, f32, i32, i32, vp, i32, i64p,
                                 vp, vp]
    lib.dit_attn_fwd_causal.argtypes = lib.dit_attn_fwd.argtypes
    lib.dit_attn_fwd_update.argtypes = [vp, vp, vp, i32, i32, i32, i32, i32, i64p, i64p, f32, i32, i32, i32, vp, i32,
                                        i64p, vp, vp, i32, i64p, vp, vp]
    lib.dit_attn_merge_lse.argtypes = [vp, i32, vp, i32, i32, i32, i32, i32, ctypes.c_int64, ctypes.c_int64, vp,
                                       i32, vp, vp]
    lib.dit_layer_norm_modulate.argtypes = [vp, vp, vp, vp, i32, i32, i32, f32, vp]
    lib.dit_rms_norm.argtypes = [vp, vp, vp, ctypes.c_int64, i32, f32, vp]
    lib.dit_quant_fp8_rows.argtypes = [vp, vp, vp, ctypes.c_int64, i32, vp]
    lib.dit_gemm_fp8.argtypes = [vp, vp, vp, vp, vp, i32, i32, i32, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64,
                                 vp]
    lib.dit_poll_device_error.argtypes = [vp]
    lib.dit_selftest_wait_timeout.argtypes = [vp]
    lib.dit_selftest_fp8_quotients.argtypes = [ctypes.POINTER(ctypes.c_uint64), vp]
    lib.dit_set_launch_overlap.argtypes = [i32]
    lib.dit_attention_host.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, i32, i32, i32,
                                       vp, i32, vp, vp, ctypes.c_size_t, vp]
    lib.dit_attention_host_workspace.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32, i32]
    lib.dit_attention_host_workspace.restype = ctypes.c_size_t
    lib.dit_attention.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, i32, i32, i32, vp,
                                  i32, vp, vp, ctypes.c_size_t, vp, vp, vp]
    lib.dit_attention_workspace.argtypes = [i32, i32, i32, i32, i32, i32, i32, i32]
    lib.dit_attention_workspace.restype = ctypes.c_size_t
    lib.dit_attention_ring_overlap_workspace.argtypes = [i32, i32, i32, i32, i32, i32]
    lib.dit_attention_ring_overlap_workspace.restype = ctypes.c_size_t
    lib.dit_attention_ring_overlap.argtypes = [vp, vp, vp, i32, ctypes.POINTER(ctypes.c_void_p),
                                               ctypes.POINTER(ctypes.c_void_p), ctypes.POINTER(ctypes.c_int), i32,
                                               i32, i32, i32, i32, f32, i32, vp, i32, vp, vp, ctypes.c_size_t, vp]
    lib.dit_attention_noalloc.argtypes = [vp, vp, vp, vp, vp, vp, vp, i32, i32, i32, i32, f32, f32, i32, i32, i32, i32,
                                          vp, i32, vp, vp]
    for name in ("dit_qk_norm_rope", "dit_attn_fwd", "dit_attn_fwd_causal", "dit_attn_merge_lse",
                 "dit_poll_device_error", "dit_selftest_wait_timeout", "dit_layer_norm_modulate", "dit_rms_norm",
                 "dit_quant_fp8_rows", "dit_gemm_fp8", "dit_attn_fwd_update", "dit_set_launch_overlap",
                 "dit_attention_host", "dit_attention", "dit_attention_noalloc", "dit_attention_ring_overlap",
                 "dit_selftest_fp8_quotients"):
        getattr(lib, name).restype = ctypes.c_int
    lib.dit_status_string.argtypes = [ctypes.c_int]
    lib.dit_status_string.restype = ctypes.c_char_p
    lib.dit_last_error_detail.argtypes = []
    lib.dit_last_error_detail.restype = ctypes.c_char_p
    if path == LIBRARY:
        _lib = lib
    return lib


def _check(status: int):
    if status != DIT_OK:
        lib = load_library()
        raise DitError(status, lib.dit_status_string(status).decode(), lib.dit_last_error_detail().decode())


def _stream(stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream()
    return stream.cuda_stream


def _cuda(*ts):
    for t in ts:
        if not t.is_cuda:
            raise ValueError("all tensors must be CUDA tensors (there is no CPU path)")


def _dtype_code(dt: torch.dtype) -> int:
    if dt == torch.bfloat16:
        return DIT_BF16
    if dt == torch.float32:
        return DIT_F32
    raise ValueError(f"unsupported dtype {dt}")


def _bshd_strides(t: torch.Tensor):
    if t.dim() != 4 or t.stride(3) != 1:
        raise ValueError("expected a [B, S, H, D] tensor with contiguous last dim")
    return (ctypes.c_int64 * 3)(t.stride(0), t.stride(1), t.stride(2))


def qk_norm_rope(q, k, wq, wk, cos, sin, eps: float = 1e-6, q_out=None, k_out=None, stream=None):
    """QK-RMSNorm + interleaved RoPE.  q, k bf16 [B, S, H, D] contiguous; wq, wk fp32 [D]; cos, sin fp32 [S, D/2]."""
    lib = load_library()
    _cuda(q, k, wq, wk, cos, sin)
    B, S, H, D = q.shape
    if k.shape != q.shape or q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16:
        raise ValueError("q and k must be bf16 tensors of the same shape")
    if not (q.is_contiguous() and k.is_contiguous() and cos.is_contiguous() and sin.is_contiguous()):
        raise ValueError("q, k, cos, sin must be contiguous")
    if wq.dtype != torch.float32 or wk.dtype != torch.float32 or cos.dtype != torch.float32 or sin.dtype != torch.float32:
        raise ValueError("weights and tables must be fp32")
    if cos.shape[0] < S or cos.shape[-1] * 2 != D or sin.shape != cos.shape:
        raise ValueError("cos/sin must be [>=S, D/2]")
    q_out = torch.empty_like(q) if q_out is None else q_out
    k_out = torch.empty_like(k) if k_out is None else k_out
    _check(lib.dit_qk_norm_rope(q.data_ptr(), k.data_ptr(), q_out.data_ptr(), k_out.data_ptr(), wq.data_ptr(),
                                wk.data_ptr(), cos.data_ptr(), sin.data_ptr(), B, S, H, D, float(eps),
                                _stream(stream)))
    return q_out, k_out


def attn_fwd(q, k, v, scale: float | None = None, kv_begin: int = 0, kv_end: int | None = None, o=None, lse=None,
             o_dtype=torch.bfloat16, stream=None, causal: bool = False):
    """Flash attention forward over keys [kv_begin, kv_end).  Returns (o [B, Sq, H, D], lse fp32 [B, H, Sq]).

    causal=True masks keys after each query (query i sees keys j <= i)."""
    lib = load_library()
    _cuda(q, k, v)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != H or k.shape[3] != D:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bf16")
    if k.stride() != v.stride():
        raise ValueError("k and v must share strides")
    kv_end = Skv if kv_end is None else kv_end
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if o is None:
        o = torch.empty((B, Sq, H, D), dtype=o_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    if lse.dtype != torch.float32 or not lse.is_contiguous() or tuple(lse.shape) != (B, H, Sq):
        raise ValueError("lse must be contiguous fp32 [B, H, Sq]")
    fn = lib.dit_attn_fwd_causal if causal else lib.dit_attn_fwd
    _check(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, Sq, Skv, D, _bshd_strides(q),
                            _bshd_strides(k), float(scale), int(kv_begin), int(kv_end), o.data_ptr(),
                            _dtype_code(o.dtype), _bshd_strides(o), lse.data_ptr(), _stream(stream)))
    return o, lse


def attn_fwd_update(q, k, v, o_acc, lse_acc, scale: float | None = None, kv_begin: int = 0, kv_end: int | None = None,
                    o=None, lse=None, o_dtype=torch.bfloat16, stream=None, causal: bool = False):
    """Attention over keys [kv_begin, kv_end) LSE-merged into the running result (o_acc, lse_acc) of earlier key
    ranges, in the attention's epilogue.  o / lse may be o_acc / lse_acc (in place).  Returns (o, lse)."""
    lib = load_library()
    _cuda(q, k, v, o_acc, lse_acc)
    B, Sq, H, D = q.shape
    Skv = k.shape[1]
    if k.shape != v.shape or k.shape[0] != B or k.shape[2] != H or k.shape[3] != D:
        raise ValueError("k and v must be [B, Skv, H, D] matching q")
    if q.dtype != torch.bfloat16 or k.dtype != torch.bfloat16 or v.dtype != torch.bfloat16:
        raise ValueError("q, k, v must be bf16")
    if k.stride() != v.stride():
        raise ValueError("k and v must share strides")
    if tuple(o_acc.shape) != (B, Sq, H, D):
        raise ValueError("o_acc must be [B, Sq, H, D]")
    for t in (lse_acc, lse):
        if t is not None and (t.dtype != torch.float32 or not t.is_contiguous() or tuple(t.shape) != (B, H, Sq)):
            raise ValueError("lse and lse_acc must be contiguous fp32 [B, H, Sq]")
    kv_end = Skv if kv_end is None else kv_end
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if o is None:
        o = torch.empty((B, Sq, H, D), dtype=o_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=q.device)
    _check(lib.dit_attn_fwd_update(q.data_ptr(), k.data_ptr(), v.data_ptr(), B, H, Sq, Skv, D, _bshd_strides(q),
                                   _bshd_strides(k), float(scale), int(kv_begin), int(kv_end), int(bool(causal)),
                                   o_acc.data_ptr(), _dtype_code(o_acc.dtype), _bshd_strides(o_acc),
                                   lse_acc.data_ptr(), o.data_ptr(), _dtype_code(o.dtype), _bshd_strides(o),
                                   lse.data_ptr(), _stream(stream)))
    return o, lse


def attn_merge_lse(o_parts, lse_parts, out_dtype=torch.bfloat16, o=None, lse=None, stream=None):
    """Merge C partials: o_parts [C, B, Sq, H, D] (bf16/fp32), lse_parts fp32 [C, B, H, Sq]."""
    lib = load_library()
    _cuda(o_parts, lse_parts)
    C, B, Sq, H, D = o_parts.shape
    if tuple(lse_parts.shape) != (C, B, H, Sq) or lse_parts.dtype != torch.float32:
        raise ValueError("lse_parts must be fp32 [C, B, H, Sq]")
    if not (o_parts[0].is_contiguous() and lse_parts[0].is_contiguous()):
        raise ValueError("each part must be contiguous")
    if o is None:
        o = torch.empty((B, Sq, H, D), dtype=out_dtype, device=o_parts.device)
    if lse is None:
        lse = torch.empty((B, H, Sq), dtype=torch.float32, device=o_parts.device)
    if not (o.is_contiguous() and lse.is_contiguous()):
        raise ValueError("outputs must be contiguous")
    _check(lib.dit_attn_merge_lse(o_parts.data_ptr(), _dtype_code(o_parts.dtype), lse_parts.data_ptr(), C, B, H, Sq,
                                  D, o_parts.stride(0), lse_parts.stride(0), o.data_ptr(), _dtype_code(o.dtype),
                                  lse.data_ptr(), _stream(stream)))
    return o, lse


def layer_norm_modulate(x, scale=None, shift=None, eps: float = 1e-6, y=None, stream=None):
    """LayerNorm over C with adaLN modulation: x bf16 [B, L, C]; scale, shift fp32 [B, C] (or None)."""
    lib = load_library()
    _cuda(x)
    B, L, C = x.shape
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("x must be contiguous bf16 [B, L, C]")
    for t in (scale, shift):
        if t is not None and (not t.is_cuda or t.dtype != torch.float32 or tuple(t.shape) != (B, C)
                              or not t.is_contiguous()):
            raise ValueError("scale / shift must be contiguous fp32 [B, C] on the GPU")
    y = torch.empty_like(x) if y is None else y
    _check(lib.dit_layer_norm_modulate(x.data_ptr(), 0 if scale is None else scale.data_ptr(),
                                       0 if shift is None else shift.data_ptr(), y.data_ptr(), B, L, C, float(eps),
                                       _stream(stream)))
    return y


def rms_norm(x, w, eps: float = 1e-6, y=None, stream=None):
    """RMSNorm over the last dim C of a contiguous bf16 tensor with fp32 weight [C]."""
    lib = load_library()
    _cuda(x, w)
    C = x.shape[-1]
    if x.dtype != torch.bfloat16 or not x.is_contiguous() or w.dtype != torch.float32 or w.numel() != C:
        raise ValueError("x must be contiguous bf16 [..., C] and w fp32 [C]")
    y = torch.empty_like(x) if y is None else y
    _check(lib.dit_rms_norm(x.data_ptr(), w.data_ptr(), y.data_ptr(), x.numel() // C, C, float(eps),
                            _stream(stream)))
    return y


def quant_fp8_rows(x, codes=None, scale=None, stream=None):
    """Per-row dynamic e4m3 quantisation of bf16 x [M, K] -> (codes uint8 [M, K], scale fp32 [M])."""
    lib = load_library()
    _cuda(x)
    M, K = x.shape
    if x.dtype != torch.bfloat16 or not x.is_contiguous():
        raise ValueError("x must be contiguous bf16 [M, K]")
    codes = torch.empty((M, K), dtype=torch.uint8, device=x.device) if codes is None else codes
    scale = torch.empty(M, dtype=torch.float32, device=x.device) if scale is None else scale
    _check(lib.dit_quant_fp8_rows(x.data_ptr(), codes.data_ptr(), scale.data_ptr(), M, K, _stream(stream)))
    return codes, scale


def gemm_fp8(a, a_scale, b, b_scale, out=None, stream=None):
    """out[m, n] = a_scale[m] b_scale[n] sum_k A[m, k] B[n, k]; a [M, K], b [N, K] uint8 e4m3 codes -> bf16 [M, N]."""
    lib = load_library()
    _cuda(a, b, a_scale, b_scale)
    M, K = a.shape
    N = b.shape[0]
    if a.dtype != torch.uint8 or b.dtype != torch.uint8 or b.shape[1] != K or a.stride(1) != 1 or b.stride(1) != 1:
        raise ValueError("a, b must be uint8 [M, K] / [N, K] with contiguous rows")
    out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device) if out is None else out
    _check(lib.dit_gemm_fp8(a.data_ptr(), a_scale.data_ptr(), b.data_ptr(), b_scale.data_ptr(), out.data_ptr(), M, N,
                            K, a.stride(0), b.stride(0), out.stride(0), _stream(stream)))
    return out


def poll_device_error(stream=None):
    """Synchronise the stream and raise DitError if a bounded device-side wait gave up since the last poll."""
    _check(load_library().dit_poll_device_error(_stream(stream)))


def set_launch_overlap(enable: bool):
    """Programmatic dependent launch for the library's kernels (default on): a kernel's launch overlaps the tail of
    the previous kernel on its stream; every kernel waits for that kernel before touching global memory."""
    _check(load_library().dit_set_launch_overlap(1 if enable else 0))


def selftest_wait_timeout(stream=None):
    """Run the bounded-wait self-test kernel; a following poll_device_error() must raise DIT_ERR_TIMEOUT."""
    _check(load_library().dit_selftest_wait_timeout(_stream(stream)))


def selftest_fp8_quotients(stream=None):
    """Exhaustive check of the fp8 quantiser's division against IEEE division; returns (fp32 quotient mismatches,
    e4m3 code mismatches) over every bf16 row maximum and element.  The codes are the output and must all agree."""
    counts = (ctypes.c_uint64 * 2)()
    _check(load_library().dit_selftest_fp8_quotients(counts, _stream(stream)))
    return int(counts[0]), int(counts[1])


def attention_workspace_bytes(B, S, H, D, chunks=1, prologue=True, partial_dtype=torch.float32,
                              merge: str = "kernel") -> int:
    """Device workspace bytes dit_attention needs for these sizes."""
    return int(load_library().dit_attention_workspace(B, S, H, D, chunks, int(bool(prologue)),
                                                      _dtype_code(partial_dtype), int(merge == "update")))


def _event_handle(ev, stream) -> int:
    # torch creates the CUDA event on its first record: record a fresh one once so the handle exists (the library
    # records it again at the right place on the stream); create events ahead of a timed region to avoid that
    if ev is None:
        return 0
    if not ev.cuda_event:
        ev.record(stream)
    return ev.cuda_event


def dit_attention(q, k, v, wq, wk, cos, sin, eps: float = 1e-6, chunks: int = 1, scale: float | None = None,
                  partial_dtype=torch.float32, out_dtype=torch.bfloat16, prologue: bool = True, stream=None,
                  merge: str = "kernel", o=None, lse=None, workspace=None, attn_events=None):
    """The whole hot path in one C call (dit_attention): prologue, attention over `chunks` KV chunks, merge.
    Returns (o, lse).

    merge="kernel": every chunk writes (O_c, LSE_c) into stacked partials and one merge kernel combines them.
    merge="update": chunk 0 writes a running result (partial_dtype), every later chunk is LSE-merged into it in
    its attention epilogue, the last one straight into the output.  `workspace`: a device uint8 tensor of at least
    attention_workspace_bytes(...) bytes (allocated here when None).  attn_events: optional pair of
    torch.cuda.Event recorded before the first and after the last attention launch."""
    if merge not in ("kernel", "update"):
        raise ValueError("merge must be 'kernel' or 'update'")
    lib = load_library()
    _cuda(q, k, v)
    for t in (q, k, v):
        if t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 [B, S, H, D] tensors")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, S, H, D]")
    B, S, H, D = q.shape
    if prologue:
        _cuda(wq, wk, cos, sin)
        for t in (wq, wk, cos, sin):
            if t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError("wq, wk, cos, sin must be contiguous fp32 tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if o is None:
        o = torch.empty((B, S, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    _cuda(o, lse)
    if not o.is_contiguous() or not lse.is_contiguous() or lse.dtype != torch.float32:
        raise ValueError("o must be contiguous; lse contiguous fp32")
    need = attention_workspace_bytes(B, S, H, D, chunks, prologue, partial_dtype, merge)
    if workspace is None:
        workspace = torch.empty(max(need, 1), dtype=torch.uint8, device=q.device)
    _cuda(workspace)
    st = torch.cuda.current_stream() if stream is None else stream
    e0, e1 = (None, None) if attn_events is None else attn_events
    ptr = (lambda t: t.data_ptr()) if prologue else (lambda t: None)
    _check(lib.dit_attention(q.data_ptr(), k.data_ptr(), v.data_ptr(), ptr(wq), ptr(wk), ptr(cos), ptr(sin), B, S, H,
                             D, eps, scale, chunks, int(bool(prologue)), _dtype_code(partial_dtype),
                             int(merge == "update"), o.data_ptr(), _dtype_code(o.dtype), lse.data_ptr(),
                             workspace.data_ptr(), workspace.numel() * workspace.element_size(),
                             _event_handle(e0, st), _event_handle(e1, st), st.cuda_stream))
    return o, lse


def attention_host_workspace_bytes(B, S, H, D, chunks=1, prologue=True, partial_dtype=torch.float32,
                                   out_dtype=torch.bfloat16, merge: str = "update") -> int:
    """Device workspace bytes dit_attention_host needs for these sizes."""
    if merge not in ("kernel", "update"):
        raise ValueError("merge must be 'kernel' or 'update'")
    return int(load_library().dit_attention_host_workspace(B, S, H, D, chunks, int(bool(prologue)),
                                                           _dtype_code(partial_dtype), int(merge == "update"),
                                                           _dtype_code(out_dtype)))


def dit_attention_host(q, k, v, wq=None, wk=None, cos=None, sin=None, eps: float = 1e-6, chunks: int = 1,
                       scale: float | None = None, partial_dtype=torch.float32, out_dtype=torch.bfloat16,
                       prologue: bool = True, merge: str = "update", o=None, lse=None, workspace=None, stream=None):
    """The whole hot path from host tensors (pinned for asynchronous copies): q, k, v bf16 [B, S, H, D]; wq, wk
    fp32 [D]; cos, sin fp32 [S, D/2].  merge="update": the value rows of each KV chunk are copied while earlier
    chunks compute, later chunks merged into a running result in their epilogue.  merge="kernel": stacked partials
    and the merge kernel over query-row ranges, each range's result copied back while the next computes.
    Returns host (o, lse); they are valid once the stream has completed the call, and the inputs must stay
    referenced until then (the copies read them asynchronously).  `workspace` is a device uint8 tensor of at
    least attention_host_workspace_bytes(...) bytes (allocated here when None)."""
    if merge not in ("kernel", "update"):
        raise ValueError("merge must be 'kernel' or 'update'")
    lib = load_library()
    for t in (q, k, v):
        if t.device.type != "cpu" or t.dtype != torch.bfloat16 or not t.is_contiguous():
            raise ValueError("q, k, v must be contiguous bf16 host tensors")
    if k.shape != q.shape or v.shape != q.shape:
        raise ValueError("q, k, v must have the same shape [B, S, H, D]")
    B, S, H, D = q.shape
    if prologue:
        for t in (wq, wk, cos, sin):
            if t is None or t.device.type != "cpu" or t.dtype != torch.float32 or not t.is_contiguous():
                raise ValueError("wq, wk, cos, sin must be contiguous fp32 host tensors")
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    pin = q.is_pinned()
    if o is None:
        o = torch.empty((B, S, H, D), dtype=out_dtype, pin_memory=pin)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, pin_memory=pin)
    if o.device.type != "cpu" or lse.device.type != "cpu" or not (o.is_contiguous() and lse.is_contiguous()):
        raise ValueError("o and lse must be contiguous host tensors")
    need = attention_host_workspace_bytes(B, S, H, D, chunks, prologue, partial_dtype, o.dtype, merge)
    if workspace is None:
        workspace = torch.empty(need, dtype=torch.uint8, device="cuda")
        if stream is not None:  # the allocator must not hand the block out again before `stream` is done with it
            workspace.record_stream(stream)
    if not workspace.is_cuda or workspace.numel() * workspace.element_size() < need:
        raise ValueError(f"workspace must be a device tensor of at least {need} bytes")
    ptr = lambda t: None if t is None else t.data_ptr()  # noqa: E731
    _check(lib.dit_attention_host(q.data_ptr(), k.data_ptr(), v.data_ptr(), ptr(wq), ptr(wk), ptr(cos), ptr(sin),
                                  B, S, H, D, float(eps), float(scale), int(chunks), int(bool(prologue)),
                                  _dtype_code(partial_dtype), int(merge == "update"), o.data_ptr(),
                                  _dtype_code(o.dtype), lse.data_ptr(), workspace.data_ptr(),
                                  workspace.numel() * workspace.element_size(), _stream(stream)))
    return o, lse


def ring_overlap_workspace_bytes(B, S, H, D, s_remote, partial_dtype=torch.float32) -> int:
    """Device workspace bytes dit_attention_ring_overlap needs (s_remote = total remote keys)."""
    return int(load_library().dit_attention_ring_overlap_workspace(B, S, H, D, s_remote, _dtype_code(partial_dtype)))


def ring_overlap_attention(q, k_local, v_local, remote_kv, scale: float | None = None, out_dtype=torch.bfloat16,
                           partial_dtype=torch.float32, o=None, lse=None, workspace=None, stream=None):
    """One rank's ring-attention overlap on one GPU (dit_attention_ring_overlap; "NPU Wan2.2-I2V model inference
    optimisation practice", section "Ring Attention Overlap").

    The attention over the local K/V runs on the stream while the remote K/V shards are copied into one contiguous
    buffer on a side stream (device copies stand in for the all-gather of a multi-GPU run); then one attention over
    the gathered shards whose epilogue LSE-merges it into the local result (update_out_and_lse).  remote_kv is a
    list of (k_i, v_i) contiguous bf16 tensors [B, S_i, H, D].  Returns (o, lse)."""
    lib = load_library()
    _cuda(q, k_local, v_local)
    B, S, H, D = q.shape
    s_local = k_local.shape[1]
    for t in [q, k_local, v_local] + [x for kv in remote_kv for x in kv]:
        if t.dtype != torch.bfloat16 or not t.is_contiguous() or t.dim() != 4:
            raise ValueError("q, k, v shards must be contiguous bf16 [B, S, H, D]")
    if k_local.shape != v_local.shape or any(kk.shape != vv.shape for kk, vv in remote_kv):
        raise ValueError("each shard's k and v must have the same shape")
    R = len(remote_kv)
    s_rem = [int(kk.shape[1]) for kk, _ in remote_kv]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    if o is None:
        o = torch.empty((B, S, H, D), dtype=out_dtype, device=q.device)
    if lse is None:
        lse = torch.empty((B, H, S), dtype=torch.float32, device=q.device)
    wsb = ring_overlap_workspace_bytes(B, S, H, D, sum(s_rem), partial_dtype) if R else 0
    if workspace is None:
        workspace = torch.empty(max(wsb, 1), dtype=torch.uint8, device=q.device)
    kp = (ctypes.c_void_p * max(R, 1))(*[kk.data_ptr() for kk, _ in remote_kv])
    vp_ = (ctypes.c_void_p * max(R, 1))(*[vv.data_ptr() for _, vv in remote_kv])
    sr = (ctypes.c_int * max(R, 1))(*s_rem)
    _check(lib.dit_attention_ring_overlap(q.data_ptr(), k_local.data_ptr(), v_local.data_ptr(), s_local, kp, vp_, sr,
                                          R, B, S, H, D, float(scale), _dtype_code(partial_dtype), o.data_ptr(),
                                          _dtype_code(o.dtype), lse.data_ptr(), workspace.data_ptr(),
                                          workspace.numel(), _stream(stream)))
    return o, lse

