"""Host-side checks of the C ABI: the library loads without a GPU, exports every
function declared in include/ditattn.h, and rejects bad arguments with a status
code before launching anything."""

import ctypes
import re
from pathlib import Path

import pytest

from diffusion_transformer_attention_dit_gb300 import build, ops

ROOT = Path(__file__).resolve().parent.parent
HEADER = ROOT / "include" / "ditattn.h"


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def _declared():
    text = HEADER.read_text()
    return sorted(set(re.findall(r"^(?:const char \*|dit_status |size_t )(dit_\w+)\(", text, flags=re.M)))


def test_header_declares_the_boundary():
    names = _declared()
    for n in ("dit_qk_norm_rope", "dit_attn_fwd", "dit_attn_merge_lse", "dit_poll_device_error",
              "dit_status_string"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    for name in _declared():
        assert hasattr(lib, name), name


def test_status_strings(lib):
    assert lib.dit_status_string(0) == b"DIT_OK"
    assert lib.dit_status_string(4) == b"DIT_ERR_TIMEOUT"
    assert lib.dit_status_string(99) == b"DIT_ERR_UNKNOWN"


A16 = 1 << 20  # a 16-byte aligned fake device address (never dereferenced: validation fails first)


def _st(*v):
    return (ctypes.c_int64 * 3)(*v)


def _attn(lib, **kw):
    a = dict(q=A16, k=A16 * 2, v=A16 * 3, B=1, H=2, Sq=256, Skv=256, D=128, qs=_st(256 * 256, 256, 128),
             kvs=_st(256 * 256, 256, 128), scale=0.088, lo=0, hi=256, o=A16 * 8, od=0, os=_st(256 * 256, 256, 128),
             lse=A16 * 16, stream=None)
    a.update(kw)
    return lib.dit_attn_fwd(a["q"], a["k"], a["v"], a["B"], a["H"], a["Sq"], a["Skv"], a["D"], a["qs"], a["kvs"],
                            a["scale"], a["lo"], a["hi"], a["o"], a["od"], a["os"], a["lse"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), ops.DIT_ERR_UNSUPPORTED),
    (dict(q=None), ops.DIT_ERR_INVALID_ARG),
    (dict(q=A16 + 8), ops.DIT_ERR_INVALID_ARG),
    (dict(lo=10, hi=10), ops.DIT_ERR_INVALID_ARG),
    (dict(lo=0, hi=257), ops.DIT_ERR_INVALID_ARG),
    (dict(lo=-1), ops.DIT_ERR_INVALID_ARG),
    (dict(scale=0.0), ops.DIT_ERR_INVALID_ARG),
    (dict(scale=float("inf")), ops.DIT_ERR_INVALID_ARG),
    (dict(qs=_st(256 * 256, 255, 128)), ops.DIT_ERR_INVALID_ARG),
    (dict(od=7), ops.DIT_ERR_INVALID_ARG),
    (dict(o=A16), ops.DIT_ERR_INVALID_ARG),          # output aliases q
    (dict(lse=A16 * 8 + 64), ops.DIT_ERR_INVALID_ARG),  # lse inside o
    (dict(B=-1), ops.DIT_ERR_INVALID_ARG),
])
def test_attn_rejects_bad_arguments(lib, kw, code):
    assert _attn(lib, **kw) == code
    assert lib.dit_last_error_detail() != b""


def test_attn_empty_work_is_ok_without_launch(lib):
    assert _attn(lib, B=0) == ops.DIT_OK
    assert _attn(lib, Sq=0) == ops.DIT_OK


def _update(lib, **kw):
    a = dict(q=A16, k=A16 * 2, v=A16 * 3, B=1, H=2, Sq=256, Skv=256, D=128, qs=_st(256 * 256, 256, 128),
             kvs=_st(256 * 256, 256, 128), scale=0.088, lo=0, hi=256, causal=0, acc=A16 * 32, ad=1,
             acs=_st(256 * 256, 256, 128), lacc=A16 * 48, o=A16 * 8, od=0, os=_st(256 * 256, 256, 128),
             lse=A16 * 16)
    a.update(kw)
    return lib.dit_attn_fwd_update(a["q"], a["k"], a["v"], a["B"], a["H"], a["Sq"], a["Skv"], a["D"], a["qs"],
                                   a["kvs"], a["scale"], a["lo"], a["hi"], a["causal"], a["acc"], a["ad"], a["acs"],
                                   a["lacc"], a["o"], a["od"], a["os"], a["lse"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(causal=2), ops.DIT_ERR_INVALID_ARG),
    (dict(acc=None), ops.DIT_ERR_INVALID_ARG),
    (dict(lacc=None), ops.DIT_ERR_INVALID_ARG),
    (dict(acs=None), ops.DIT_ERR_INVALID_ARG),
    (dict(ad=7), ops.DIT_ERR_INVALID_ARG),
    (dict(acc=A16 * 32 + 8), ops.DIT_ERR_INVALID_ARG),          # misaligned
    (dict(acs=_st(256 * 256, 254, 128)), ops.DIT_ERR_INVALID_ARG),  # fp32 stride not a multiple of 16 bytes
    (dict(acc=A16 * 8 + 256), ops.DIT_ERR_INVALID_ARG),         # overlaps o without being it
    (dict(acc=A16 * 8), ops.DIT_ERR_INVALID_ARG),               # same pointer as o but another dtype
    (dict(lacc=A16 * 8 + 64), ops.DIT_ERR_INVALID_ARG),         # running LSE inside o
    (dict(lacc=A16 * 16 + 4), ops.DIT_ERR_INVALID_ARG),         # running LSE overlaps lse without being it
    (dict(lo=5, hi=5), ops.DIT_ERR_INVALID_ARG),
    (dict(D=96), ops.DIT_ERR_UNSUPPORTED),
])
def test_update_rejects_bad_arguments(lib, kw, code):
    assert _update(lib, **kw) == code
    assert lib.dit_last_error_detail() != b""


def test_update_empty_work_is_ok_without_launch(lib):
    assert _update(lib, Sq=0) == ops.DIT_OK
    assert _update(lib, B=0, acc=None) == ops.DIT_OK


def _ring(lib, **kw):
    a = dict(q=A16, kl=A16 * 2, vl=A16 * 3, sl=256, kr=[A16 * 4], vr=[A16 * 5], sr=[256], B=1, S=256, H=2, D=128,
             scale=0.088, pdt=1, o=A16 * 8, odt=0, lse=A16 * 16, ws=A16 * 64, wsb=1 << 30)
    a.update(kw)
    R = len(a["kr"])
    kr = (ctypes.c_void_p * max(R, 1))(*a["kr"])
    vr = (ctypes.c_void_p * max(R, 1))(*a["vr"])
    sr = (ctypes.c_int * max(len(a["sr"]), 1))(*a["sr"])
    return lib.dit_attention_ring_overlap(a["q"], a["kl"], a["vl"], a["sl"], kr, vr, sr, a.get("R", R), a["B"],
                                          a["S"], a["H"], a["D"], a["scale"], a["pdt"], a["o"], a["odt"], a["lse"],
                                          a["ws"], a["wsb"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(R=-1), ops.DIT_ERR_INVALID_ARG),
    (dict(sl=0), ops.DIT_ERR_INVALID_ARG),
    (dict(sr=[0]), ops.DIT_ERR_INVALID_ARG),              # an empty remote shard
    (dict(kr=[None]), ops.DIT_ERR_INVALID_ARG),
    (dict(vr=[A16 * 5 + 8]), ops.DIT_ERR_INVALID_ARG),    # remote shard misaligned
    (dict(D=80), ops.DIT_ERR_UNSUPPORTED),
    (dict(pdt=4), ops.DIT_ERR_INVALID_ARG),
    (dict(q=A16 + 4), ops.DIT_ERR_INVALID_ARG),
    (dict(scale=0.0), ops.DIT_ERR_INVALID_ARG),
    (dict(o=A16 * 4), ops.DIT_ERR_INVALID_ARG),           # output over a remote shard
    (dict(lse=A16 * 8 + 64), ops.DIT_ERR_INVALID_ARG),    # lse inside o
    (dict(ws=None), ops.DIT_ERR_INVALID_ARG),
    (dict(ws=A16 * 64 + 16), ops.DIT_ERR_INVALID_ARG),    # workspace misaligned
    (dict(wsb=1024), ops.DIT_ERR_INVALID_ARG),            # workspace too small
    (dict(ws=A16 * 8), ops.DIT_ERR_INVALID_ARG),          # workspace over o
])
def test_ring_overlap_rejects_bad_arguments(lib, kw, code):
    assert _ring(lib, **kw) == code
    assert lib.dit_last_error_detail() != b""


def test_ring_overlap_workspace_and_empty_work(lib):
    assert lib.dit_attention_ring_overlap_workspace(1, 256, 2, 128, 256, 1) >= 2 * 256 * 2 * 128 * 2 + 256 * 2 * 128 * 4
    assert lib.dit_attention_ring_overlap_workspace(1, 256, 2, 128, -1, 1) == 0
    assert _ring(lib, B=0) == ops.DIT_OK


def _prologue(lib, **kw):
    a = dict(q=A16, k=A16 * 2, qo=A16 * 3, ko=A16 * 4, wq=A16 * 5, wk=A16 * 6, cos=A16 * 7, sin=A16 * 8, B=1, S=16,
             H=2, D=128, eps=1e-6)
    a.update(kw)
    return lib.dit_qk_norm_rope(a["q"], a["k"], a["qo"], a["ko"], a["wq"], a["wk"], a["cos"], a["sin"], a["B"],
                                a["S"], a["H"], a["D"], a["eps"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(D=80), ops.DIT_ERR_UNSUPPORTED),
    (dict(cos=None), ops.DIT_ERR_INVALID_ARG),
    (dict(qo=A16 + 4), ops.DIT_ERR_INVALID_ARG),
    (dict(eps=-1.0), ops.DIT_ERR_INVALID_ARG),
    (dict(ko=A16), ops.DIT_ERR_INVALID_ARG),        # k_out overlaps q
    (dict(qo=A16 + 1024), ops.DIT_ERR_INVALID_ARG),  # partial overlap with q
])
def test_prologue_rejects_bad_arguments(lib, kw, code):
    assert _prologue(lib, **kw) == code


def test_prologue_empty_is_ok(lib):
    assert _prologue(lib, S=0) == ops.DIT_OK


def _merge(lib, **kw):
    a = dict(op=A16, idt=0, lp=A16 * 64, C=4, B=1, H=2, Sq=64, D=128, pso=64 * 2 * 128, psl=2 * 64, o=A16 * 128,
             odt=0, lse=A16 * 160)
    a.update(kw)
    return lib.dit_attn_merge_lse(a["op"], a["idt"], a["lp"], a["C"], a["B"], a["H"], a["Sq"], a["D"], a["pso"],
                                  a["psl"], a["o"], a["odt"], a["lse"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(C=0), ops.DIT_ERR_INVALID_ARG),
    (dict(D=32), ops.DIT_ERR_UNSUPPORTED),
    (dict(pso=100), ops.DIT_ERR_INVALID_ARG),
    (dict(idt=3), ops.DIT_ERR_INVALID_ARG),
    (dict(o=A16 + 4096), ops.DIT_ERR_INVALID_ARG),   # o inside the parts
    (dict(C=5000), ops.DIT_ERR_UNSUPPORTED),
])
def test_merge_rejects_bad_arguments(lib, kw, code):
    assert _merge(lib, **kw) == code


def test_merge_empty_is_ok(lib):
    assert _merge(lib, Sq=0) == ops.DIT_OK


@pytest.mark.parametrize("C,code", [(12, ops.DIT_ERR_UNSUPPORTED), (8200, ops.DIT_ERR_UNSUPPORTED),
                                    (64, ops.DIT_OK)])
def test_norm_entry_points_check_channels(lib, C, code):
    # B = 0 makes the valid case empty work (no launch)
    assert lib.dit_layer_norm_modulate(A16, None, None, A16 * 2, 0 if code == ops.DIT_OK else 1, 4, C, 1e-6,
                                       None) == code
    assert lib.dit_rms_norm(A16, A16 * 4, A16 * 2, 0 if code == ops.DIT_OK else 4, C, 1e-6, None) == code


def test_norm_rejects_overlap(lib):
    assert lib.dit_layer_norm_modulate(A16, None, None, A16 + 64, 1, 4, 64, 1e-6, None) == ops.DIT_ERR_INVALID_ARG
    assert lib.dit_rms_norm(A16, A16 * 4, A16 + 64, 4, 64, 1e-6, None) == ops.DIT_ERR_INVALID_ARG


def test_binding_refuses_cpu_tensors(lib):
    import torch

    q = torch.zeros(1, 8, 1, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        ops.attn_fwd(q, q, q)


def test_launch_overlap_setting(lib):
    assert lib.dit_set_launch_overlap(2) == ops.DIT_ERR_INVALID_ARG
    assert lib.dit_set_launch_overlap(0) == ops.DIT_OK
    assert lib.dit_set_launch_overlap(1) == ops.DIT_OK


def _host(lib, **kw):
    B, S, H, D = kw.pop("B", 1), kw.pop("S", 64), kw.pop("H", 2), kw.pop("D", 128)
    chunks, prologue, mu = kw.pop("chunks", 2), kw.pop("prologue", 1), kw.pop("merge_update", 1)
    need = lib.dit_attention_host_workspace(B, S, H, D, chunks, 1, 1, 1 if mu not in (0, 1) else mu, 0)
    a = dict(q=A16, k=A16 * 2, v=A16 * 3, wq=A16 * 4, wk=A16 * 5, cos=A16 * 6, sin=A16 * 7, o=A16 * 8, lse=A16 * 9,
             ws=A16 * 16, wsb=need, pdt=1, odt=0)
    a.update(kw)
    return lib.dit_attention_host(a["q"], a["k"], a["v"], a["wq"], a["wk"], a["cos"], a["sin"], B, S, H, D, 1e-6,
                                  0.088, chunks, prologue, a["pdt"], mu, a["o"], a["odt"], a["lse"], a["ws"],
                                  a["wsb"], None)


def test_host_workspace_size(lib):
    B, S, H, D = 2, 100, 3, 128
    act = B * S * H * D * 2
    n = lib.dit_attention_host_workspace(B, S, H, D, 2, 1, 1, 1, 0)
    # q, k, v, an fp32 running result, a bf16 output, LSE, tables: at least their sum
    assert n >= 3 * act + 2 * act + act + B * H * S * 4 + 2 * S * (D // 2) * 4
    assert lib.dit_attention_host_workspace(B, S, H, D, 1, 0, 1, 1, 0) < n  # no running result, no tables
    assert lib.dit_attention_host_workspace(B, S, H, D, 0, 1, 1, 1, 0) == 0
    # stacked partials (one query range at this size): q, k, v, C fp32 parts and their LSEs, two output stages
    m = lib.dit_attention_host_workspace(B, S, H, D, 3, 0, 1, 0, 0)
    assert m >= 3 * act + 3 * 2 * act + 3 * B * H * S * 4 + 2 * (act + B * H * S * 4)


def test_host_workspace_query_ranges(lib):
    """Stacked partials over query ranges: the partial buffers hold one range (at most ceil(S/8) rounded up to
    256 rows plus the ragged last range), not the whole sequence."""
    B, S, H, D, C = 1, 75600, 40, 128, 8
    act = B * S * H * D * 2
    n = lib.dit_attention_host_workspace(B, S, H, D, C, 0, 0, 0, 0)
    whole = 3 * act + C * act  # q, k, v and every chunk's full-length bf16 partial
    assert 3 * act + C * act // 8 < n < whole


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), ops.DIT_ERR_UNSUPPORTED),
    (dict(chunks=0), ops.DIT_ERR_INVALID_ARG),
    (dict(chunks=65), ops.DIT_ERR_INVALID_ARG),
    (dict(prologue=2), ops.DIT_ERR_INVALID_ARG),
    (dict(q=None), ops.DIT_ERR_INVALID_ARG),
    (dict(cos=None), ops.DIT_ERR_INVALID_ARG),
    (dict(ws=A16 * 16 + 128), ops.DIT_ERR_INVALID_ARG),   # workspace not 256-byte aligned
    (dict(wsb=1024), ops.DIT_ERR_INVALID_ARG),            # workspace too small
    (dict(pdt=5), ops.DIT_ERR_INVALID_ARG),
    (dict(merge_update=2), ops.DIT_ERR_INVALID_ARG),
    (dict(merge_update=0, S=2048, chunks=1100, wsb=1 << 40), ops.DIT_ERR_UNSUPPORTED),  # > the merge's part limit
])
def test_host_path_rejects_bad_arguments(lib, kw, code):
    assert _host(lib, **kw) == code
    assert lib.dit_last_error_detail() != b""


def test_host_path_empty_work_is_ok(lib):
    assert _host(lib, B=0) == ops.DIT_OK


def _device_path(lib, **kw):
    B, S, H, D = kw.pop("B", 1), kw.pop("S", 64), kw.pop("H", 2), kw.pop("D", 128)
    chunks, prologue, merge_update = kw.pop("chunks", 2), kw.pop("prologue", 1), kw.pop("merge_update", 1)
    need = lib.dit_attention_workspace(B, S, H, D, chunks, 1, 1, 0)
    a = dict(q=A16, k=A16 * 2, v=A16 * 3, wq=A16 * 4, wk=A16 * 5, cos=A16 * 6, sin=A16 * 7, o=A16 * 8, lse=A16 * 9,
             ws=A16 * 16, wsb=need, pdt=1, odt=0)
    a.update(kw)
    return lib.dit_attention(a["q"], a["k"], a["v"], a["wq"], a["wk"], a["cos"], a["sin"], B, S, H, D, 1e-6, 0.088,
                             chunks, prologue, a["pdt"], merge_update, a["o"], a["odt"], a["lse"], a["ws"], a["wsb"],
                             None, None, None)


def test_device_path_workspace_size(lib):
    B, S, H, D, C = 2, 100, 3, 128, 4
    act, lse = B * S * H * D, B * H * S * 4
    # prologue outputs (bf16 q, k) + an fp32 running result; stacked partials and LSE for the merge kernel
    upd = lib.dit_attention_workspace(B, S, H, D, C, 1, 1, 1)
    assert upd >= 2 * act * 2 + act * 4
    ker = lib.dit_attention_workspace(B, S, H, D, C, 1, 1, 0)
    assert ker >= 2 * act * 2 + C * (act * 4 + lse)
    assert lib.dit_attention_workspace(B, S, H, D, 1, 0, 1, 0) == 0   # one chunk, no prologue: nothing
    assert lib.dit_attention_workspace(B, S, H, D, 1, 1, 1, 0) >= 2 * act * 2
    assert lib.dit_attention_workspace(B, S, H, D, 0, 1, 1, 0) == 0


@pytest.mark.parametrize("kw,code", [
    (dict(D=96), ops.DIT_ERR_UNSUPPORTED),
    (dict(chunks=0), ops.DIT_ERR_INVALID_ARG),
    (dict(chunks=65), ops.DIT_ERR_INVALID_ARG),
    (dict(prologue=2), ops.DIT_ERR_INVALID_ARG),
    (dict(merge_update=2), ops.DIT_ERR_INVALID_ARG),
    (dict(q=None), ops.DIT_ERR_INVALID_ARG),
    (dict(cos=None), ops.DIT_ERR_INVALID_ARG),
    (dict(ws=None), ops.DIT_ERR_INVALID_ARG),
    (dict(ws=A16 * 16 + 128), ops.DIT_ERR_INVALID_ARG),   # workspace not 256-byte aligned
    (dict(wsb=1024), ops.DIT_ERR_INVALID_ARG),            # workspace too small
    (dict(ws=A16 * 8), ops.DIT_ERR_INVALID_ARG),          # workspace overlaps the output
    (dict(pdt=5), ops.DIT_ERR_INVALID_ARG),
    (dict(odt=7), ops.DIT_ERR_INVALID_ARG),
])
def test_device_path_rejects_bad_arguments(lib, kw, code):
    assert _device_path(lib, **kw) == code
    assert lib.dit_last_error_detail() != b""


def test_device_path_empty_work_is_ok(lib):
    assert _device_path(lib, B=0) == ops.DIT_OK
    assert _device_path(lib, S=0, chunks=1) == ops.DIT_OK


def test_device_path_checks_the_merge_before_launching(lib):
    # more stacked partials than the merge kernel takes: refused before anything is launched
    assert _device_path(lib, S=2048, chunks=1100, merge_update=0, wsb=1 << 40) == ops.DIT_ERR_UNSUPPORTED
    assert b"merge" in lib.dit_last_error_detail()
