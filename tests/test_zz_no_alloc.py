"""dit_attention_noalloc: the whole attention path for callers that cannot
allocate device memory (a host callback, a plugin handed only its input and
output buffers, a process whose device memory belongs to someone else).  It
runs on a 32 MiB scratch array built into the library, so it is checked here
against dit_attention, which takes a caller-provided workspace.  This file is
collected last on purpose: it exercises the library's one shared scratch."""

import pytest
import torch

from diffusion_transformer_attention_dit_gb300 import build, inputs, ops
from parity import check_lse, check_o, dev_bf16, dev_f32, host_f64


@pytest.fixture(scope="module")
def lib():
    build.build()
    return ops.load_library()


def _noalloc(lib, q, k, v, tabs, o, lse, chunks, merge, partial_dtype, prologue):
    B, S, H, D = q.shape
    return lib.dit_attention_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), *(t.data_ptr() for t in tabs), B, S,
                                     H, D, 1e-6, D ** -0.5, chunks, int(prologue), ops._dtype_code(partial_dtype),
                                     int(merge == "update"), o.data_ptr(), ops._dtype_code(o.dtype), lse.data_ptr(),
                                     torch.cuda.current_stream().cuda_stream)


# (seed, chunks, merge, partial dtype, prologue): running result in fp32; stacked bf16 partials; one chunk without
# the prologue (no workspace at all: the scratch is not even looked up); stacked fp32 partials
CALLS = ((21, 2, "update", torch.float32, True), (22, 3, "kernel", torch.bfloat16, True),
         (23, 1, "kernel", torch.float32, False), (24, 4, "kernel", torch.float32, True))


@pytest.mark.gpu
def test_noalloc_matches_dit_attention_on_calls_in_a_row(lib):
    """Calls in a row share the scratch (each finds another layout left in it): each matches the entry point that
    takes a workspace, within the parity tolerances.  The first call on a device may bring the scratch in (the
    CUDA runtime loads a library's device data on first use); every later call changes the device's free memory
    by nothing."""
    B, S, H, D = 1, 1000, 4, 128
    for call, (seed, chunks, merge, pdt, prologue) in enumerate(CALLS):
        q, k, v, wq, wk, cos, sin = inputs.small_case(B, S, H, D, seed=seed)
        tq, tk, tv = dev_bf16(q), dev_bf16(k), dev_bf16(v)
        tabs = [dev_f32(t) for t in (wq, wk, cos, sin)]
        ref_o, ref_lse = ops.dit_attention(tq, tk, tv, *tabs, eps=1e-6, chunks=chunks, partial_dtype=pdt,
                                           merge=merge, prologue=prologue)
        o = torch.empty((B, S, H, D), dtype=torch.bfloat16, device="cuda")
        lse = torch.empty((B, H, S), dtype=torch.float32, device="cuda")
        torch.cuda.synchronize()
        free_before = torch.cuda.mem_get_info()[0]
        status = _noalloc(lib, tq, tk, tv, tabs, o, lse, chunks, merge, pdt, prologue)
        assert status == ops.DIT_OK, lib.dit_last_error_detail()
        torch.cuda.synchronize()
        if call > 0:
            assert torch.cuda.mem_get_info()[0] == free_before
        ops.poll_device_error()
        what = f"no-alloc path, {merge} merge, {chunks} chunks, prologue {prologue}"
        check_o(host_f64(o), host_f64(ref_o), what=what)
        check_lse(host_f64(lse), host_f64(ref_lse), what=what)


def test_noalloc_refuses_sizes_beyond_its_scratch(lib):
    """A request whose workspace would exceed the 32 MiB scratch is refused before anything is launched (no GPU
    needed: the size check comes first)."""
    A16 = 1 << 20  # fake, aligned device addresses: never dereferenced
    B, S, H, D = 1, 4312, 24, 128  # q' and k' alone take 53 MB
    status = lib.dit_attention_noalloc(A16, 2 * A16, 3 * A16, 4 * A16, 5 * A16, 6 * A16, 7 * A16, B, S, H, D, 1e-6,
                                       D ** -0.5, 2, 1, ops.DIT_F32, 1, 8 * A16, ops.DIT_BF16, 9 * A16, None)
    assert status == ops.DIT_ERR_UNSUPPORTED
    assert b"32 MiB" in lib.dit_last_error_detail()
