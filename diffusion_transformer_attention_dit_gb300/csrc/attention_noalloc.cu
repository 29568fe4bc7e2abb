// dit_attention_noalloc: the whole path of dit_attention for callers that
// cannot allocate device memory.
//
// Some callers have no way to get a device workspace: code that runs where
// cudaMalloc is not allowed or not wanted (inside a host callback, under a
// memory budget owned by someone else, in a plugin whose host framework hands
// it only the input and output buffers).  This entry point runs the same
// prologue, chunked attention and merge as dit_attention, with the workspace
// taken from a fixed scratch array that is part of the library itself.
//
//   - The scratch is one file-scope static device array of kScratchBytes
//     (32 MiB).  With the CUDA runtime's default lazy module loading, the array
//     is placed on a device when the first call on that device uses it and it
//     stays reserved until the process exits; with eager loading
//     (CUDA_MODULE_LOADING=EAGER) every device on which the process creates a
//     context reserves it as soon as the library's module is loaded, whether or
//     not this entry point is ever called.  Requests whose workspace would not
//     fit are refused (DIT_ERR_UNSUPPORTED) before anything is launched.
//   - Every call looks the array's device address up again
//     (cudaGetSymbolAddress, with the call's device current), so a context
//     that was torn down and rebuilt (cudaDeviceReset) is never handed a stale
//     address.  The first call on a device may load the library's module
//     there; make that first call before any stream capture.
//   - All calls share the array.  Nothing in it has to start at zero (every
//     byte a call reads, that call has written first), but calls that run at
//     the same time on the GPU -- on different streams, or different host
//     threads -- race on it.
//   - No cudaMalloc, cudaFree or allocating library routine is called.

#include <cuda_runtime.h>

#include "../../include/ditattn.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = size_t(32) << 20;

}  // namespace

static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

namespace {

// Device address of the scratch array on the current device (host code may not
// use the array's name as an address).  Looked up on every call: the lookup is
// cheap once the module is loaded, and a cached address would outlive a reset
// of the device's context.
cudaError_t scratch_address(void **out) {
  void *p = nullptr;
  const cudaError_t e = cudaGetSymbolAddress(&p, g_noalloc_scratch);
  if (e != cudaSuccess) return e;
  *out = p;
  return cudaSuccess;
}

}  // namespace

extern "C" {

dit_status dit_attention_noalloc(const void *q, const void *k, const void *v, const float *wq, const float *wk,
                                 const float *cos_tab, const float *sin_tab, int B, int S, int H, int D, float eps,
                                 float scale, int chunks, int prologue, dit_dtype partial_dtype, int merge_update,
                                 void *o, dit_dtype o_dtype, float *lse, struct CUstream_st *stream) {
  ditattn::set_error_detail("");
  const size_t need = dit_attention_workspace(B, S, H, D, chunks, prologue, partial_dtype, merge_update);
  if (need > kScratchBytes) {
    ditattn::set_error_detail("these sizes need more workspace than the library's 32 MiB static scratch");
    return DIT_ERR_UNSUPPORTED;
  }
  void *ws = nullptr;
  if (need > 0 && (int64_t)B * S * H > 0) {
    const cudaError_t e = scratch_address(&ws);
    if (e != cudaSuccess) {
      ditattn::set_error_detail(cudaGetErrorString(e));
      return DIT_ERR_CUDA;
    }
  }
  // the same path as dit_attention, on the static scratch (its own argument checks apply)
  return dit_attention(q, k, v, wq, wk, cos_tab, sin_tab, B, S, H, D, eps, scale, chunks, prologue, partial_dtype,
                       merge_update, o, o_dtype, lse, ws, ws ? kScratchBytes : 0, nullptr, nullptr, stream);
}

}  // extern "C"
