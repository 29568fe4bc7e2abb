// The whole hot path from host buffers: the inputs are copied to a caller-owned
// device workspace, the prologue, the chunked attention and the LSE merge run
// there, and O / LSE are copied back -- with the copies pipelined against the
// kernels.
//
// Order of work (copy stream = an internal non-blocking stream per device):
//   copy stream:  q, k (+ weights, rotary tables) | v rows of chunk 0 | v rows of chunk 1 | ...
//   caller stream:            prologue (waits q, k) | attention chunk 0 (waits its v rows) |
//                             chunk 1 in the update form (waits its v rows) | ... | O, LSE to the host
// so the value rows of later chunks travel while earlier chunks compute.  The
// attention kernels are the ones behind dit_attn_fwd / dit_attn_fwd_update, in
// the chunk sequence dit_attention uses (attention_path.cu), and the prologue is
// dit_qk_norm_rope; chunk c covers keys [c*S/C, (c+1)*S/C).

#include <cuda_runtime.h>

#include <mutex>
#include <vector>

#include "../../include/ditattn.h"
#include "internal.h"

namespace {

struct WsLayout {
  size_t q, k, v, wq, wk, cs, sn, acc, o, lse, total;
};

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

WsLayout plan(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype, dit_dtype o_dtype) {
  WsLayout L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t elems = (size_t)B * S * H * D;
  L.q = take(elems * 2);
  L.k = take(elems * 2);
  L.v = take(elems * 2);
  if (prologue) {
    L.wq = take((size_t)D * 4);
    L.wk = take((size_t)D * 4);
    L.cs = take((size_t)S * (D / 2) * 4);
    L.sn = take((size_t)S * (D / 2) * 4);
  }
  if (chunks > 1) L.acc = take(elems * (partial_dtype == DIT_F32 ? 4 : 2));
  L.o = take(elems * (o_dtype == DIT_F32 ? 4 : 2));
  L.lse = take((size_t)B * H * S * 4);
  L.total = off;
  return L;
}

std::mutex g_streams_mu;
cudaStream_t g_copy_streams[64] = {};

cudaError_t copy_stream(cudaStream_t *out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lock(g_streams_mu);
  if (!g_copy_streams[dev]) {
    e = cudaStreamCreateWithFlags(&g_copy_streams[dev], cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
  }
  *out = g_copy_streams[dev];
  return cudaSuccess;
}

dit_status host_fail(dit_status s, const char *why) {
  ditattn::set_error_detail(why);
  return s;
}

// Events of one call; destroyed when the call returns (destruction is deferred
// by the runtime until recorded work completes).
struct Events {
  std::vector<cudaEvent_t> ev;
  ~Events() {
    for (cudaEvent_t e : ev) cudaEventDestroy(e);
  }
  cudaError_t make(size_t n) {
    ev.assign(n, nullptr);
    for (size_t i = 0; i < n; ++i) {
      cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
      if (e != cudaSuccess) return e;
    }
    return cudaSuccess;
  }
};

}  // namespace

extern "C" {

size_t dit_attention_host_workspace(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype,
                                    dit_dtype o_dtype) {
  if (B < 0 || S < 0 || H < 0 || D <= 0 || chunks < 1) return 0;
  return plan(B, S, H, D, chunks, prologue, partial_dtype, o_dtype).total;
}

dit_status dit_attention_host(const void *q, const void *k, const void *v, const float *wq, const float *wk,
                              const float *cos_tab, const float *sin_tab, int B, int S, int H, int D, float eps,
                              float scale, int chunks, int prologue, dit_dtype partial_dtype, void *o,
                              dit_dtype o_dtype, float *lse, void *workspace, size_t workspace_bytes,
                              struct CUstream_st *stream_) {
  ditattn::set_error_detail("");
  if (B < 0 || S < 0 || H < 0) return host_fail(DIT_ERR_INVALID_ARG, "negative size");
  if (D != 64 && D != 128) return host_fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (prologue != 0 && prologue != 1) return host_fail(DIT_ERR_INVALID_ARG, "prologue must be 0 or 1");
  if ((partial_dtype != DIT_BF16 && partial_dtype != DIT_F32) || (o_dtype != DIT_BF16 && o_dtype != DIT_F32))
    return host_fail(DIT_ERR_INVALID_ARG, "unknown dtype");
  if ((int64_t)B * S * H == 0) return DIT_OK;
  if (chunks < 1 || chunks > S) return host_fail(DIT_ERR_INVALID_ARG, "chunks must satisfy 1 <= chunks <= S");
  if (!q || !k || !v || !o || !lse || !workspace) return host_fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (prologue && (!wq || !wk || !cos_tab || !sin_tab)) return host_fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return host_fail(DIT_ERR_INVALID_ARG, "workspace misaligned");
  const WsLayout L = plan(B, S, H, D, chunks, prologue, partial_dtype, o_dtype);
  if (workspace_bytes < L.total) return host_fail(DIT_ERR_INVALID_ARG, "workspace too small");

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  cudaStream_t cs = nullptr;
  cudaError_t e = copy_stream(&cs);
  Events evs;
  // [0] entry, [1] q/k (and tables) resident, [2 + c] value rows of chunk c resident
  if (e == cudaSuccess) e = evs.make(2 + (size_t)chunks);
  if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  char *ws = static_cast<char *>(workspace);
  const size_t act = (size_t)B * S * H * D * 2, row = (size_t)H * D * 2;  // bytes of q and of one (b, s) row
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };

  // the workspace may still be in use by earlier work on the caller's stream
  ok(cudaEventRecord(evs.ev[0], stream)) && ok(cudaStreamWaitEvent(cs, evs.ev[0], 0));
  ok(cudaMemcpyAsync(ws + L.q, q, act, cudaMemcpyHostToDevice, cs)) &&
      ok(cudaMemcpyAsync(ws + L.k, k, act, cudaMemcpyHostToDevice, cs));
  if (prologue) {
    const size_t tab = (size_t)S * (D / 2) * 4;
    ok(cudaMemcpyAsync(ws + L.wq, wq, (size_t)D * 4, cudaMemcpyHostToDevice, cs)) &&
        ok(cudaMemcpyAsync(ws + L.wk, wk, (size_t)D * 4, cudaMemcpyHostToDevice, cs)) &&
        ok(cudaMemcpyAsync(ws + L.cs, cos_tab, tab, cudaMemcpyHostToDevice, cs)) &&
        ok(cudaMemcpyAsync(ws + L.sn, sin_tab, tab, cudaMemcpyHostToDevice, cs));
  }
  ok(cudaEventRecord(evs.ev[1], cs));
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int lo = (int)((int64_t)c * S / chunks), hi = (int)((int64_t)(c + 1) * S / chunks);
    // rows [lo, hi) of every batch entry: B runs of (hi - lo) * H * D elements, S * H * D apart
    ok(cudaMemcpy2DAsync(ws + L.v + lo * row, (size_t)S * row, static_cast<const char *>(v) + lo * row,
                         (size_t)S * row, (size_t)(hi - lo) * row, B, cudaMemcpyHostToDevice, cs)) &&
        ok(cudaEventRecord(evs.ev[2 + c], cs));
  }
  if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));

  if (!ok(cudaStreamWaitEvent(stream, evs.ev[1], 0))) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  void *dq = ws + L.q, *dk = ws + L.k, *dv = ws + L.v;
  dit_status st = DIT_OK;
  if (prologue)
    st = dit_qk_norm_rope(dq, dk, dq, dk, reinterpret_cast<const float *>(ws + L.wq),
                          reinterpret_cast<const float *>(ws + L.wk), reinterpret_cast<const float *>(ws + L.cs),
                          reinterpret_cast<const float *>(ws + L.sn), B, S, H, D, eps, stream_);
  if (st != DIT_OK) return st;  // the entry point has set the detail
  float *dlse = reinterpret_cast<float *>(ws + L.lse);
  // chunk c waits only for its own value rows (copy event 2 + c)
  struct Ctx {
    cudaStream_t stream;
    cudaEvent_t *ev;
  } ctx = {stream, evs.ev.data()};
  auto before_chunk = [](void *p, int c) -> cudaError_t {
    const Ctx *x = static_cast<const Ctx *>(p);
    return cudaStreamWaitEvent(x->stream, x->ev[2 + c], 0);
  };
  st = ditattn::run_attention_chunks(dq, dk, dv, B, S, H, D, scale, chunks, partial_dtype, true,
                                     chunks > 1 ? ws + L.acc : nullptr, nullptr, ws + L.o, o_dtype, dlse, nullptr,
                                     nullptr, before_chunk, &ctx, stream);
  if (st != DIT_OK) return st;
  const size_t o_bytes = (size_t)B * S * H * D * (o_dtype == DIT_F32 ? 4 : 2);
  ok(cudaMemcpyAsync(o, ws + L.o, o_bytes, cudaMemcpyDeviceToHost, stream)) &&
      ok(cudaMemcpyAsync(lse, dlse, (size_t)B * H * S * 4, cudaMemcpyDeviceToHost, stream));
  if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  return DIT_OK;
}

}  // extern "C"
