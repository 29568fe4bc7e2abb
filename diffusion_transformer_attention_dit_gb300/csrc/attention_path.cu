// The whole hot path on device buffers (dit_attention): QK-RMSNorm + RoPE, the
// attention over KV chunks and their LSE merge, as one call; and the chunk
// sequence it shares with the host-buffer path (dit_attention_host).
//
// Chunk c (c >= 1) is launched with the deferred dependency wait: it reads only
// q, k, v -- complete before chunk 0 started -- until its epilogue, so its CTAs
// fill the SMs the previous chunk's last wave leaves idle and wait for that
// chunk only where they need its results (see attn_fwd.cu).  The launches still
// complete in stream order.

#include <cuda_runtime.h>

#include "../../include/ditattn.h"
#include "internal.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct DeviceWs {
  size_t qn, kn, acc, lse_parts, total;
};

DeviceWs plan(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype, int merge_update) {
  DeviceWs L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t elems = (size_t)B * S * H * D, psize = partial_dtype == DIT_F32 ? 4 : 2;
  if (prologue) {
    L.qn = take(elems * 2);
    L.kn = take(elems * 2);
  }
  if (chunks > 1) {
    if (merge_update) {
      L.acc = take(elems * psize);
    } else {
      L.acc = take(elems * psize * chunks);
      L.lse_parts = take((size_t)B * H * S * 4 * chunks);
    }
  }
  L.total = off;
  return L;
}

dit_status fail(dit_status s, const char *why) {
  ditattn::set_error_detail(why);
  return s;
}

}  // namespace

dit_status ditattn::run_attention_chunks(const void *q, const void *k, const void *v, int B, int S, int H, int D,
                                         float scale, int chunks, dit_dtype partial_dtype, bool merge_update,
                                         void *acc, float *lse_parts, void *o, dit_dtype o_dtype, float *lse,
                                         cudaEvent_t attn_begin, cudaEvent_t attn_end,
                                         cudaError_t (*before_chunk)(void *ctx, int c), void *ctx,
                                         cudaStream_t stream) {
  const int64_t st[3] = {(int64_t)S * H * D, (int64_t)H * D, D};
  const int64_t part_o = (int64_t)B * S * H * D, part_l = (int64_t)B * H * S;
  const size_t psize = partial_dtype == DIT_F32 ? 4 : 2;
  cudaError_t e = attn_begin ? cudaEventRecord(attn_begin, stream) : cudaSuccess;
  if (e != cudaSuccess) return fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  for (int c = 0; c < chunks; ++c) {
    const int lo = (int)((int64_t)c * S / chunks), hi = (int)((int64_t)(c + 1) * S / chunks);
    if (before_chunk && (e = before_chunk(ctx, c)) != cudaSuccess) return fail(DIT_ERR_CUDA, cudaGetErrorString(e));
    const bool last = c == chunks - 1;
    dit_status r;
    if (chunks == 1) {
      r = attn_checked(q, k, v, B, H, S, S, D, st, st, scale, lo, hi, false, o, o_dtype, st, lse, nullptr, DIT_BF16,
                       nullptr, nullptr, -1, stream);
    } else if (merge_update) {
      if (c == 0)
        r = attn_checked(q, k, v, B, H, S, S, D, st, st, scale, lo, hi, false, acc, partial_dtype, st, lse, nullptr,
                         DIT_BF16, nullptr, nullptr, c, stream);
      else
        r = attn_checked(q, k, v, B, H, S, S, D, st, st, scale, lo, hi, false, last ? o : acc,
                         last ? o_dtype : partial_dtype, st, lse, acc, partial_dtype, st, lse, c, stream);
    } else {
      r = attn_checked(q, k, v, B, H, S, S, D, st, st, scale, lo, hi, false,
                       static_cast<char *>(acc) + (size_t)c * part_o * psize, partial_dtype, st,
                       lse_parts + (size_t)c * part_l, nullptr, DIT_BF16, nullptr, nullptr, c, stream);
    }
    if (r != DIT_OK) return r;  // the entry point has set the detail
  }
  e = attn_end ? cudaEventRecord(attn_end, stream) : cudaSuccess;
  if (e != cudaSuccess) return fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  if (chunks > 1 && !merge_update)
    return dit_attn_merge_lse(acc, partial_dtype, lse_parts, chunks, B, H, S, D, part_o, part_l, o, o_dtype, lse,
                              reinterpret_cast<struct CUstream_st *>(stream));
  return DIT_OK;
}

extern "C" {

size_t dit_attention_workspace(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype,
                               int merge_update) {
  if (B < 0 || S < 0 || H < 0 || D <= 0 || chunks < 1) return 0;
  return plan(B, S, H, D, chunks, prologue != 0, partial_dtype, merge_update != 0).total;
}

dit_status dit_attention(const void *q, const void *k, const void *v, const float *wq, const float *wk,
                         const float *cos_tab, const float *sin_tab, int B, int S, int H, int D, float eps, float scale,
                         int chunks, int prologue, dit_dtype partial_dtype, int merge_update, void *o,
                         dit_dtype o_dtype, float *lse, void *workspace, size_t workspace_bytes,
                         struct CUevent_st *attn_begin, struct CUevent_st *attn_end, struct CUstream_st *stream) {
  ditattn::set_error_detail("");
  if (B < 0 || S < 0 || H < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (D != 64 && D != 128) return fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (prologue != 0 && prologue != 1) return fail(DIT_ERR_INVALID_ARG, "prologue must be 0 or 1");
  if (merge_update != 0 && merge_update != 1) return fail(DIT_ERR_INVALID_ARG, "merge_update must be 0 or 1");
  if ((partial_dtype != DIT_BF16 && partial_dtype != DIT_F32) || (o_dtype != DIT_BF16 && o_dtype != DIT_F32))
    return fail(DIT_ERR_INVALID_ARG, "unknown dtype");
  if ((int64_t)B * S * H == 0) return DIT_OK;
  if (chunks < 1 || chunks > S) return fail(DIT_ERR_INVALID_ARG, "chunks must satisfy 1 <= chunks <= S");
  if (chunks > 1 && !merge_update && !ditattn::merge_fits(chunks, H))
    return fail(DIT_ERR_UNSUPPORTED, "chunks * H too large for the merge kernel");
  if (!q || !k || !v || !o || !lse) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (prologue && (!wq || !wk || !cos_tab || !sin_tab)) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  const DeviceWs L = plan(B, S, H, D, chunks, prologue, partial_dtype, merge_update);
  if (L.total > 0 && !workspace) return fail(DIT_ERR_INVALID_ARG, "null workspace");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return fail(DIT_ERR_INVALID_ARG, "workspace misaligned");
  if (workspace_bytes < L.total) return fail(DIT_ERR_INVALID_ARG, "workspace too small");
  const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + L.total;
  const size_t act = (size_t)B * S * H * D;
  auto inside = [&](const void *p, size_t bytes) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p);
    return L.total > 0 && a < w1 && w0 < a + bytes;
  };
  if (inside(q, act * 2) || inside(k, act * 2) || inside(v, act * 2) || inside(o, act * (o_dtype == DIT_F32 ? 4 : 2)) ||
      inside(lse, (size_t)B * H * S * 4))
    return fail(DIT_ERR_INVALID_ARG, "workspace overlaps an input or output");
  char *ws = static_cast<char *>(workspace);
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  const void *aq = q, *ak = k;
  if (prologue) {
    dit_status r = dit_qk_norm_rope(q, k, ws + L.qn, ws + L.kn, wq, wk, cos_tab, sin_tab, B, S, H, D, eps, stream);
    if (r != DIT_OK) return r;
    aq = ws + L.qn;
    ak = ws + L.kn;
  }
  return ditattn::run_attention_chunks(aq, ak, v, B, S, H, D, scale, chunks, partial_dtype, merge_update != 0,
                                       chunks > 1 ? ws + L.acc : nullptr,
                                       chunks > 1 && !merge_update ? reinterpret_cast<float *>(ws + L.lse_parts)
                                                                   : nullptr,
                                       o, o_dtype, lse, reinterpret_cast<cudaEvent_t>(attn_begin),
                                       reinterpret_cast<cudaEvent_t>(attn_end), nullptr, nullptr, s);
}

}  // extern "C"
