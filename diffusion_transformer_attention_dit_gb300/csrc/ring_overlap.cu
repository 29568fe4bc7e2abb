// The ring-attention overlap of one rank, on one GPU ("NPU Wan2.2-I2V model
// inference optimisation practice", section "Ring Attention Overlap"): the
// attention over the rank's local key shard runs while the other ranks' shards
// are gathered, then one attention over the gathered keys is LSE-merged into
// the local result (update_out_and_lse, "feat: support Ascend NPU backend
// (torch_npu) for Qwen-Image pipelines - #274", item 2).
//
// On one GPU the all-gather is stood in for by device-to-device copies of the
// remote shards into one contiguous [B, S_remote, H, D] buffer of the
// caller's workspace, issued on a stream the call creates (and releases once
// its work is done), so they run on the copy engines beside the local
// attention on the caller's stream.  The merge is the update form of the
// attention kernel (dit_attn_fwd_update): the gathered keys' result never
// reaches memory, only the merged O and LSE.

#include <cuda_runtime.h>
#include <math.h>

#include "../../include/ditattn.h"
#include "internal.h"

namespace {

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

struct RingWs {
  size_t k, v, acc, total;
};

RingWs ring_plan(int B, int S, int H, int D, int s_remote, dit_dtype partial_dtype) {
  RingWs L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t row = (size_t)H * D;
  L.k = take((size_t)B * s_remote * row * 2);
  L.v = take((size_t)B * s_remote * row * 2);
  L.acc = take((size_t)B * S * row * (partial_dtype == DIT_F32 ? 4 : 2));
  L.total = off;
  return L;
}

dit_status ring_fail(dit_status s, const char *why) {
  ditattn::set_error_detail(why);
  return s;
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// The side stream and events of one call; released when the call returns (the
// runtime defers the release until the work recorded on them has completed).
struct RingResources {
  cudaStream_t side = nullptr;
  cudaEvent_t ready = nullptr, gathered = nullptr;
  ~RingResources() {
    if (ready) cudaEventDestroy(ready);
    if (gathered) cudaEventDestroy(gathered);
    if (side) cudaStreamDestroy(side);
  }
  cudaError_t make() {
    cudaError_t e = cudaStreamCreateWithFlags(&side, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&ready, cudaEventDisableTiming);
    if (e == cudaSuccess) e = cudaEventCreateWithFlags(&gathered, cudaEventDisableTiming);
    return e;
  }
};

}  // namespace

extern "C" {

size_t dit_attention_ring_overlap_workspace(int B, int S, int H, int D, int s_remote, dit_dtype partial_dtype) {
  if (B < 0 || S < 0 || H < 0 || D <= 0 || s_remote < 0) return 0;
  return ring_plan(B, S, H, D, s_remote, partial_dtype).total;
}

dit_status dit_attention_ring_overlap(const void *q, const void *k_local, const void *v_local, int s_local,
                                      const void *const *k_remote, const void *const *v_remote,
                                      const int *s_remote, int R, int B, int S, int H, int D, float scale,
                                      dit_dtype partial_dtype, void *o, dit_dtype o_dtype, float *lse,
                                      void *workspace, size_t workspace_bytes, struct CUstream_st *stream_) {
  ditattn::set_error_detail("");
  if (B < 0 || S < 0 || H < 0 || s_local < 0 || R < 0) return ring_fail(DIT_ERR_INVALID_ARG, "negative size");
  if (D != 64 && D != 128) return ring_fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if ((partial_dtype != DIT_BF16 && partial_dtype != DIT_F32) || (o_dtype != DIT_BF16 && o_dtype != DIT_F32))
    return ring_fail(DIT_ERR_INVALID_ARG, "unknown dtype");
  if (s_local < 1) return ring_fail(DIT_ERR_INVALID_ARG, "the local shard must hold at least one key");
  if (R > 0 && (!k_remote || !v_remote || !s_remote)) return ring_fail(DIT_ERR_INVALID_ARG, "null remote arrays");
  int64_t s_rt = 0;
  for (int r = 0; r < R; ++r) {
    if (s_remote[r] < 1) return ring_fail(DIT_ERR_INVALID_ARG, "every remote shard must hold at least one key");
    if (!k_remote[r] || !v_remote[r]) return ring_fail(DIT_ERR_INVALID_ARG, "null remote shard");
    if (!aligned16(k_remote[r]) || !aligned16(v_remote[r]))
      return ring_fail(DIT_ERR_INVALID_ARG, "remote shard misaligned");
    s_rt += s_remote[r];
  }
  if (s_rt > (int64_t)1 << 30) return ring_fail(DIT_ERR_INVALID_ARG, "remote shards too long");
  if ((int64_t)B * S * H == 0) return DIT_OK;
  if (!(scale > 0.f) || isinf(scale)) return ring_fail(DIT_ERR_INVALID_ARG, "scale must be finite and > 0");
  // the checks the attention launches would make, before any copy is queued
  if (!q || !k_local || !v_local || !o || !lse) return ring_fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (!aligned16(q) || !aligned16(k_local) || !aligned16(v_local) || !aligned16(o) ||
      (reinterpret_cast<uintptr_t>(lse) & 3))
    return ring_fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  {
    const size_t act = (size_t)B * S * H * D, osz = o_dtype == DIT_F32 ? 4 : 2;
    const uintptr_t o0 = reinterpret_cast<uintptr_t>(o), o1 = o0 + act * osz;
    const uintptr_t l0 = reinterpret_cast<uintptr_t>(lse), l1 = l0 + (size_t)B * H * S * 4;
    auto hits = [&](const void *p, size_t bytes) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = a + bytes;
      return (a < o1 && o0 < b) || (a < l1 && l0 < b);
    };
    if ((o0 < l1 && l0 < o1) || hits(q, act * 2) || hits(k_local, (size_t)B * s_local * H * D * 2) ||
        hits(v_local, (size_t)B * s_local * H * D * 2))
      return ring_fail(DIT_ERR_INVALID_ARG, "outputs overlap inputs or each other");
    for (int r = 0; r < R; ++r) {
      const size_t shard = (size_t)B * s_remote[r] * H * D * 2;
      if (hits(k_remote[r], shard) || hits(v_remote[r], shard))
        return ring_fail(DIT_ERR_INVALID_ARG, "outputs overlap a remote shard");
    }
  }
  const RingWs L = ring_plan(B, S, H, D, (int)s_rt, partial_dtype);
  if (R > 0) {
    if (!workspace) return ring_fail(DIT_ERR_INVALID_ARG, "null workspace");
    if (reinterpret_cast<uintptr_t>(workspace) % 256) return ring_fail(DIT_ERR_INVALID_ARG, "workspace misaligned");
    if (workspace_bytes < L.total) return ring_fail(DIT_ERR_INVALID_ARG, "workspace too small");
    // the workspace must not overlap an input or output (the kernels check their own arguments)
    const uintptr_t w0 = reinterpret_cast<uintptr_t>(workspace), w1 = w0 + L.total;
    const size_t act = (size_t)B * S * H * D;
    auto inside = [&](const void *p, size_t bytes) {
      const uintptr_t a = reinterpret_cast<uintptr_t>(p);
      return a < w1 && w0 < a + bytes;
    };
    if (inside(q, act * 2) || inside(o, act * (o_dtype == DIT_F32 ? 4 : 2)) || inside(lse, (size_t)B * H * S * 4) ||
        inside(k_local, (size_t)B * s_local * H * D * 2) || inside(v_local, (size_t)B * s_local * H * D * 2))
      return ring_fail(DIT_ERR_INVALID_ARG, "workspace overlaps an input or output");
    for (int r = 0; r < R; ++r)
      if (inside(k_remote[r], (size_t)B * s_remote[r] * H * D * 2) ||
          inside(v_remote[r], (size_t)B * s_remote[r] * H * D * 2))
        return ring_fail(DIT_ERR_INVALID_ARG, "workspace overlaps a remote shard");
  }
  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int64_t st_q[3] = {(int64_t)S * H * D, (int64_t)H * D, D};
  const int64_t st_l[3] = {(int64_t)s_local * H * D, (int64_t)H * D, D};
  if (R == 0)  // a ring of one rank: the attention over the local shard is the result
    return ditattn::attn_checked(q, k_local, v_local, B, H, S, s_local, D, st_q, st_l, scale, 0, s_local, false, o,
                                 o_dtype, st_q, lse, nullptr, DIT_BF16, nullptr, nullptr, -1, stream);

  RingResources res;
  cudaError_t e = res.make();
  if (e != cudaSuccess) return ring_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  char *ws = static_cast<char *>(workspace);
  // gather: the remote shards are the caller's earlier work on `stream`
  e = cudaEventRecord(res.ready, stream);
  if (e == cudaSuccess) e = cudaStreamWaitEvent(res.side, res.ready, 0);
  const size_t row = (size_t)H * D * 2;
  int64_t off = 0;
  for (int r = 0; r < R && e == cudaSuccess; ++r) {
    const size_t w = (size_t)s_remote[r] * row;
    e = cudaMemcpy2DAsync(ws + L.k + off * row, (size_t)s_rt * row, k_remote[r], w, w, B, cudaMemcpyDeviceToDevice,
                          res.side);
    if (e == cudaSuccess)
      e = cudaMemcpy2DAsync(ws + L.v + off * row, (size_t)s_rt * row, v_remote[r], w, w, B,
                            cudaMemcpyDeviceToDevice, res.side);
    off += s_remote[r];
  }
  if (e == cudaSuccess) e = cudaEventRecord(res.gathered, res.side);
  if (e != cudaSuccess) return ring_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  // the local shard, meanwhile, into the running result (acc, lse)
  dit_status st = ditattn::attn_checked(q, k_local, v_local, B, H, S, s_local, D, st_q, st_l, scale, 0, s_local, false,
                                        ws + L.acc, partial_dtype, st_q, lse, nullptr, DIT_BF16, nullptr, nullptr, -1,
                                        stream);
  if (st != DIT_OK) return st;
  // then the gathered shards, merged into it in the attention's epilogue
  e = cudaStreamWaitEvent(stream, res.gathered, 0);
  if (e != cudaSuccess) return ring_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  const int64_t st_r[3] = {(int64_t)s_rt * H * D, (int64_t)H * D, D};
  return ditattn::attn_checked(q, ws + L.k, ws + L.v, B, H, S, (int)s_rt, D, st_q, st_r, scale, 0, (int)s_rt, false,
                               o, o_dtype, st_q, lse, ws + L.acc, partial_dtype, st_q, lse, -1, stream);
}

}  // extern "C"
