// The whole hot path from host buffers: the inputs are copied to a caller-owned
// device workspace, the prologue, the chunked attention and the LSE merge run
// there, and O / LSE are copied back -- with the copies pipelined against the
// kernels.  Three streams take part: an input-copy stream and an output-copy
// stream (created for the call and released when its work is done) and the
// caller's stream, on which the kernels run.
//
// Running form (merge_update = 1, more than one chunk): the inputs go in the
// order q, k (tables) | v rows of chunk 0 | v rows of chunk 1 | ... (without the
// prologue the key rows travel with their chunk's value rows); the prologue
// waits for q and k, chunk c for its own rows, and chunk c >= 1 is merged into
// the running result in its epilogue (dit_attn_fwd_update).  O and LSE go back
// at the end.
//
// Query-range form (merge_update = 0, or a single chunk): the query rows are
// processed in R ranges (large problems: six, of 3/8 down to 1/16 of the rows)
// whose edges are multiples of 256 rows (one attention CTA's rows), so each
// range runs exactly the tiles the one-call device path runs and gives
// bit-identical results.  For range r: every KV chunk's
// attention over the range's rows into stacked partials, the merge kernel into
// one of two output staging buffers, and -- on the output-copy stream -- the
// copy of that range's O and LSE to the host, which overlaps the next range's
// kernels.  Inputs: q rows of range 0 | k, v rows of chunk 0 | ... | q rows of
// range 1 | ... (with the prologue, q and k in full first), so the first
// attention starts after one range of queries and one chunk of keys.
//
// The attention kernels are the ones behind dit_attn_fwd / dit_attn_fwd_update,
// the merge is dit_attn_merge_lse and the prologue dit_qk_norm_rope; chunk c
// covers keys [c*S/C, (c+1)*S/C).

#include <cuda_runtime.h>

#include <algorithm>
#include <vector>

#include "../../include/ditattn.h"
#include "internal.h"

namespace {

constexpr int kRangeRows = 256;        // query rows of one attention CTA: range edges are multiples of this
constexpr int kMaxRanges = 8;
constexpr int64_t kMinRangeCtas = 608;  // at least four waves of a 152-SM GB300 in each range's launches

size_t align256(size_t x) { return (x + 255) & ~size_t(255); }

bool range_form(int chunks, int merge_update) { return chunks == 1 || merge_update == 0; }

// Tapered ranges, for problems large enough that a sixteenth of the rows still
// makes kMinRangeCtas CTAs: six ranges ending at 6, 10, 12, 14, 15 and 16
// sixteenths of the rows.  The first range's attention (3/8 of the work) then
// outlasts the copy of every chunk's keys and values even over a host link
// shared with other work (it needs all of them), and the last range, whose
// output copy is the one left exposed, is 1/16 of the rows.
constexpr int kTaperRanges = 6;
constexpr int kTaperEnd[kTaperRanges] = {6, 10, 12, 14, 15, 16};

bool tapered(int B, int S, int H) { return (int64_t)B * H * (S / 16 / kRangeRows) >= kMinRangeCtas; }

// Number of query ranges: the tapered six, or as many equal ranges as keep every
// range's launches at least kMinRangeCtas CTAs, at most kMaxRanges.
int query_ranges(int B, int S, int H) {
  if (tapered(B, S, H)) return kTaperRanges;
  const int64_t bh = std::max<int64_t>(1, (int64_t)B * H);
  const int64_t rows_min = (kMinRangeCtas + bh - 1) / bh * kRangeRows;
  return (int)std::max<int64_t>(1, std::min<int64_t>(kMaxRanges, S / rows_min));
}

// First row of range r of the R = query_ranges(B, S, H) ranges over S rows
// (edges rounded down to kRangeRows).
int range_edge(int r, int R, int B, int S, int H) {
  if (r <= 0) return 0;
  if (r >= R) return S;
  if (tapered(B, S, H)) return (int)((int64_t)S * kTaperEnd[r - 1] / 16 / kRangeRows * kRangeRows);
  return (int)((int64_t)r * S / R / kRangeRows * kRangeRows);
}

int max_range_rows(int R, int B, int S, int H) {
  int m = 0;
  for (int r = 0; r < R; ++r) m = std::max(m, range_edge(r + 1, R, B, S, H) - range_edge(r, R, B, S, H));
  return m;
}

struct WsLayout {
  size_t q, k, v, wq, wk, cs, sn;
  size_t acc, o, lse;              // running form
  size_t parts, lse_parts, ob[2], lb[2];  // query-range form
  int ranges, range_rows;
  size_t total;
};

WsLayout plan(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype, int merge_update,
              dit_dtype o_dtype) {
  WsLayout L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    const size_t at = off;
    off = align256(off + bytes);
    return at;
  };
  const size_t elems = (size_t)B * S * H * D, psize = partial_dtype == DIT_F32 ? 4 : 2,
               osize = o_dtype == DIT_F32 ? 4 : 2;
  L.q = take(elems * 2);
  L.k = take(elems * 2);
  L.v = take(elems * 2);
  if (prologue) {
    L.wq = take((size_t)D * 4);
    L.wk = take((size_t)D * 4);
    L.cs = take((size_t)S * (D / 2) * 4);
    L.sn = take((size_t)S * (D / 2) * 4);
  }
  if (range_form(chunks, merge_update)) {
    L.ranges = query_ranges(B, S, H);
    L.range_rows = max_range_rows(L.ranges, B, S, H);
    const size_t relems = (size_t)B * L.range_rows * H * D, rlse = (size_t)B * H * L.range_rows * 4;
    if (chunks > 1) {
      L.parts = take(relems * psize * chunks);
      L.lse_parts = take(rlse * chunks);
    }
    for (int i = 0; i < 2; ++i) {
      L.ob[i] = take(relems * osize);
      L.lb[i] = take(rlse);
    }
  } else {
    L.acc = take(elems * psize);
    L.o = take(elems * osize);
    L.lse = take((size_t)B * H * S * 4);
  }
  L.total = off;
  return L;
}

dit_status host_fail(dit_status s, const char *why) {
  ditattn::set_error_detail(why);
  return s;
}

// Streams and events of one call; released when the call returns (the runtime
// defers the release until the work recorded on them has completed).
struct CallResources {
  cudaStream_t in = nullptr, out = nullptr;
  std::vector<cudaEvent_t> ev;
  ~CallResources() {
    for (cudaEvent_t e : ev)
      if (e) cudaEventDestroy(e);
    if (in) cudaStreamDestroy(in);
    if (out) cudaStreamDestroy(out);
  }
  cudaError_t make(size_t n_events) {
    cudaError_t e = cudaStreamCreateWithFlags(&in, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&out, cudaStreamNonBlocking);
    if (e != cudaSuccess) return e;
    ev.assign(n_events, nullptr);
    for (size_t i = 0; i < n_events; ++i)
      if ((e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming)) != cudaSuccess) return e;
    return cudaSuccess;
  }
};

// Rows [lo, hi) of every batch entry of a [B, S, H, D] bf16 tensor (B runs of
// (hi - lo) rows, S rows apart), host to device at the same offsets.
cudaError_t copy_rows_in(char *dst, const void *src, int B, int S, size_t row, int lo, int hi, cudaStream_t s) {
  if (hi <= lo) return cudaSuccess;
  return cudaMemcpy2DAsync(dst + lo * row, (size_t)S * row, static_cast<const char *>(src) + lo * row,
                           (size_t)S * row, (size_t)(hi - lo) * row, B, cudaMemcpyHostToDevice, s);
}

}  // namespace

extern "C" {

size_t dit_attention_host_workspace(int B, int S, int H, int D, int chunks, int prologue, dit_dtype partial_dtype,
                                    int merge_update, dit_dtype o_dtype) {
  if (B < 0 || S < 0 || H < 0 || D <= 0 || chunks < 1) return 0;
  return plan(B, S, H, D, chunks, prologue != 0, partial_dtype, merge_update != 0, o_dtype).total;
}

dit_status dit_attention_host(const void *q, const void *k, const void *v, const float *wq, const float *wk,
                              const float *cos_tab, const float *sin_tab, int B, int S, int H, int D, float eps,
                              float scale, int chunks, int prologue, dit_dtype partial_dtype, int merge_update,
                              void *o, dit_dtype o_dtype, float *lse, void *workspace, size_t workspace_bytes,
                              struct CUstream_st *stream_) {
  ditattn::set_error_detail("");
  if (B < 0 || S < 0 || H < 0) return host_fail(DIT_ERR_INVALID_ARG, "negative size");
  if (D != 64 && D != 128) return host_fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (prologue != 0 && prologue != 1) return host_fail(DIT_ERR_INVALID_ARG, "prologue must be 0 or 1");
  if (merge_update != 0 && merge_update != 1) return host_fail(DIT_ERR_INVALID_ARG, "merge_update must be 0 or 1");
  if ((partial_dtype != DIT_BF16 && partial_dtype != DIT_F32) || (o_dtype != DIT_BF16 && o_dtype != DIT_F32))
    return host_fail(DIT_ERR_INVALID_ARG, "unknown dtype");
  if ((int64_t)B * S * H == 0) return DIT_OK;
  if (chunks < 1 || chunks > S) return host_fail(DIT_ERR_INVALID_ARG, "chunks must satisfy 1 <= chunks <= S");
  if (!q || !k || !v || !o || !lse || !workspace) return host_fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (prologue && (!wq || !wk || !cos_tab || !sin_tab)) return host_fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (reinterpret_cast<uintptr_t>(workspace) % 256) return host_fail(DIT_ERR_INVALID_ARG, "workspace misaligned");
  const WsLayout L = plan(B, S, H, D, chunks, prologue, partial_dtype, merge_update, o_dtype);
  if (workspace_bytes < L.total) return host_fail(DIT_ERR_INVALID_ARG, "workspace too small");
  const bool ranged = range_form(chunks, merge_update);
  if (ranged && chunks > 1 && !ditattn::merge_fits(chunks, H))
    return host_fail(DIT_ERR_UNSUPPORTED, "chunks * H too large for the merge kernel");

  cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_);
  const int R = ranged ? L.ranges : 0;
  // events: [0] entry, [1] q/k (and tables) resident, [2 + c] key/value rows of chunk c resident;
  // query-range form also [2 + C + r] q rows of range r resident, [2 + C + R + r] range r merged,
  // [2 + C + 2R + r] range r copied out
  CallResources res;
  cudaError_t e = res.make(2 + (size_t)chunks + 3 * (size_t)R);
  if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  cudaEvent_t *ev = res.ev.data();
  cudaEvent_t *ev_q = ev + 2 + chunks, *ev_merged = ev_q + R, *ev_out = ev_merged + R;
  const cudaStream_t cin = res.in, cout = res.out;
  char *ws = static_cast<char *>(workspace);
  const size_t act = (size_t)B * S * H * D * 2, row = (size_t)H * D * 2;  // bytes of q and of one (b, s) row
  auto ok = [&](cudaError_t r) {
    if (e == cudaSuccess) e = r;
    return e == cudaSuccess;
  };
  auto chunk_lo = [&](int c) { return (int)((int64_t)c * S / chunks); };

  // ---------------------------------------------------------------- inputs, on the input-copy stream
  // the workspace may still be in use by earlier work on the caller's stream
  ok(cudaEventRecord(ev[0], stream)) && ok(cudaStreamWaitEvent(cin, ev[0], 0)) &&
      ok(cudaStreamWaitEvent(cout, ev[0], 0));
  if (prologue || !ranged) {
    ok(cudaMemcpyAsync(ws + L.q, q, act, cudaMemcpyHostToDevice, cin));
    if (prologue) {
      const size_t tab = (size_t)S * (D / 2) * 4;
      ok(cudaMemcpyAsync(ws + L.k, k, act, cudaMemcpyHostToDevice, cin)) &&
          ok(cudaMemcpyAsync(ws + L.wq, wq, (size_t)D * 4, cudaMemcpyHostToDevice, cin)) &&
          ok(cudaMemcpyAsync(ws + L.wk, wk, (size_t)D * 4, cudaMemcpyHostToDevice, cin)) &&
          ok(cudaMemcpyAsync(ws + L.cs, cos_tab, tab, cudaMemcpyHostToDevice, cin)) &&
          ok(cudaMemcpyAsync(ws + L.sn, sin_tab, tab, cudaMemcpyHostToDevice, cin));
    }
  } else {
    ok(copy_rows_in(ws + L.q, q, B, S, row, 0, range_edge(1, R, B, S, H), cin)) && ok(cudaEventRecord(ev_q[0], cin));
  }
  ok(cudaEventRecord(ev[1], cin));
  for (int c = 0; c < chunks && e == cudaSuccess; ++c) {
    const int lo = chunk_lo(c), hi = chunk_lo(c + 1);
    if (!prologue) ok(copy_rows_in(ws + L.k, k, B, S, row, lo, hi, cin));
    ok(copy_rows_in(ws + L.v, v, B, S, row, lo, hi, cin)) && ok(cudaEventRecord(ev[2 + c], cin));
  }
  for (int r = 1; r < R && !prologue && e == cudaSuccess; ++r)
    ok(copy_rows_in(ws + L.q, q, B, S, row, range_edge(r, R, B, S, H), range_edge(r + 1, R, B, S, H), cin)) &&
        ok(cudaEventRecord(ev_q[r], cin));
  if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));

  // ---------------------------------------------------------------- kernels, on the caller's stream
  void *dq = ws + L.q, *dk = ws + L.k, *dv = ws + L.v;
  dit_status st = DIT_OK;
  if (prologue) {
    if (!ok(cudaStreamWaitEvent(stream, ev[1], 0))) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
    st = dit_qk_norm_rope(dq, dk, dq, dk, reinterpret_cast<const float *>(ws + L.wq),
                          reinterpret_cast<const float *>(ws + L.wk), reinterpret_cast<const float *>(ws + L.cs),
                          reinterpret_cast<const float *>(ws + L.sn), B, S, H, D, eps, stream_);
    if (st != DIT_OK) return st;  // the entry point has set the detail
  }

  if (!ranged) {
    if (!prologue && !ok(cudaStreamWaitEvent(stream, ev[1], 0))) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
    float *dlse = reinterpret_cast<float *>(ws + L.lse);
    // chunk c waits only for its own key / value rows (event 2 + c)
    struct Ctx {
      cudaStream_t stream;
      cudaEvent_t *ev;
    } ctx = {stream, ev};
    auto before_chunk = [](void *p, int c) -> cudaError_t {
      const Ctx *x = static_cast<const Ctx *>(p);
      return cudaStreamWaitEvent(x->stream, x->ev[2 + c], 0);
    };
    st = ditattn::run_attention_chunks(dq, dk, dv, B, S, H, D, scale, chunks, partial_dtype, true, ws + L.acc,
                                       nullptr, ws + L.o, o_dtype, dlse, nullptr, nullptr, before_chunk, &ctx, stream);
    if (st != DIT_OK) return st;
    const size_t o_bytes = (size_t)B * S * H * D * (o_dtype == DIT_F32 ? 4 : 2);
    ok(cudaMemcpyAsync(o, ws + L.o, o_bytes, cudaMemcpyDeviceToHost, stream)) &&
        ok(cudaMemcpyAsync(lse, dlse, (size_t)B * H * S * 4, cudaMemcpyDeviceToHost, stream));
    if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
    return DIT_OK;
  }

  const size_t psize = partial_dtype == DIT_F32 ? 4 : 2, osize = o_dtype == DIT_F32 ? 4 : 2;
  const int64_t kv_st[3] = {(int64_t)S * H * D, (int64_t)H * D, D};
  for (int r = 0; r < R; ++r) {
    const int r0 = range_edge(r, R, B, S, H), rows = range_edge(r + 1, R, B, S, H) - r0;
    const int64_t part_o = (int64_t)B * rows * H * D, part_l = (int64_t)B * H * rows;
    const int64_t o_st[3] = {(int64_t)rows * H * D, (int64_t)H * D, D};
    const char *qr = static_cast<const char *>(dq) + (size_t)r0 * row;
    char *ob = ws + L.ob[r & 1];
    float *lb = reinterpret_cast<float *>(ws + L.lb[r & 1]);
    if (!prologue && !ok(cudaStreamWaitEvent(stream, ev_q[r], 0))) break;
    for (int c = 0; c < chunks; ++c) {
      if (r == 0 && !ok(cudaStreamWaitEvent(stream, ev[2 + c], 0))) break;
      // range r's output buffers were last read by the copy-out of range r - 2
      if (chunks == 1 && r >= 2 && !ok(cudaStreamWaitEvent(stream, ev_out[r - 2], 0))) break;
      void *oc = chunks == 1 ? static_cast<void *>(ob) : ws + L.parts + (size_t)c * part_o * psize;
      float *lc = chunks == 1 ? lb : reinterpret_cast<float *>(ws + L.lse_parts) + (size_t)c * part_l;
      st = ditattn::attn_checked(qr, dk, dv, B, H, rows, S, D, kv_st, kv_st, scale, chunk_lo(c), chunk_lo(c + 1),
                                 false, oc, chunks == 1 ? o_dtype : partial_dtype, o_st, lc, nullptr, DIT_BF16,
                                 nullptr, nullptr, c, stream);
      if (st != DIT_OK) return st;
    }
    if (e != cudaSuccess) break;
    if (chunks > 1) {
      if (r >= 2 && !ok(cudaStreamWaitEvent(stream, ev_out[r - 2], 0))) break;
      st = dit_attn_merge_lse(ws + L.parts, partial_dtype, reinterpret_cast<float *>(ws + L.lse_parts), chunks, B, H,
                              rows, D, part_o, part_l, ob, o_dtype, lb, stream_);
      if (st != DIT_OK) return st;
    }
    // this range's O and LSE to the host while the next range computes
    ok(cudaEventRecord(ev_merged[r], stream)) && ok(cudaStreamWaitEvent(cout, ev_merged[r], 0)) &&
        ok(cudaMemcpy2DAsync(static_cast<char *>(o) + (size_t)r0 * H * D * osize, (size_t)S * H * D * osize, ob,
                             (size_t)rows * H * D * osize, (size_t)rows * H * D * osize, B, cudaMemcpyDeviceToHost,
                             cout)) &&
        ok(cudaMemcpy2DAsync(lse + r0, (size_t)S * 4, lb, (size_t)rows * 4, (size_t)rows * 4, (size_t)B * H,
                             cudaMemcpyDeviceToHost, cout)) &&
        ok(cudaEventRecord(ev_out[r], cout));
    if (e != cudaSuccess) break;
  }
  // the call is complete on `stream` once the last copy-out is
  if (e == cudaSuccess) ok(cudaStreamWaitEvent(stream, ev_out[R - 1], 0));
  if (e != cudaSuccess) return host_fail(DIT_ERR_CUDA, cudaGetErrorString(e));
  return DIT_OK;
}

}  // extern "C"
