// C ABI of the DiT attention core: argument validation, then one launcher per
// entry point.  Declarations and the full contract are in include/ditattn.h.

#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>

#include <atomic>

#include "../../include/ditattn.h"
#include "internal.h"

namespace {

thread_local const char *g_detail = "";
std::atomic<int> g_launch_overlap{1};

dit_status fail(dit_status s, const char *why) {
  g_detail = why;
  return s;
}

bool aligned(const void *p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// Byte range [lo, hi) covered by a BSHD tensor with element strides {b, s, h} and contiguous D.
struct Range {
  uintptr_t lo, hi;
};
Range bshd_range(const void *p, int B, int S, int H, int D, const int64_t st[3], int esize) {
  const int64_t last = (int64_t)(B - 1) * st[0] + (int64_t)(S - 1) * st[1] + (int64_t)(H - 1) * st[2] + D;
  const uintptr_t lo = reinterpret_cast<uintptr_t>(p);
  return {lo, lo + static_cast<uintptr_t>(last) * esize};
}
bool overlap(Range a, Range b) { return a.lo < b.hi && b.lo < a.hi; }

dit_status from_cuda(cudaError_t e, const char *detail) {
  if (e == cudaSuccess) return DIT_OK;
  g_detail = detail ? detail : cudaGetErrorString(e);
  return DIT_ERR_CUDA;
}

}  // namespace

bool ditattn::launch_overlap_enabled() { return g_launch_overlap.load(std::memory_order_relaxed) != 0; }
void ditattn::set_error_detail(const char *why) { g_detail = why; }

extern "C" {

dit_status dit_set_launch_overlap(int enable) {
  g_detail = "";
  if (enable != 0 && enable != 1) return fail(DIT_ERR_INVALID_ARG, "enable must be 0 or 1");
  g_launch_overlap.store(enable, std::memory_order_relaxed);
  return DIT_OK;
}

const char *dit_status_string(dit_status s) {
  switch (s) {
    case DIT_OK: return "DIT_OK";
    case DIT_ERR_INVALID_ARG: return "DIT_ERR_INVALID_ARG";
    case DIT_ERR_UNSUPPORTED: return "DIT_ERR_UNSUPPORTED";
    case DIT_ERR_CUDA: return "DIT_ERR_CUDA";
    case DIT_ERR_TIMEOUT: return "DIT_ERR_TIMEOUT";
  }
  return "DIT_ERR_UNKNOWN";
}

const char *dit_last_error_detail(void) { return g_detail; }

dit_status dit_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out, const float *wq, const float *wk,
                            const float *cos_tab, const float *sin_tab, int B, int S, int H, int D, float eps,
                            struct CUstream_st *stream) {
  g_detail = "";
  if (B < 0 || S < 0 || H < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (D != 64 && D != 128) return fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (!(eps >= 0.f) || isinf(eps)) return fail(DIT_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if ((int64_t)B * S * H == 0) return DIT_OK;
  if (!q || !k || !q_out || !k_out || !wq || !wk || !cos_tab || !sin_tab)
    return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(q_out, 16) || !aligned(k_out, 16) || !aligned(cos_tab, 16) ||
      !aligned(sin_tab, 16) || !aligned(wq, 4) || !aligned(wk, 4))
    return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const int64_t st[3] = {(int64_t)S * H * D, (int64_t)H * D, D};
  const Range rq = bshd_range(q, B, S, H, D, st, 2), rk = bshd_range(k, B, S, H, D, st, 2);
  const Range rqo = bshd_range(q_out, B, S, H, D, st, 2), rko = bshd_range(k_out, B, S, H, D, st, 2);
  if ((q_out != q && overlap(rqo, rq)) || overlap(rqo, rk) || (k_out != k && overlap(rko, rk)) || overlap(rko, rq) ||
      overlap(rqo, rko))
    return fail(DIT_ERR_INVALID_ARG, "outputs overlap inputs (only exact in-place is allowed)");
  return from_cuda(ditattn::launch_qk_norm_rope(q, k, q_out, k_out, wq, wk, cos_tab, sin_tab, B, S, H, D, eps,
                                                reinterpret_cast<cudaStream_t>(stream)),
                   nullptr);
}

}  // extern "C"

namespace {

// o_acc == nullptr: plain form.  Otherwise the update form, whose running result
// (o_acc, lse_acc) may be the output itself (same pointer, dtype and strides) or
// must not overlap any other argument.
dit_status attn_common(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                       const int64_t q_strides[3], const int64_t kv_strides[3], float scale, int kv_begin, int kv_end,
                       bool causal, void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                       struct CUstream_st *stream, bool update = false, const void *o_acc = nullptr,
                       dit_dtype acc_dtype = DIT_BF16, const int64_t acc_strides[3] = nullptr,
                       const float *lse_acc = nullptr, bool defer_wait = false) {
  g_detail = "";
  if (B < 0 || H < 0 || Sq < 0 || Skv < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (D != 64 && D != 128) return fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if (o_dtype != DIT_BF16 && o_dtype != DIT_F32) return fail(DIT_ERR_INVALID_ARG, "unknown output dtype");
  if (!(scale > 0.f) || isinf(scale)) return fail(DIT_ERR_INVALID_ARG, "scale must be finite and > 0");
  if (!q_strides || !kv_strides || !o_strides) return fail(DIT_ERR_INVALID_ARG, "null stride array");
  if ((int64_t)B * H * Sq == 0) return DIT_OK;
  if (kv_begin < 0 || kv_begin >= kv_end || kv_end > Skv)
    return fail(DIT_ERR_INVALID_ARG, "key range must satisfy 0 <= kv_begin < kv_end <= Skv");
  if (!q || !k || !v || !o || !lse) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (update) {
    if (!o_acc || !lse_acc) return fail(DIT_ERR_INVALID_ARG, "null pointer");
    if (!acc_strides) return fail(DIT_ERR_INVALID_ARG, "null stride array");
    if (acc_dtype != DIT_BF16 && acc_dtype != DIT_F32) return fail(DIT_ERR_INVALID_ARG, "unknown running-output dtype");
  }
  const int osz = o_dtype == DIT_F32 ? 4 : 2;
  for (int i = 0; i < 3; ++i) {
    if (q_strides[i] <= 0 || kv_strides[i] <= 0 || o_strides[i] <= 0)
      return fail(DIT_ERR_INVALID_ARG, "strides must be positive");
    if ((q_strides[i] * 2) % 16 || (kv_strides[i] * 2) % 16 || (o_strides[i] * osz) % 16)
      return fail(DIT_ERR_INVALID_ARG, "byte strides must be multiples of 16");
    if (q_strides[i] * 2 >= (int64_t(1) << 40) || kv_strides[i] * 2 >= (int64_t(1) << 40))
      return fail(DIT_ERR_INVALID_ARG, "stride too large for a tensor map");
  }
  if (!aligned(q, 16) || !aligned(k, 16) || !aligned(v, 16) || !aligned(o, 16) || !aligned(lse, 4))
    return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const Range ro = bshd_range(o, B, Sq, H, D, o_strides, osz);
  const Range rl = {reinterpret_cast<uintptr_t>(lse), reinterpret_cast<uintptr_t>(lse) + (uintptr_t)B * H * Sq * 4};
  const Range rq = bshd_range(q, B, Sq, H, D, q_strides, 2);
  const Range rk = bshd_range(k, B, Skv, H, D, kv_strides, 2), rv = bshd_range(v, B, Skv, H, D, kv_strides, 2);
  if (overlap(ro, rq) || overlap(ro, rk) || overlap(ro, rv) || overlap(rl, rq) || overlap(rl, rk) ||
      overlap(rl, rv) || overlap(rl, ro))
    return fail(DIT_ERR_INVALID_ARG, "outputs overlap inputs or each other");
  if (update) {
    const int asz = acc_dtype == DIT_F32 ? 4 : 2;
    for (int i = 0; i < 3; ++i) {
      if (acc_strides[i] <= 0) return fail(DIT_ERR_INVALID_ARG, "strides must be positive");
      if ((acc_strides[i] * asz) % 16) return fail(DIT_ERR_INVALID_ARG, "byte strides must be multiples of 16");
    }
    if (!aligned(o_acc, 16) || !aligned(lse_acc, 4)) return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
    const Range ra = bshd_range(o_acc, B, Sq, H, D, acc_strides, asz);
    const Range rla = {reinterpret_cast<uintptr_t>(lse_acc),
                       reinterpret_cast<uintptr_t>(lse_acc) + (uintptr_t)B * H * Sq * 4};
    const bool acc_in_place = o_acc == o && acc_dtype == o_dtype && acc_strides[0] == o_strides[0] &&
                              acc_strides[1] == o_strides[1] && acc_strides[2] == o_strides[2];
    if ((!acc_in_place && overlap(ra, ro)) || overlap(ra, rl) || (lse_acc != lse && overlap(rla, rl)) ||
        overlap(rla, ro))
      return fail(DIT_ERR_INVALID_ARG, "running result overlaps an output (only exact in-place is allowed)");
  }
  const char *detail = nullptr;
  cudaError_t e = ditattn::launch_attn_fwd(q, k, v, B, H, Sq, Skv, D, q_strides, kv_strides, scale, kv_begin, kv_end,
                                           causal, o, o_dtype == DIT_F32, o_strides, lse, update ? o_acc : nullptr,
                                           acc_dtype == DIT_F32, acc_strides, lse_acc, defer_wait,
                                           reinterpret_cast<cudaStream_t>(stream), &detail);
  return from_cuda(e, detail);
}

}  // namespace

dit_status ditattn::attn_checked(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                                 const int64_t q_strides[3], const int64_t kv_strides[3], float scale, int kv_begin,
                                 int kv_end, bool causal, void *o, dit_dtype o_dtype, const int64_t o_strides[3],
                                 float *lse, const void *o_acc, dit_dtype acc_dtype, const int64_t acc_strides[3],
                                 const float *lse_acc, int sequence_chunk, cudaStream_t stream) {
  // Only a later chunk of a chunk sequence may defer its dependency wait: its
  // predecessor on the stream is the previous chunk, which itself waited at its
  // start (chunk 0) or deferred under this same rule.
  return attn_common(q, k, v, B, H, Sq, Skv, D, q_strides, kv_strides, scale, kv_begin, kv_end, causal, o, o_dtype,
                     o_strides, lse, reinterpret_cast<struct CUstream_st *>(stream), o_acc != nullptr, o_acc,
                     acc_dtype, acc_strides, lse_acc, sequence_chunk >= 1);
}

extern "C" {

dit_status dit_attn_fwd(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                        const int64_t q_strides[3], const int64_t kv_strides[3], float scale, int kv_begin,
                        int kv_end, void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                        struct CUstream_st *stream) {
  return attn_common(q, k, v, B, H, Sq, Skv, D, q_strides, kv_strides, scale, kv_begin, kv_end, false, o, o_dtype,
                     o_strides, lse, stream);
}

dit_status dit_attn_fwd_causal(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                               const int64_t q_strides[3], const int64_t kv_strides[3], float scale, int kv_begin,
                               int kv_end, void *o, dit_dtype o_dtype, const int64_t o_strides[3], float *lse,
                               struct CUstream_st *stream) {
  return attn_common(q, k, v, B, H, Sq, Skv, D, q_strides, kv_strides, scale, kv_begin, kv_end, true, o, o_dtype,
                     o_strides, lse, stream);
}

dit_status dit_attn_fwd_update(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                               const int64_t q_strides[3], const int64_t kv_strides[3], float scale, int kv_begin,
                               int kv_end, int causal, const void *o_acc, dit_dtype acc_dtype,
                               const int64_t acc_strides[3], const float *lse_acc, void *o, dit_dtype o_dtype,
                               const int64_t o_strides[3], float *lse, struct CUstream_st *stream) {
  if (causal != 0 && causal != 1) return fail(DIT_ERR_INVALID_ARG, "causal must be 0 or 1");
  return attn_common(q, k, v, B, H, Sq, Skv, D, q_strides, kv_strides, scale, kv_begin, kv_end, causal == 1, o,
                     o_dtype, o_strides, lse, stream, true, o_acc, acc_dtype, acc_strides, lse_acc);
}

dit_status dit_attn_merge_lse(const void *o_parts, dit_dtype in_dtype, const float *lse_parts, int C, int B, int H,
                              int Sq, int D, int64_t part_stride_o, int64_t part_stride_lse, void *o,
                              dit_dtype out_dtype, float *lse, struct CUstream_st *stream) {
  g_detail = "";
  if (B < 0 || H < 0 || Sq < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (C < 1) return fail(DIT_ERR_INVALID_ARG, "C must be >= 1");
  if (D != 64 && D != 128) return fail(DIT_ERR_UNSUPPORTED, "head dim must be 64 or 128");
  if ((in_dtype != DIT_BF16 && in_dtype != DIT_F32) || (out_dtype != DIT_BF16 && out_dtype != DIT_F32))
    return fail(DIT_ERR_INVALID_ARG, "unknown dtype");
  if (!ditattn::merge_fits(C, H)) return fail(DIT_ERR_UNSUPPORTED, "C * H too large for the merge kernel");
  if ((int64_t)B * H * Sq == 0) return DIT_OK;
  if (!o_parts || !lse_parts || !o || !lse) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  const int isz = in_dtype == DIT_F32 ? 4 : 2, osz = out_dtype == DIT_F32 ? 4 : 2;
  const int64_t part_o = (int64_t)B * Sq * H * D, part_l = (int64_t)B * H * Sq;
  if (C > 1 && (part_stride_o < part_o || part_stride_lse < part_l))
    return fail(DIT_ERR_INVALID_ARG, "part strides smaller than one part (parts would overlap)");
  if ((part_stride_o * isz) % 16) return fail(DIT_ERR_INVALID_ARG, "part stride of O must be a multiple of 16 bytes");
  if (!aligned(o_parts, 16) || !aligned(o, 16) || !aligned(lse_parts, 4) || !aligned(lse, 4))
    return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const uintptr_t op = reinterpret_cast<uintptr_t>(o_parts), lp = reinterpret_cast<uintptr_t>(lse_parts);
  const Range rin = {op, op + (uintptr_t)((C - 1) * part_stride_o + part_o) * isz};
  const Range rlin = {lp, lp + (uintptr_t)((C - 1) * part_stride_lse + part_l) * 4};
  const Range ro = {reinterpret_cast<uintptr_t>(o), reinterpret_cast<uintptr_t>(o) + (uintptr_t)part_o * osz};
  const Range rl = {reinterpret_cast<uintptr_t>(lse), reinterpret_cast<uintptr_t>(lse) + (uintptr_t)part_l * 4};
  if (overlap(ro, rin) || overlap(ro, rlin) || overlap(rl, rin) || overlap(rl, rlin) || overlap(ro, rl))
    return fail(DIT_ERR_INVALID_ARG, "outputs overlap inputs or each other");
  return from_cuda(ditattn::launch_merge_lse(o_parts, in_dtype == DIT_F32, lse_parts, C, B, H, Sq, D, part_stride_o,
                                             part_stride_lse, o, out_dtype == DIT_F32, lse,
                                             reinterpret_cast<cudaStream_t>(stream)),
                   nullptr);
}

dit_status dit_poll_device_error(struct CUstream_st *stream) {
  g_detail = "";
  unsigned int va = 0, vp = 0, vm = 0;
  cudaError_t e = cudaStreamSynchronize(reinterpret_cast<cudaStream_t>(stream));
  if (e == cudaSuccess) e = ditattn::read_and_clear_attn_error(&va);
  if (e == cudaSuccess) e = ditattn::read_and_clear_prologue_error(&vp);
  if (e == cudaSuccess) e = ditattn::read_and_clear_merge_error(&vm);
  unsigned int vf = 0;
  if (e == cudaSuccess) e = ditattn::read_and_clear_fp8_error(&vf);
  if (e != cudaSuccess) return from_cuda(e, nullptr);
  if (va | vp | vm | vf) return fail(DIT_ERR_TIMEOUT, "a bounded device-side wait gave up");
  return DIT_OK;
}

dit_status dit_layer_norm_modulate(const void *x, const float *scale, const float *shift, void *y, int B, int L,
                                   int C, float eps, struct CUstream_st *stream) {
  g_detail = "";
  if (B < 0 || L < 0 || C < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (C % 8 || C > ditattn::row_norm_max_channels())
    return fail(DIT_ERR_UNSUPPORTED, "C must be a multiple of 8 and at most 8192");
  if (!(eps >= 0.f) || isinf(eps)) return fail(DIT_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if ((int64_t)B * L * C == 0) return DIT_OK;
  if (!x || !y) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(scale, 16) || !aligned(shift, 16))
    return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const uintptr_t n = (uintptr_t)B * L * C * 2;
  const Range rx = {reinterpret_cast<uintptr_t>(x), reinterpret_cast<uintptr_t>(x) + n};
  const Range ry = {reinterpret_cast<uintptr_t>(y), reinterpret_cast<uintptr_t>(y) + n};
  if (x != y && overlap(rx, ry)) return fail(DIT_ERR_INVALID_ARG, "y overlaps x (only exact in-place is allowed)");
  return from_cuda(ditattn::launch_layer_norm_modulate(x, scale, shift, y, B, L, C, eps,
                                                       reinterpret_cast<cudaStream_t>(stream)),
                   nullptr);
}

dit_status dit_rms_norm(const void *x, const float *w, void *y, int64_t rows, int C, float eps,
                        struct CUstream_st *stream) {
  g_detail = "";
  if (rows < 0 || C < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (C % 8 || C > ditattn::row_norm_max_channels())
    return fail(DIT_ERR_UNSUPPORTED, "C must be a multiple of 8 and at most 8192");
  if (!(eps >= 0.f) || isinf(eps)) return fail(DIT_ERR_INVALID_ARG, "eps must be finite and >= 0");
  if (rows * C == 0) return DIT_OK;
  if (!x || !y || !w) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(y, 16) || !aligned(w, 16)) return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const uintptr_t n = (uintptr_t)rows * C * 2;
  const Range rx = {reinterpret_cast<uintptr_t>(x), reinterpret_cast<uintptr_t>(x) + n};
  const Range ry = {reinterpret_cast<uintptr_t>(y), reinterpret_cast<uintptr_t>(y) + n};
  if (x != y && overlap(rx, ry)) return fail(DIT_ERR_INVALID_ARG, "y overlaps x (only exact in-place is allowed)");
  return from_cuda(ditattn::launch_rms_norm(x, w, y, rows, C, eps, reinterpret_cast<cudaStream_t>(stream)), nullptr);
}

dit_status dit_quant_fp8_rows(const void *x, void *codes, float *scale, int64_t M, int K, struct CUstream_st *stream) {
  g_detail = "";
  if (M < 0 || K < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if (K % 16 || K > ditattn::quant_fp8_max_k())
    return fail(DIT_ERR_UNSUPPORTED, "K must be a multiple of 16 and at most 8192");
  if (M * K == 0) return DIT_OK;
  if (!x || !codes || !scale) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (!aligned(x, 16) || !aligned(codes, 16) || !aligned(scale, 4)) return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const Range rx = {reinterpret_cast<uintptr_t>(x), reinterpret_cast<uintptr_t>(x) + (uintptr_t)M * K * 2};
  const Range rc = {reinterpret_cast<uintptr_t>(codes), reinterpret_cast<uintptr_t>(codes) + (uintptr_t)M * K};
  const Range rs = {reinterpret_cast<uintptr_t>(scale), reinterpret_cast<uintptr_t>(scale) + (uintptr_t)M * 4};
  if (overlap(rx, rc) || overlap(rx, rs) || overlap(rc, rs)) return fail(DIT_ERR_INVALID_ARG, "buffers overlap");
  return from_cuda(ditattn::launch_quant_fp8_rows(x, codes, scale, M, K, reinterpret_cast<cudaStream_t>(stream)),
                   nullptr);
}

dit_status dit_gemm_fp8(const void *a, const float *a_scale, const void *b, const float *b_scale, void *out, int M,
                        int N, int K, int64_t lda, int64_t ldb, int64_t ldo, struct CUstream_st *stream) {
  g_detail = "";
  if (M < 0 || N < 0 || K < 0) return fail(DIT_ERR_INVALID_ARG, "negative size");
  if ((int64_t)M * N == 0) return DIT_OK;
  if (K <= 0 || K % 16) return fail(DIT_ERR_UNSUPPORTED, "K must be a positive multiple of 16");
  if (!a || !b || !a_scale || !b_scale || !out) return fail(DIT_ERR_INVALID_ARG, "null pointer");
  if (lda < K || ldb < K || ldo < N || lda % 16 || ldb % 16 || ldo % 8)
    return fail(DIT_ERR_INVALID_ARG, "leading dimensions must cover a row and be multiples of 16 bytes");
  if (!aligned(a, 16) || !aligned(b, 16) || !aligned(out, 16) || !aligned(a_scale, 4) || !aligned(b_scale, 4))
    return fail(DIT_ERR_INVALID_ARG, "pointer misaligned");
  const Range ro = {reinterpret_cast<uintptr_t>(out), reinterpret_cast<uintptr_t>(out) + (uintptr_t)((M - 1) * ldo + N) * 2};
  const Range ra = {reinterpret_cast<uintptr_t>(a), reinterpret_cast<uintptr_t>(a) + (uintptr_t)((M - 1) * lda + K)};
  const Range rb = {reinterpret_cast<uintptr_t>(b), reinterpret_cast<uintptr_t>(b) + (uintptr_t)((N - 1) * ldb + K)};
  if (overlap(ro, ra) || overlap(ro, rb)) return fail(DIT_ERR_INVALID_ARG, "output overlaps an input");
  const char *detail = nullptr;
  cudaError_t e = ditattn::launch_gemm_fp8(a, a_scale, b, b_scale, out, M, N, K, lda, ldb, ldo,
                                           reinterpret_cast<cudaStream_t>(stream), &detail);
  return from_cuda(e, detail);
}

dit_status dit_selftest_wait_timeout(struct CUstream_st *stream) {
  g_detail = "";
  return from_cuda(ditattn::launch_wait_timeout_selftest(reinterpret_cast<cudaStream_t>(stream)), nullptr);
}

dit_status dit_selftest_fp8_quotients(uint64_t counts[2], struct CUstream_st *stream) {
  g_detail = "";
  if (!counts) return fail(DIT_ERR_INVALID_ARG, "null counts");
  unsigned long long c[2] = {0ull, 0ull};
  const cudaError_t e = ditattn::run_fp8_quotient_selftest(c, reinterpret_cast<cudaStream_t>(stream));
  const dit_status st = from_cuda(e, nullptr);
  counts[0] = c[0];
  counts[1] = c[1];
  return st;
}

}  // extern "C"
