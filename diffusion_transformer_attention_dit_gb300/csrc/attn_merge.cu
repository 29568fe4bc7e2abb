// Blockwise log-sum-exp merge of per-chunk attention partials for GB300 (sm_103a).
//
// Operation (the update_out_and_lse step of the ring attention loop in "feat:
// support Ascend NPU backend (torch_npu) for Qwen-Image pipelines - #274", item 2,
// and the LSE combination of two attention outputs in "NPU Wan2.2-I2V model
// inference optimisation practice", section "Ring Attention Overlap"), for
// every (b, h, i):
//   L = m + ln sum_c exp(L_c - m),  m = max_c L_c;   O = sum_c exp(L_c - L) O_c
//
// HBM-bound: C partial rows in, one row out.  The O tensors are contiguous
// BSHD, so rows (b, i, h) are consecutive D-element runs; each row is spread
// over D/N lanes holding one 16-byte vector (N elements) each, and a CTA
// covers 256/(D/N) consecutive rows.  Every lane of a row reads the same C
// partial LSEs (one broadcast transaction each), forms the weights in fp32,
// issues up to 4 partial loads before accumulating, and writes its vector of
// the merged row; lane 0 of the row writes the merged LSE.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"

namespace ditattn {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxC = 1024;
constexpr int kGroup = 4;  // partial loads in flight per lane (x the CTAs resident per SM)

__device__ __forceinline__ void load_vec(const float *p, float (&v)[4]) {
  const float4 a = __ldcs(reinterpret_cast<const float4 *>(p));
  v[0] = a.x;
  v[1] = a.y;
  v[2] = a.z;
  v[3] = a.w;
}
__device__ __forceinline__ void load_vec(const __nv_bfloat16 *p, float (&v)[8]) {
  const uint4 a = __ldcs(reinterpret_cast<const uint4 *>(p));
  const uint32_t w[4] = {a.x, a.y, a.z, a.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <int N>
__device__ __forceinline__ void store_vec(float *p, const float (&v)[8]) {
  reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
  if (N == 8) reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
}
template <int N>
__device__ __forceinline__ void store_vec(__nv_bfloat16 *p, const float (&v)[8]) {
  if (N == 4)
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
  else
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
}

template <typename Tin, typename Tout, int D>
__global__ void __launch_bounds__(kThreads, 4) merge_lse_kernel(const Tin *__restrict__ o_parts,
                                                             const float *__restrict__ lse_parts, int C, int H,
                                                             int Sq, long long n_rows, long long pso, long long psl,
                                                             Tout *o, float *lse) {
  constexpr int N = 16 / sizeof(Tin);  // elements per 16-byte vector
  constexpr int kLanes = D / N;        // lanes per row
  constexpr int kRows = kThreads / kLanes;
  const long long row = (long long)blockIdx.x * kRows + threadIdx.x / kLanes;
  const int lane = threadIdx.x % kLanes;
  if (row >= n_rows) return;
  const int h = static_cast<int>(row % H);
  const long long bq = row / H;
  const long long q = bq % Sq, b = bq / Sq;
  const long long li = (b * H + h) * Sq + q;
  const long long off = row * D + (long long)lane * N;

  float mx = -INFINITY;
  for (int c = 0; c < C; ++c) mx = fmaxf(mx, lse_parts[c * psl + li]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (mx == -INFINITY) {  // no block holds any key for this row
    store_vec<N>(o + off, acc);
    if (lane == 0) lse[li] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int c = 0; c < C; ++c) sum += expf(lse_parts[c * psl + li] - mx);
  const float L = mx + logf(sum);
  for (int c0 = 0; c0 < C; c0 += kGroup) {
    float v[kGroup][N], w[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      if (c0 + u < C) {
        load_vec(o_parts + (c0 + u) * pso + off, v[u]);
        w[u] = expf(lse_parts[(c0 + u) * psl + li] - L);
      }
    }
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      if (c0 + u < C) {
#pragma unroll
        for (int i = 0; i < N; ++i) acc[i] = fmaf(w[u], v[u][i], acc[i]);
      }
    }
  }
  store_vec<N>(o + off, acc);
  if (lane == 0) lse[li] = L;
}

template <typename Tin, typename Tout, int D>
cudaError_t launch_typed(const void *o_parts, const float *lse_parts, int C, int B, int H, int Sq, long long pso,
                         long long psl, void *o, float *lse, cudaStream_t stream) {
  constexpr int kRows = kThreads / (D / (16 / sizeof(Tin)));
  const long long n_rows = (long long)B * Sq * H;
  const long long blocks = (n_rows + kRows - 1) / kRows;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  merge_lse_kernel<Tin, Tout, D><<<(unsigned)blocks, kThreads, 0, stream>>>(
      static_cast<const Tin *>(o_parts), lse_parts, C, H, Sq, n_rows, pso, psl, static_cast<Tout *>(o), lse);
  return cudaGetLastError();
}

template <typename Tin, typename Tout>
cudaError_t launch_d(const void *o_parts, const float *lse_parts, int C, int B, int H, int Sq, int D, long long pso,
                     long long psl, void *o, float *lse, cudaStream_t stream) {
  if (D == 64) return launch_typed<Tin, Tout, 64>(o_parts, lse_parts, C, B, H, Sq, pso, psl, o, lse, stream);
  return launch_typed<Tin, Tout, 128>(o_parts, lse_parts, C, B, H, Sq, pso, psl, o, lse, stream);
}

}  // namespace

int merge_max_parts() { return kMaxC; }

bool merge_fits(int C, int H) { return C <= kMaxC && H >= 1; }

cudaError_t launch_merge_lse(const void *o_parts, bool in_f32, const float *lse_parts, int C, int B, int H, int Sq,
                             int D, int64_t part_stride_o, int64_t part_stride_lse, void *o, bool out_f32,
                             float *lse, cudaStream_t stream) {
  if (in_f32 && out_f32)
    return launch_d<float, float>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse, o, lse, stream);
  if (in_f32)
    return launch_d<float, __nv_bfloat16>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse, o, lse,
                                          stream);
  if (out_f32)
    return launch_d<__nv_bfloat16, float>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse, o, lse,
                                          stream);
  return launch_d<__nv_bfloat16, __nv_bfloat16>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse,
                                                o, lse, stream);
}

}  // namespace ditattn
