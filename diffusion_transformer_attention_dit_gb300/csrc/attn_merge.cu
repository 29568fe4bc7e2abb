// Blockwise log-sum-exp merge of per-chunk attention partials for GB300 (sm_103a).
//
// Operation (the update_out_and_lse step of the ring attention loop in "feat:
// support Ascend NPU backend (torch_npu) for Qwen-Image pipelines - #274", item 2,
// and the LSE combination of two attention outputs in "NPU Wan2.2-I2V model
// inference optimisation practice", section "Ring Attention Overlap"), for
// every (b, h, i):
//   L = m + ln sum_c exp(L_c - m),  m = max_c L_c;   O = sum_c exp(L_c - L) O_c
//
// HBM-bound: C partial rows in, one row out.  A CTA owns TQ consecutive query
// rows of one batch for all heads.  Phase 1 turns the C partial LSEs of each
// (h, i) into weights in shared memory (LSE reads are contiguous in i) and
// writes the merged LSE.  Phase 2 streams the O partials as 16-byte vectors,
// all C loads of a vector issued before the fp32 accumulation, and writes the
// merged row.

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>

#include "internal.h"

namespace ditattn {
namespace {

constexpr int kThreads = 256;
constexpr int kMaxC = 64;
constexpr int kSmemBudget = 48 * 1024;

template <typename T>
struct Vec;
template <>
struct Vec<float> {
  static constexpr int N = 4;
};
template <>
struct Vec<__nv_bfloat16> {
  static constexpr int N = 8;
};

__device__ __forceinline__ void load_vec(const float *p, float (&v)[8]) {
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
  if (N == 4) {
    *reinterpret_cast<float4 *>(p) = make_float4(v[0], v[1], v[2], v[3]);
  } else {
    reinterpret_cast<float4 *>(p)[0] = make_float4(v[0], v[1], v[2], v[3]);
    reinterpret_cast<float4 *>(p)[1] = make_float4(v[4], v[5], v[6], v[7]);
  }
}
template <int N>
__device__ __forceinline__ void store_vec(__nv_bfloat16 *p, const float (&v)[8]) {
  if (N == 4) {
    *reinterpret_cast<uint2 *>(p) = make_uint2(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]));
  } else {
    *reinterpret_cast<uint4 *>(p) =
        make_uint4(pack_bf16(v[0], v[1]), pack_bf16(v[2], v[3]), pack_bf16(v[4], v[5]), pack_bf16(v[6], v[7]));
  }
}

template <typename Tin, typename Tout>
__global__ void __launch_bounds__(kThreads) merge_lse_kernel(const Tin *__restrict__ o_parts,
                                                             const float *__restrict__ lse_parts, int C, int H,
                                                             int Sq, int D, long long pso, long long psl, Tout *o,
                                                             float *lse, int TQ) {
  extern __shared__ float wgt[];  // [TQ][H][C]
  const int b = blockIdx.y;
  const int q0 = blockIdx.x * TQ;
  const int nq = min(TQ, Sq - q0);

  for (int idx = threadIdx.x; idx < H * TQ; idx += kThreads) {
    const int h = idx / TQ, qq = idx % TQ;
    if (qq >= nq) continue;
    const long long li = ((long long)b * H + h) * Sq + q0 + qq;
    float mx = -INFINITY;
    for (int c = 0; c < C; ++c) mx = fmaxf(mx, lse_parts[c * psl + li]);
    float *w = wgt + ((long long)qq * H + h) * C;
    if (mx == -INFINITY) {
      for (int c = 0; c < C; ++c) w[c] = 0.f;
      lse[li] = -INFINITY;
    } else {
      float sum = 0.f;
      for (int c = 0; c < C; ++c) sum += expf(lse_parts[c * psl + li] - mx);
      const float L = mx + logf(sum);
      for (int c = 0; c < C; ++c) w[c] = expf(lse_parts[c * psl + li] - L);
      lse[li] = L;
    }
  }
  __syncthreads();

  constexpr int N = Vec<Tin>::N;
  const int vpr = D / N;  // vectors per row
  const long long row0 = ((long long)b * Sq + q0) * H;
  const int items = nq * H * vpr;
  for (int it = threadIdx.x; it < items; it += kThreads) {
    const int rh = it / vpr, dv = it % vpr;  // rh = qq * H + h
    const long long off = (row0 + rh) * D + (long long)dv * N;
    const float *w = wgt + (long long)rh * C;
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    int c = 0;
    for (; c + 4 <= C; c += 4) {
      float v0[8], v1[8], v2[8], v3[8];
      load_vec(o_parts + c * pso + off, v0);
      load_vec(o_parts + (c + 1) * pso + off, v1);
      load_vec(o_parts + (c + 2) * pso + off, v2);
      load_vec(o_parts + (c + 3) * pso + off, v3);
#pragma unroll
      for (int i = 0; i < N; ++i) {
        acc[i] = fmaf(w[c], v0[i], acc[i]);
        acc[i] = fmaf(w[c + 1], v1[i], acc[i]);
        acc[i] = fmaf(w[c + 2], v2[i], acc[i]);
        acc[i] = fmaf(w[c + 3], v3[i], acc[i]);
      }
    }
    for (; c < C; ++c) {
      float v0[8];
      load_vec(o_parts + c * pso + off, v0);
#pragma unroll
      for (int i = 0; i < N; ++i) acc[i] = fmaf(w[c], v0[i], acc[i]);
    }
    store_vec<N>(o + off, acc);
  }
}

template <typename Tin, typename Tout>
cudaError_t launch_typed(const void *o_parts, const float *lse_parts, int C, int B, int H, int Sq, int D,
                         long long pso, long long psl, void *o, float *lse, cudaStream_t stream) {
  int TQ = 32;
  while (TQ > 1 && (long long)TQ * H * C * 4 > kSmemBudget) TQ >>= 1;
  const size_t smem = (size_t)TQ * H * C * 4;
  dim3 grid((Sq + TQ - 1) / TQ, B);
  merge_lse_kernel<Tin, Tout><<<grid, kThreads, smem, stream>>>(static_cast<const Tin *>(o_parts), lse_parts, C, H,
                                                                Sq, D, pso, psl, static_cast<Tout *>(o), lse, TQ);
  return cudaGetLastError();
}

}  // namespace

int merge_max_parts() { return kMaxC; }

bool merge_fits(int C, int H) { return C <= kMaxC && (long long)H * C * 4 <= kSmemBudget; }

cudaError_t launch_merge_lse(const void *o_parts, bool in_f32, const float *lse_parts, int C, int B, int H, int Sq,
                             int D, int64_t part_stride_o, int64_t part_stride_lse, void *o, bool out_f32,
                             float *lse, cudaStream_t stream) {
  if (in_f32 && out_f32)
    return launch_typed<float, float>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse, o, lse,
                                      stream);
  if (in_f32)
    return launch_typed<float, __nv_bfloat16>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse, o,
                                              lse, stream);
  if (out_f32)
    return launch_typed<__nv_bfloat16, float>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o, part_stride_lse, o,
                                              lse, stream);
  return launch_typed<__nv_bfloat16, __nv_bfloat16>(o_parts, lse_parts, C, B, H, Sq, D, part_stride_o,
                                                    part_stride_lse, o, lse, stream);
}

}  // namespace ditattn
