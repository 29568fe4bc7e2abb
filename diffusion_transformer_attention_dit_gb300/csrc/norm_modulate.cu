// Row normalisations of a DiT block on GB300 (sm_103a): LayerNorm with adaLN
// modulation, and RMSNorm over all C channels of a token.
//
// LayerNorm-modulate ("NPU Wan2.2-I2V model inference optimisation practice",
// section "NPU layer_norm_eval operator adaptation": WanLayerNorm without
// affine parameters, and FusedLayerNormModulate passing 1 + scale as the
// weight and shift as the bias of one layer-norm call), per row x of C:
//   y = (x - mean) / sqrt(var + eps) * (1 + scale[b]) + shift[b]   (biased var)
// RMSNorm over C (same page, section "NPU rms_norm operator adaptation":
// WanRMSNorm on [B, L, C]):   y = x * w / sqrt(mean(x^2) + eps)
// fp32 arithmetic, one bf16 rounding.
//
// HBM-bound (2 bytes read + 2 written per element).  One CTA of 128 threads
// per row (grid-stride beyond 2^31 rows); the row sits in registers as 16-byte
// vectors (C <= 8192, C a multiple of 8), so the two passes (mean, then the
// squared deviations) read HBM once.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace ditattn {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxVec = 8;  // 16-byte vectors per thread: C <= 8 * 8 * 128 = 8192

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Sum over the CTA; every thread gets the result.  `red` holds 4 floats.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  __syncthreads();  // `red` may still be read from the previous reduction
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return (red[0] + red[1]) + (red[2] + red[3]);
}

template <bool kLayerNorm>
__global__ void __launch_bounds__(kThreads) row_norm_kernel(const uint4 *__restrict__ x, uint4 *y,
                                                            const float *__restrict__ a, const float *__restrict__ c,
                                                            long long rows, int C, int L, float eps) {
  __shared__ float red[4];
  const int nvec = C / 8;
  const float inv_c = 1.0f / C;
  for (long long r = blockIdx.x; r < rows; r += gridDim.x) {
    const uint4 *xr = x + r * nvec;
    float v[kMaxVec][8];
#pragma unroll
    for (int u = 0; u < kMaxVec; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i < nvec) {
        const uint4 w = __ldcs(xr + i);
        const uint32_t ww[4] = {w.x, w.y, w.z, w.w};
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          v[u][2 * e] = __uint_as_float(ww[e] << 16);
          v[u][2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
        }
      }
    }
    float inv, mu = 0.f;
    if (kLayerNorm) {
      float s = 0.f;
#pragma unroll
      for (int u = 0; u < kMaxVec; ++u)
        if (threadIdx.x + u * kThreads < nvec)
#pragma unroll
          for (int e = 0; e < 8; ++e) s += v[u][e];
      mu = block_sum(s, red) * inv_c;
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < kMaxVec; ++u)
        if (threadIdx.x + u * kThreads < nvec)
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(v[u][e] - mu, v[u][e] - mu, ss);
      inv = rsqrtf(fmaf(block_sum(ss, red), inv_c, eps));
    } else {
      float ss = 0.f;
#pragma unroll
      for (int u = 0; u < kMaxVec; ++u)
        if (threadIdx.x + u * kThreads < nvec)
#pragma unroll
          for (int e = 0; e < 8; ++e) ss = fmaf(v[u][e], v[u][e], ss);
      inv = rsqrtf(fmaf(block_sum(ss, red), inv_c, eps));
    }
    // LayerNorm: a = scale [B, C], c = shift [B, C] (either may be null); RMSNorm: a = weight [C]
    const long long arow = kLayerNorm ? (r / L) * C : 0;
#pragma unroll
    for (int u = 0; u < kMaxVec; ++u) {
      const int i = threadIdx.x + u * kThreads;
      if (i < nvec) {
        uint32_t out[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float o2[2];
#pragma unroll
          for (int h = 0; h < 2; ++h) {
            const int ch = i * 8 + 2 * e + h;
            if (kLayerNorm) {
              const float sc = a ? a[arow + ch] : 0.f, sh = c ? c[arow + ch] : 0.f;
              o2[h] = (v[u][2 * e + h] - mu) * inv * (1.0f + sc) + sh;
            } else {
              o2[h] = v[u][2 * e + h] * inv * a[ch];
            }
          }
          out[e] = pack_bf16(o2[0], o2[1]);
        }
        y[r * nvec + i] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
  }
}

}  // namespace

int row_norm_max_channels() { return kMaxVec * 8 * kThreads; }

cudaError_t launch_layer_norm_modulate(const void *x, const float *scale, const float *shift, void *y, int B, int L,
                                       int C, float eps, cudaStream_t stream) {
  const long long rows = (long long)B * L;
  const long long grid = rows < 0x7fffffffLL ? rows : 0x7fffffffLL;
  row_norm_kernel<true><<<(unsigned)grid, kThreads, 0, stream>>>(static_cast<const uint4 *>(x), static_cast<uint4 *>(y),
                                                                 scale, shift, rows, C, L, eps);
  return cudaGetLastError();
}

cudaError_t launch_rms_norm(const void *x, const float *w, void *y, long long rows, int C, float eps,
                            cudaStream_t stream) {
  const long long grid = rows < 0x7fffffffLL ? rows : 0x7fffffffLL;
  row_norm_kernel<false><<<(unsigned)grid, kThreads, 0, stream>>>(static_cast<const uint4 *>(x),
                                                                  static_cast<uint4 *>(y), w, nullptr, rows, C, 1, eps);
  return cudaGetLastError();
}

}  // namespace ditattn
