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
// HBM-bound (2 bytes read + 2 written per element).  A row is spread over 128
// threads as 16-byte vectors held in registers (C <= 8192, C a multiple of 8)
// and read from HBM once.  LayerNorm takes the mean and variance in one
// reduction of the sums of (x - K) and (x - K)^2 with K the row's first
// element (the shifted-data form of the variance, which avoids the
// cancellation of E[x^2] - mean^2 when |mean| >> std): one barrier per row, as
// RMSNorm.  Persistent CTAs (8 per SM) issue the next row's loads before
// reducing the current one.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace ditattn {
namespace {

constexpr int kThreads = 128;
constexpr int kMaxVec = 8;  // 16-byte vectors per thread: C <= 8 * 8 * 128 = 8192

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Sums over the CTA; every thread gets the results.  `red` holds 4 floats per
// value.  One barrier per call: the callers alternate between two `red`
// buffers, and the barrier of the next call on the other buffer orders each
// buffer's reads before its next writes.
__device__ __forceinline__ float block_sum(float v, float *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) v += __shfl_xor_sync(0xffffffffu, v, off);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
  __syncthreads();
  return (red[0] + red[1]) + (red[2] + red[3]);
}
__device__ __forceinline__ float2 block_sum2(float v, float w, float *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    v += __shfl_xor_sync(0xffffffffu, v, off);
    w += __shfl_xor_sync(0xffffffffu, w, off);
  }
  if ((threadIdx.x & 31) == 0) {
    red[threadIdx.x >> 5] = v;
    red[4 + (threadIdx.x >> 5)] = w;
  }
  __syncthreads();
  return make_float2((red[0] + red[1]) + (red[2] + red[3]), (red[4] + red[5]) + (red[6] + red[7]));
}

// Normalise one row whose 16-byte vectors this thread holds in `raw`, and store it.
template <bool kLayerNorm, int kVec>
__device__ __forceinline__ void norm_row(const uint4 (&raw)[kVec], uint32_t first, uint4 *y,
                                         const float *__restrict__ a, const float *__restrict__ c, long long r,
                                         int nvec, int C, int L, float eps, float *red) {
  const float inv_c = 1.0f / C;
  float v[kVec][8];
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const uint32_t ww[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[u][2 * e] = __uint_as_float(ww[e] << 16);
      v[u][2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
    }
  }
  float inv, mu = 0.f;
  if (kLayerNorm) {
    // shifted sums: K = the row's first element (every thread loaded it with the row)
    const float K = __uint_as_float(first << 16);
    float s = 0.f, ss = 0.f;
#pragma unroll
    for (int u = 0; u < kVec; ++u)
      if (threadIdx.x + u * kThreads < nvec)
#pragma unroll
        for (int e = 0; e < 8; ++e) {
          const float d = v[u][e] - K;
          s += d;
          ss = fmaf(d, d, ss);
        }
    const float2 t = block_sum2(s, ss, red);
    const float dm = t.x * inv_c;  // mean - K
    mu = K + dm;
    inv = rsqrtf(fmaxf(fmaf(t.y, inv_c, -dm * dm), 0.f) + eps);
  } else {
    float ss = 0.f;
#pragma unroll
    for (int u = 0; u < kVec; ++u)
      if (threadIdx.x + u * kThreads < nvec)
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(v[u][e], v[u][e], ss);
    inv = rsqrtf(fmaf(block_sum(ss, red), inv_c, eps));  // the caller alternates `red` between rows
  }
  // LayerNorm: a = scale [B, C], c = shift [B, C] (either may be null); RMSNorm: a = weight [C].
  // The per-channel factors are read as two 16-byte vectors per 8 channels.
  const long long arow = kLayerNorm ? (r / L) * C : 0;
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < nvec) {
      float fa[8], fc[8];
      if (a) {
        const float4 a0 = __ldg(reinterpret_cast<const float4 *>(a + arow) + 2 * i);
        const float4 a1 = __ldg(reinterpret_cast<const float4 *>(a + arow) + 2 * i + 1);
        fa[0] = a0.x, fa[1] = a0.y, fa[2] = a0.z, fa[3] = a0.w, fa[4] = a1.x, fa[5] = a1.y, fa[6] = a1.z, fa[7] = a1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) fa[e] = 0.f;
      }
      if (kLayerNorm && c) {
        const float4 c0 = __ldg(reinterpret_cast<const float4 *>(c + arow) + 2 * i);
        const float4 c1 = __ldg(reinterpret_cast<const float4 *>(c + arow) + 2 * i + 1);
        fc[0] = c0.x, fc[1] = c0.y, fc[2] = c0.z, fc[3] = c0.w, fc[4] = c1.x, fc[5] = c1.y, fc[6] = c1.z, fc[7] = c1.w;
      } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) fc[e] = 0.f;
      }
      uint32_t out[4];
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        float o2[2];
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int ch = 2 * e + h;
          o2[h] = kLayerNorm ? (v[u][ch] - mu) * inv * (1.0f + fa[ch]) + fc[ch] : v[u][ch] * inv * fa[ch];
        }
        out[e] = pack_bf16(o2[0], o2[1]);
      }
      __stcs(y + r * nvec + i, make_uint4(out[0], out[1], out[2], out[3]));
    }
  }
}

template <bool kLayerNorm, int kVec>
__device__ __forceinline__ void load_row(uint4 (&raw)[kVec], uint32_t &first, const uint4 *__restrict__ x,
                                         long long r, int nvec) {
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < nvec) raw[u] = __ldcs(x + r * nvec + i);
  }
  // the row's first element (LayerNorm's shift), one broadcast load per warp
  if (kLayerNorm) first = __ldg(reinterpret_cast<const unsigned int *>(x + r * nvec));
}

// Persistent CTAs walk rows r = blockIdx.x, + gridDim.x, ...; the next row's
// loads are issued before the current row's reductions, so two rows per CTA
// are in flight.
template <bool kLayerNorm, int kVec>
__global__ void __launch_bounds__(kThreads) row_norm_kernel(const uint4 *__restrict__ x, uint4 *y,
                                                            const float *__restrict__ a, const float *__restrict__ c,
                                                            long long rows, int C, int L, float eps) {
  __shared__ float red[16];
  const int nvec = C / 8;
  uint4 cur[kVec], nxt[kVec];
  uint32_t fcur = 0, fnxt = 0;
  griddep_wait();
  griddep_launch_dependents();
  long long r = blockIdx.x;
  if (r < rows) load_row<kLayerNorm, kVec>(cur, fcur, x, r, nvec);
  // one barrier per row: consecutive rows alternate between red[0..7] and red[8..15]
  for (; r < rows; r += 2LL * gridDim.x) {
    const long long r1 = r + gridDim.x;
    if (r1 < rows) load_row<kLayerNorm, kVec>(nxt, fnxt, x, r1, nvec);
    norm_row<kLayerNorm, kVec>(cur, fcur, y, a, c, r, nvec, C, L, eps, red);
    if (r1 >= rows) break;
    const long long r2 = r1 + gridDim.x;
    if (r2 < rows) load_row<kLayerNorm, kVec>(cur, fcur, x, r2, nvec);
    norm_row<kLayerNorm, kVec>(nxt, fnxt, y, a, c, r1, nvec, C, L, eps, red + 8);
  }
}

// Persistent grid: as many CTAs as can be resident (registers decide, since a
// thread holds kVec row vectors twice), capped at 8 per SM.
template <bool kLayerNorm, int kVec>
cudaError_t launch_rows_vec(const uint4 *x, const float *a, const float *c, uint4 *y, long long rows, int C, int L,
                            float eps, cudaStream_t stream) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, row_norm_kernel<kLayerNorm, kVec>, kThreads, 0);
  if (e != cudaSuccess) return e;
  const long long cap = (long long)(per_sm < 1 ? 1 : per_sm > 8 ? 8 : per_sm) * sms;
  const unsigned grid = static_cast<unsigned>(rows < cap ? rows : cap);
  return launch_kernel(row_norm_kernel<kLayerNorm, kVec>, dim3(grid), dim3(kThreads), 0, stream, x, y, a, c, rows, C,
                       L, eps);
}

// kVec = the number of 16-byte vectors each of the 128 threads holds: exactly
// ceil(C / 8 / 128), so no registers go to vectors past the row's end.
template <bool kLayerNorm>
cudaError_t launch_rows(const void *x, const float *a, const float *c, void *y, long long rows, int C, int L,
                        float eps, cudaStream_t stream) {
  const uint4 *xx = static_cast<const uint4 *>(x);
  uint4 *yy = static_cast<uint4 *>(y);
  switch ((C / 8 + kThreads - 1) / kThreads) {
    case 1: return launch_rows_vec<kLayerNorm, 1>(xx, a, c, yy, rows, C, L, eps, stream);
    case 2: return launch_rows_vec<kLayerNorm, 2>(xx, a, c, yy, rows, C, L, eps, stream);
    case 3: return launch_rows_vec<kLayerNorm, 3>(xx, a, c, yy, rows, C, L, eps, stream);
    case 4: return launch_rows_vec<kLayerNorm, 4>(xx, a, c, yy, rows, C, L, eps, stream);
    case 5: return launch_rows_vec<kLayerNorm, 5>(xx, a, c, yy, rows, C, L, eps, stream);
    case 6: return launch_rows_vec<kLayerNorm, 6>(xx, a, c, yy, rows, C, L, eps, stream);
    case 7: return launch_rows_vec<kLayerNorm, 7>(xx, a, c, yy, rows, C, L, eps, stream);
    default: return launch_rows_vec<kLayerNorm, kMaxVec>(xx, a, c, yy, rows, C, L, eps, stream);
  }
}

}  // namespace

int row_norm_max_channels() { return kMaxVec * 8 * kThreads; }

cudaError_t launch_layer_norm_modulate(const void *x, const float *scale, const float *shift, void *y, int B, int L,
                                       int C, float eps, cudaStream_t stream) {
  return launch_rows<true>(x, scale, shift, y, (long long)B * L, C, L, eps, stream);
}

cudaError_t launch_rms_norm(const void *x, const float *w, void *y, long long rows, int C, float eps,
                            cudaStream_t stream) {
  return launch_rows<false>(x, w, nullptr, y, rows, C, 1, eps, stream);
}

}  // namespace ditattn
