// Row kernels of a DiT block on GB300 (sm_103a): LayerNorm with adaLN
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
// HBM-bound (a read and a write per element).  A row is spread over 128
// threads as 16-byte vectors held in registers as loaded (C <= 8192, C a
// multiple of 8) and read from HBM once.  Each row is reduced once: the sums
// of (x - K) and (x - K)^2 with K the row's first element (the shifted-data
// form of the variance, which avoids the cancellation of E[x^2] - mean^2 when
// |mean| >> std), or the sum of squares; one barrier per row or row pair.  The
// arithmetic runs on pairs of channels in the packed fp32 pipes (FADD2 /
// FFMA2 / FMUL2).
//
// Two kernels.  The one-row kernel (RMSNorm; LayerNorm at C = 8192): persistent
// CTAs issue the next row's loads before reducing the current one (RMSNorm at
// C = 5120 with a 7-CTA residency target: 0.95 of the measured HBM bandwidth
// at the Wan2.2 720p shape).  The
// two-row kernel (LayerNorm-modulate up to C = 7168): a step loads, reduces
// and writes two rows, loading each thread's scale / shift vectors once for
// both -- those per-row factor reads (twice the row's own bytes, through L1)
// are what held the one-row kernel at 0.84 of the measured HBM bandwidth at
// the Wan2.2 720p shape; two rows a step run at 0.92.  (Also measured on GB300
// and slower: three rows a step, the next pair prefetched, deeper prefetch in
// registers or a ring of rows in shared memory filled by cp.async or by bulk
// copies, one warp per row, and fewer CTAs per SM.)

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_math.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace ditattn {
namespace {

using attn::f2;
using attn::f2_add;
using attn::f2_fma;
using attn::f2_mul;
using attn::f2_split;

enum Mode { kLayerNormModulate = 0, kRmsNorm = 1 };

constexpr int kThreads = 128;
constexpr int kMaxVec = 8;  // 16-byte vectors per thread: C <= 8 * 8 * 128 = 8192
constexpr int kMaxCtasPerSm = 8;

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// The two bf16 channels of one 32-bit word as a packed fp32 pair.
__device__ __forceinline__ uint64_t bf16x2_to_f2(uint32_t w) {
  return f2(__uint_as_float(w << 16), __uint_as_float(w & 0xFFFF0000u));
}

// Sums over the CTA; every thread gets the results.  `red` holds 8 floats.  One
// barrier per call: the callers alternate between two `red` buffers, and the
// barrier of the next call on the other buffer orders each buffer's reads
// before its next writes.
__device__ __forceinline__ float2 block_reduce2(float v, float w, float *red) {
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

// Eight consecutive fp32 (32-byte aligned) as four packed pairs.
__device__ __forceinline__ void load_f2x4(const float *p, uint64_t (&f)[4]) {
  const float4 a0 = __ldg(reinterpret_cast<const float4 *>(p));
  const float4 a1 = __ldg(reinterpret_cast<const float4 *>(p) + 1);
  f[0] = f2(a0.x, a0.y), f[1] = f2(a0.z, a0.w), f[2] = f2(a1.x, a1.y), f[3] = f2(a1.z, a1.w);
}

// This thread's part of a row's reduction, on channel pairs: the sums of
// (x - K) and (x - K)^2 with K the row's first element (LayerNorm), or of x^2.
template <int kMode, int kVec>
__device__ __forceinline__ void partial_sums(const uint4 (&raw)[kVec], uint32_t first, int nvec, float &s,
                                             float &q) {
  uint64_t s2 = 0ull, ss2 = 0ull;  // (0.0f, 0.0f)
  const float K = __uint_as_float(first << 16);
  const uint64_t negk2 = f2(-K, -K);
#pragma unroll
  for (int u = 0; u < kVec; ++u)
    if (threadIdx.x + u * kThreads < nvec) {
      const uint32_t w[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
      for (int e = 0; e < 4; ++e) {
        const uint64_t v2 = bf16x2_to_f2(w[e]);
        if (kMode == kLayerNormModulate) {
          const uint64_t d2 = f2_add(v2, negk2);
          s2 = f2_add(s2, d2);
          ss2 = f2_fma(d2, d2, ss2);
        } else {
          ss2 = f2_fma(v2, v2, ss2);
        }
      }
    }
  float s0, s1, q0, q1;
  f2_split(s2, s0, s1);
  f2_split(ss2, q0, q1);
  s = s0 + s1, q = q0 + q1;
}

// A row's statistics from its sums over the CTA: -mean (LayerNorm; 0 for
// RMSNorm) and the inverse standard deviation / root mean square, each as a pair.
template <int kMode>
__device__ __forceinline__ void row_stats(float ts, float tq, uint32_t first, float inv_c, float eps,
                                          uint64_t &neg_mu2, uint64_t &inv2) {
  if (kMode == kLayerNormModulate) {
    const float dm = ts * inv_c;  // mean - K
    const float mu = __uint_as_float(first << 16) + dm, inv = rsqrtf(fmaxf(fmaf(tq, inv_c, -dm * dm), 0.f) + eps);
    neg_mu2 = f2(-mu, -mu);
    inv2 = f2(inv, inv);
  } else {
    const float inv = rsqrtf(fmaf(tq, inv_c, eps));
    neg_mu2 = 0ull;
    inv2 = f2(inv, inv);
  }
}

// Eight outputs from one 16-byte vector of the row and its channels' factors
// (LayerNorm-modulate: fa = scale, fc = shift; RMSNorm: fa = weight).
template <int kMode>
__device__ __forceinline__ uint4 out_vec(uint4 raw, const uint64_t (&fa)[4], const uint64_t (&fc)[4],
                                         uint64_t neg_mu2, uint64_t inv2) {
  const uint32_t w[4] = {raw.x, raw.y, raw.z, raw.w};
  uint32_t o[4];
#pragma unroll
  for (int e = 0; e < 4; ++e) {
    const uint64_t v2 = bf16x2_to_f2(w[e]);
    uint64_t y2;
    if (kMode == kLayerNormModulate) {
      // (x - mu) * (inv * (1 + scale)) + shift; a missing scale or shift reads as zeros
      const uint64_t g2 = f2_fma(inv2, fa[e], inv2);
      y2 = f2_fma(f2_add(v2, neg_mu2), g2, fc[e]);
    } else {
      y2 = f2_mul(f2_mul(v2, inv2), fa[e]);
    }
    float lo, hi;
    f2_split(y2, lo, hi);
    o[e] = pack_bf16x2(lo, hi);
  }
  return make_uint4(o[0], o[1], o[2], o[3]);
}

// One row whose 16-byte vectors this thread holds in `raw` (kLayerNormModulate:
// a = scale [B, C], c = shift [B, C], either may be null, L rows per batch
// entry; kRmsNorm: a = weight [C]).
template <int kMode, int kVec>
__device__ __forceinline__ void process_row(const uint4 (&raw)[kVec], uint32_t first, uint8_t *y, const float *a,
                                            const float *c, long long r, int nvec, int C, int L,
                                            float eps, float *red) {
  float s, q;
  partial_sums<kMode, kVec>(raw, first, nvec, s, q);
  const float2 tot = block_reduce2(s, q, red);
  uint64_t neg_mu2, inv2;
  row_stats<kMode>(tot.x, tot.y, first, 1.0f / C, eps, neg_mu2, inv2);
  const long long frow = kMode == kLayerNormModulate ? (r / L) * C : 0;
  uint4 *yv = reinterpret_cast<uint4 *>(y) + r * nvec;
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < nvec) {
      uint64_t fa[4] = {0ull, 0ull, 0ull, 0ull}, fc[4] = {0ull, 0ull, 0ull, 0ull};
      if (a) load_f2x4(a + frow + 8 * i, fa);
      if (kMode == kLayerNormModulate && c) load_f2x4(c + frow + 8 * i, fc);
      __stcs(yv + i, out_vec<kMode>(raw[u], fa, fc, neg_mu2, inv2));
    }
  }
}

template <int kVec>
__device__ __forceinline__ void load_row(uint4 (&raw)[kVec], uint32_t &first, const uint4 *__restrict__ x,
                                         long long r, int nvec) {
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < nvec) raw[u] = __ldcs(x + r * nvec + i);
  }
  // the row's first element (LayerNorm's shift), one broadcast load per warp
  first = __ldg(reinterpret_cast<const unsigned int *>(x + r * nvec));
}

// Persistent CTAs walk rows r = blockIdx.x, + gridDim.x, ...; the next row's
// loads are issued before the current row's reduction, so two rows per CTA
// are in flight.  One barrier per row: consecutive rows alternate between
// red[0..7] and red[8..15].
template <int kMode, int kVec>
__device__ __forceinline__ void row_loop(const uint4 *__restrict__ x, uint8_t *y, const float *__restrict__ a,
                                         const float *__restrict__ c, long long rows, int C, int L, float eps) {
  __shared__ float red[16];
  const int nvec = C / 8;
  uint4 cur[kVec], nxt[kVec];
  uint32_t fcur = 0, fnxt = 0;
  griddep_wait();
  griddep_launch_dependents();
  long long r = blockIdx.x;
  if (r < rows) load_row<kVec>(cur, fcur, x, r, nvec);
  for (; r < rows; r += 2LL * gridDim.x) {
    const long long r1 = r + gridDim.x;
    if (r1 < rows) load_row<kVec>(nxt, fnxt, x, r1, nvec);
    process_row<kMode, kVec>(cur, fcur, y, a, c, r, nvec, C, L, eps, red);
    if (r1 >= rows) break;
    const long long r2 = r1 + gridDim.x;
    if (r2 < rows) load_row<kVec>(cur, fcur, x, r2, nvec);
    process_row<kMode, kVec>(nxt, fnxt, y, a, c, r1, nvec, C, L, eps, red + 8);
  }
}

template <int kMode, int kVec>
__global__ void __launch_bounds__(kThreads) row_kernel(const uint4 *__restrict__ x, uint8_t *y,
                                                       const float *__restrict__ a, const float *__restrict__ c,
                                                       long long rows, int C, int L, float eps) {
  row_loop<kMode, kVec>(x, y, a, c, rows, C, L, eps);
}

// The same with a residency target of 7 CTAs per SM (registers capped at 72).
// RMSNorm at 5 vectors per thread (C = 4097 ... 5120) measured faster so
// (68 registers, 7 CTAs, against the compiler's 64 registers and 8 CTAs): the
// Wan2.2 shapes 0.92 -> 0.95 (720p) and 0.89 -> 0.90 (480p) of HBM.  At 4
// vectors the same target was slower, and at 6-8 it spills.
template <int kMode, int kVec>
__global__ void __launch_bounds__(kThreads, 7) row_kernel_res7(const uint4 *__restrict__ x, uint8_t *y,
                                                               const float *__restrict__ a,
                                                               const float *__restrict__ c, long long rows, int C,
                                                               int L, float eps) {
  row_loop<kMode, kVec>(x, y, a, c, rows, C, L, eps);
}

// Sums of four values over the CTA, as block_reduce2 (`red` holds 16 floats).
__device__ __forceinline__ float4 block_reduce4(float v0, float v1, float v2, float v3, float *red) {
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) {
    v0 += __shfl_xor_sync(0xffffffffu, v0, off);
    v1 += __shfl_xor_sync(0xffffffffu, v1, off);
    v2 += __shfl_xor_sync(0xffffffffu, v2, off);
    v3 += __shfl_xor_sync(0xffffffffu, v3, off);
  }
  if ((threadIdx.x & 31) == 0) {
    const int w = threadIdx.x >> 5;
    red[w] = v0, red[4 + w] = v1, red[8 + w] = v2, red[12 + w] = v3;
  }
  __syncthreads();
  return make_float4((red[0] + red[1]) + (red[2] + red[3]), (red[4] + red[5]) + (red[6] + red[7]),
                     (red[8] + red[9]) + (red[10] + red[11]), (red[12] + red[13]) + (red[14] + red[15]));
}

// LayerNorm-modulate on rows r and r + 1 (the second only if has_b): one
// barrier for both reductions, and each thread's scale / shift vectors loaded
// once for both rows unless row r + 1 starts another batch entry.
template <int kVec>
__device__ __forceinline__ void process_pair(const uint4 (&ra)[kVec], uint32_t first_a, const uint4 (&rb)[kVec],
                                             uint32_t first_b, bool has_b, uint8_t *y, const float *a,
                                             const float *c, long long r, int nvec, int C, int L, float eps,
                                             float *red) {
  float sa, qa, sb = 0.f, qb = 0.f;
  partial_sums<kLayerNormModulate, kVec>(ra, first_a, nvec, sa, qa);
  if (has_b) partial_sums<kLayerNormModulate, kVec>(rb, first_b, nvec, sb, qb);
  const float4 tot = block_reduce4(sa, qa, sb, qb, red);
  const float inv_c = 1.0f / C;
  uint64_t neg_mu_a, inv_a, neg_mu_b, inv_b;
  row_stats<kLayerNormModulate>(tot.x, tot.y, first_a, inv_c, eps, neg_mu_a, inv_a);
  row_stats<kLayerNormModulate>(tot.z, tot.w, first_b, inv_c, eps, neg_mu_b, inv_b);
  const long long frow_a = (r / L) * C, frow_b = ((r + 1) / L) * C;
  uint4 *yv = reinterpret_cast<uint4 *>(y) + r * nvec;
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const int i = threadIdx.x + u * kThreads;
    if (i < nvec) {
      uint64_t fa[4] = {0ull, 0ull, 0ull, 0ull}, fc[4] = {0ull, 0ull, 0ull, 0ull};
      if (a) load_f2x4(a + frow_a + 8 * i, fa);
      if (c) load_f2x4(c + frow_a + 8 * i, fc);
      __stcs(yv + i, out_vec<kLayerNormModulate>(ra[u], fa, fc, neg_mu_a, inv_a));
      if (has_b) {
        if (frow_b != frow_a) {
          if (a) load_f2x4(a + frow_b + 8 * i, fa);
          if (c) load_f2x4(c + frow_b + 8 * i, fc);
        }
        __stcs(yv + nvec + i, out_vec<kLayerNormModulate>(rb[u], fa, fc, neg_mu_b, inv_b));
      }
    }
  }
}

// LayerNorm-modulate two rows at a time: persistent CTAs walk row pairs
// (2p, 2p + 1), p = blockIdx.x, + gridDim.x, ...  A step loads both rows and
// then reduces and writes them; no loads are carried across steps (holding
// the next pair too costs the registers of two more rows, and the residency
// that pays for it), the other CTAs on the SM keep HBM busy meanwhile.
// Loading each factor vector once per pair halves the factor reads that
// bound the one-row kernel.
// Residency targets of the two-row kernel (CTAs per SM, i.e. a register cap of
// 65536 / (128 x target)).  Left to itself the compiler gives 4-5 vectors per
// thread 92-96 registers, 5 CTAs per SM; capped at 80 (no spills there) they
// run 6, which measured faster (Wan2.2 shapes, C = 5120: 0.89 -> 0.92 of HBM).
// The other widths keep the residency they get uncapped (56-116 registers);
// a 6 there would lower it (1-3 vectors) or spill (6-7).
constexpr int pair_min_blocks(int vec) { return vec <= 2 ? 8 : vec == 3 ? 7 : vec <= 5 ? 6 : vec == 6 ? 5 : 4; }

template <int kVec>
__global__ void __launch_bounds__(kThreads, pair_min_blocks(kVec)) row_pair_kernel(const uint4 *__restrict__ x, uint8_t *y,
                                                            const float *__restrict__ a,
                                                            const float *__restrict__ c, long long rows, int C,
                                                            int L, float eps) {
  __shared__ float red[32];
  const int nvec = C / 8;
  const long long pairs = (rows + 1) / 2;
  uint4 ra[kVec], rb[kVec];
  uint32_t first_a = 0, first_b = 0;
  griddep_wait();
  griddep_launch_dependents();
  int buf = 0;
  for (long long p = blockIdx.x; p < pairs; p += gridDim.x, buf ^= 16) {
    const bool has_b = 2 * p + 1 < rows;
    load_row<kVec>(ra, first_a, x, 2 * p, nvec);
    if (has_b) load_row<kVec>(rb, first_b, x, 2 * p + 1, nvec);
    process_pair<kVec>(ra, first_a, rb, first_b, has_b, y, a, c, 2 * p, nvec, C, L, eps, red + buf);
  }
}

// Persistent grid over `units` (rows or row pairs): as many CTAs as can be
// resident (registers decide, since a thread holds two rows), capped at 8 per SM.
template <typename Kernel>
cudaError_t launch_persistent(Kernel kernel, long long units, const void *x, void *y, const float *a,
                              const float *c, long long rows, int C, int L, float eps, cudaStream_t stream) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess) e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kernel, kThreads, 0);
  if (e != cudaSuccess) return e;
  const long long cap = (long long)(per_sm < 1 ? 1 : per_sm > kMaxCtasPerSm ? kMaxCtasPerSm : per_sm) * sms;
  const unsigned grid = static_cast<unsigned>(units < cap ? units : cap);
  return launch_kernel(kernel, dim3(grid), dim3(kThreads), 0, stream, static_cast<const uint4 *>(x),
                       static_cast<uint8_t *>(y), a, c, rows, C, L, eps);
}

// LayerNorm-modulate takes the two-row kernel up to 7 vectors per thread
// (C <= 7168); at 8 its registers leave too few CTAs per SM and the one-row
// kernel is faster.  RMSNorm (one factor vector, read once per row) is faster
// one row at a time at every width.
template <int kMode, int kVec>
cudaError_t launch_vec(const void *x, void *y, const float *a, const float *c, long long rows, int C,
                       int L, float eps, cudaStream_t stream) {
  if constexpr (kMode == kLayerNormModulate && kVec <= 7)
    return launch_persistent(row_pair_kernel<kVec>, (rows + 1) / 2, x, y, a, c, rows, C, L, eps, stream);
  else if constexpr (kMode == kRmsNorm && kVec == 5)
    return launch_persistent(row_kernel_res7<kMode, kVec>, rows, x, y, a, c, rows, C, L, eps, stream);
  else
    return launch_persistent(row_kernel<kMode, kVec>, rows, x, y, a, c, rows, C, L, eps, stream);
}

// kVec = the number of 16-byte vectors each of the 128 threads holds: exactly
// ceil(C / 8 / 128), so no registers go to vectors past the row's end.
template <int kMode>
cudaError_t launch(const void *x, void *y, const float *a, const float *c, long long rows, int C,
                   int L, float eps, cudaStream_t stream) {
  switch ((C / 8 + kThreads - 1) / kThreads) {
    case 1: return launch_vec<kMode, 1>(x, y, a, c, rows, C, L, eps, stream);
    case 2: return launch_vec<kMode, 2>(x, y, a, c, rows, C, L, eps, stream);
    case 3: return launch_vec<kMode, 3>(x, y, a, c, rows, C, L, eps, stream);
    case 4: return launch_vec<kMode, 4>(x, y, a, c, rows, C, L, eps, stream);
    case 5: return launch_vec<kMode, 5>(x, y, a, c, rows, C, L, eps, stream);
    case 6: return launch_vec<kMode, 6>(x, y, a, c, rows, C, L, eps, stream);
    case 7: return launch_vec<kMode, 7>(x, y, a, c, rows, C, L, eps, stream);
    default: return launch_vec<kMode, kMaxVec>(x, y, a, c, rows, C, L, eps, stream);
  }
}

}  // namespace

int row_norm_max_channels() { return kMaxVec * 8 * kThreads; }

cudaError_t launch_layer_norm_modulate(const void *x, const float *scale, const float *shift, void *y, int B, int L,
                                       int C, float eps, cudaStream_t stream) {
  return launch<kLayerNormModulate>(x, y, scale, shift, (long long)B * L, C, L, eps, stream);
}

cudaError_t launch_rms_norm(const void *x, const float *w, void *y, long long rows, int C, float eps,
                            cudaStream_t stream) {
  return launch<kRmsNorm>(x, y, w, nullptr, rows, C, 1, eps, stream);
}

}  // namespace ditattn
