// Fused per-head QK-RMSNorm + interleaved RoPE for GB300 (sm_103a).
//
// Operation ("Cosmos Ascend NPU multi-card parallel optimisation notes",
// sections 3.2 and 3.3; "NPU Wan2.2-I2V model inference optimisation practice",
// sections "NPU rms_norm operator adaptation" and "NPU rotary_mul operator
// adaptation", rotary_mode "interleave"), for every (b, s, h) row of q and of k:
//   y_d = x_d * w_d / sqrt(mean_d x_d^2 + eps)
//   (y_2i, y_2i+1) -> (y_2i c - y_2i+1 s, y_2i s + y_2i+1 c),  c, s = cos/sin[s, i]
// fp32 arithmetic, one bf16 rounding at the end.
//
// HBM-bound: every element is read once and written once.  One CTA iteration
// handles one sequence position (b, s) for all heads of q and k, so the cos/sin
// values of that position are loaded once per thread and reused for 2H rows.
// A row of D channels is held by D/8 lanes, each with one 16-byte vector of 8
// channels (4 rotary pairs); the mean square is a shuffle reduction over those
// lanes.  Four rows per thread are loaded before any is used to keep enough
// bytes in flight.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "internal.h"

namespace ditattn {
namespace {

constexpr int kThreads = 256;
constexpr int kUnroll = 4;

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 2) qk_norm_rope_kernel(const uint4 *__restrict__ q, const uint4 *__restrict__ k,
                                                                uint4 *q_out, uint4 *k_out,
                                                                const float *__restrict__ wq,
                                                                const float *__restrict__ wk,
                                                                const float4 *__restrict__ cos_tab,
                                                                const float4 *__restrict__ sin_tab, int S, int H,
                                                                float eps, long long n_pos) {
  constexpr int kLanes = D / 8;               // lanes per row
  constexpr int kGroups = kThreads / kLanes;  // rows in flight per CTA step
  const int g = threadIdx.x / kLanes, li = threadIdx.x % kLanes;
  const float inv_d = 1.0f / D;

  float w_q[8], w_k[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w_q[i] = wq[li * 8 + i];
    w_k[i] = wk[li * 8 + i];
  }

  const int rows = 2 * H;  // q heads then k heads
  for (long long pos = blockIdx.x; pos < n_pos; pos += gridDim.x) {
    const int s = static_cast<int>(pos % S);
    const float4 c4 = cos_tab[(long long)s * kLanes + li];
    const float4 s4 = sin_tab[(long long)s * kLanes + li];
    const float cs[4] = {c4.x, c4.y, c4.z, c4.w};
    const float sn[4] = {s4.x, s4.y, s4.z, s4.w};
    for (int r0 = g; r0 < rows; r0 += kGroups * kUnroll) {
      uint4 x[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = r0 + u * kGroups;
        if (r < rows) {
          const uint4 *src = r < H ? q : k;
          const int hh = r < H ? r : r - H;
          x[u] = src[(pos * H + hh) * kLanes + li];
        }
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = r0 + u * kGroups;
        // every lane of a row group shares r, so the shuffle masks below stay within live lanes
        if (r >= rows) continue;
        const uint32_t wv[4] = {x[u].x, x[u].y, x[u].z, x[u].w};
        float v[8];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          v[2 * i] = bf16_lo(wv[i]);
          v[2 * i + 1] = bf16_hi(wv[i]);
        }
        float ss = 0.f;
#pragma unroll
        for (int i = 0; i < 8; ++i) ss = fmaf(v[i], v[i], ss);
#pragma unroll
        for (int off = kLanes / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off, kLanes);
        const float inv = rsqrtf(fmaf(ss, inv_d, eps));
        const bool is_q = r < H;
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = v[2 * i] * inv * (is_q ? w_q[2 * i] : w_k[2 * i]);
          const float b = v[2 * i + 1] * inv * (is_q ? w_q[2 * i + 1] : w_k[2 * i + 1]);
          out[i] = pack_bf16(a * cs[i] - b * sn[i], a * sn[i] + b * cs[i]);
        }
        uint4 *dst = r < H ? q_out : k_out;
        const int hh = r < H ? r : r - H;
        dst[(pos * H + hh) * kLanes + li] = make_uint4(out[0], out[1], out[2], out[3]);
      }
    }
  }
}

}  // namespace

cudaError_t launch_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out, const float *wq,
                                const float *wk, const float *cos_tab, const float *sin_tab, int B, int S, int H,
                                int D, float eps, cudaStream_t stream) {
  const long long n_pos = (long long)B * S;
  // one CTA per sequence position while the grid fits; grid-stride beyond that
  const long long blocks = n_pos < 0x7fffffffLL ? n_pos : 0x7fffffffLL;
  if (D == 64)
    qk_norm_rope_kernel<64><<<(unsigned)blocks, kThreads, 0, stream>>>(
        static_cast<const uint4 *>(q), static_cast<const uint4 *>(k), static_cast<uint4 *>(q_out),
        static_cast<uint4 *>(k_out), wq, wk, reinterpret_cast<const float4 *>(cos_tab),
        reinterpret_cast<const float4 *>(sin_tab), S, H, eps, n_pos);
  else
    qk_norm_rope_kernel<128><<<(unsigned)blocks, kThreads, 0, stream>>>(
        static_cast<const uint4 *>(q), static_cast<const uint4 *>(k), static_cast<uint4 *>(q_out),
        static_cast<uint4 *>(k_out), wq, wk, reinterpret_cast<const float4 *>(cos_tab),
        reinterpret_cast<const float4 *>(sin_tab), S, H, eps, n_pos);
  return cudaGetLastError();
}

}  // namespace ditattn
