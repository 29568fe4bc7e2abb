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
// HBM-bound: every element is read once and written once.  q and k are flat
// arrays of B*S*H rows of D channels; a unit is 8 KB of consecutive rows of
// each.  A persistent CTA (four per SM) streams its units through a 3-stage
// shared-memory ring with 1-D bulk copies (TMA), rewrites each unit in place
// and bulk-stores it, so about 128 KB of loads per SM are in flight.  (Swept
// on GB300 over unit size, ring depth, CTAs per SM and threads per CTA: four
// small pipelines per SM beat two deep ones, 6.5 vs 6.1 TB/s on 1.36 GB.)  A row is held by
// D/8 lanes with one 16-byte vector (4 rotary pairs) each; the mean square is a
// shuffle reduction over those lanes.

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include <atomic>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace ditattn {
namespace {

__device__ unsigned int g_prologue_error = 0;

constexpr int kThreads = 256;
constexpr int kStages = 3;
constexpr int kUnitBytes = 8192;   // bytes of q (and of k) per unit
constexpr int kSmem = kStages * 2 * kUnitBytes + 8 * kStages;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    // two bounds: elapsed time, and an iteration count that ends the wait even if
    // the global timer were not advancing
    if ((i & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || i > kWaitLimitIters)) {
      atomicOr(&g_prologue_error, 1u);
      return false;
    }
  }
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xFFFF0000u); }

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

__device__ __forceinline__ uint4 ld_shared_v4(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}

template <int D>
__global__ void __launch_bounds__(kThreads, 4)
    qk_norm_rope_kernel(const __nv_bfloat16 *q, const __nv_bfloat16 *k, __nv_bfloat16 *q_out,
                        __nv_bfloat16 *k_out, const float *__restrict__ wq, const float *__restrict__ wk,
                        const float4 *__restrict__ cos_tab, const float4 *__restrict__ sin_tab, int S, int H,
                        float eps, long long n_rows, long long n_units) {
  constexpr int kLanes = D / 8;                // lanes per row
  constexpr int kGroups = kThreads / kLanes;   // rows per pass
  constexpr int kRows = kUnitBytes / (D * 2);  // rows per unit
  constexpr int kPasses = kRows / kGroups;
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  const uint32_t bars = base + kStages * 2 * kUnitBytes;
  auto stage_q = [&](int st) { return base + st * 2 * kUnitBytes; };
  auto full = [&](int st) { return bars + 8u * st; };

  const int g = threadIdx.x / kLanes, li = threadIdx.x % kLanes;
  // shuffles name only this row group's lanes: groups past the last row of a unit skip the work
  const unsigned gmask = (kLanes == 32 ? 0xffffffffu : ((1u << kLanes) - 1u)) << ((threadIdx.x & 31) & ~(kLanes - 1));
  const float inv_d = 1.0f / D;
  float w_q[8], w_k[8];
  griddep_wait();
  griddep_launch_dependents();
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    w_q[i] = wq[li * 8 + i];
    w_k[i] = wk[li * 8 + i];
  }

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(full(st), 1);
    mbar_fence_init();
  }
  __syncthreads();

  auto issue = [&](long long u, int st) {
    const long long r0 = u * kRows;
    const uint32_t bytes = static_cast<uint32_t>((n_rows - r0 < kRows ? n_rows - r0 : kRows) * D * 2);
    mbar_arrive_expect_tx(full(st), 2 * bytes);
    bulk_load(stage_q(st), q + r0 * D, bytes, full(st));
    bulk_load(stage_q(st) + kUnitBytes, k + r0 * D, bytes, full(st));
  };
  int issued = 0;  // units whose loads thread 0 has issued
  if (threadIdx.x == 0)
    for (int i = 0; i < kStages - 1; ++i) {
      const long long u = blockIdx.x + (long long)i * gridDim.x;
      if (u < n_units) {
        issue(u, i);
        ++issued;
      }
    }

  int it = 0;
  for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
    const int st = it % kStages;
    if (!__syncthreads_and(wait_bounded(full(st), (it / kStages) & 1))) break;
    const long long r0 = u * kRows;
    const int rows = static_cast<int>(n_rows - r0 < kRows ? n_rows - r0 : kRows);
    // rotary tables of every row this thread handles, loaded before any arithmetic
    float4 c4[kPasses], s4[kPasses];
#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
      const int row = p * kGroups + g;
      if (row < rows) {
        const long long pos = ((r0 + row) / H) % S;
        c4[p] = cos_tab[pos * kLanes + li];
        s4[p] = sin_tab[pos * kLanes + li];
      }
    }
#pragma unroll
    for (int p = 0; p < kPasses; ++p) {
      const int row = p * kGroups + g;
      if (row >= rows) continue;  // the whole row group skips together
      const float cs[4] = {c4[p].x, c4[p].y, c4[p].z, c4[p].w};
      const float sn[4] = {s4[p].x, s4[p].y, s4[p].z, s4[p].w};
#pragma unroll
      for (int which = 0; which < 2; ++which) {
        const uint32_t addr = stage_q(st) + which * kUnitBytes + row * (D * 2) + li * 16;
        const uint4 x = ld_shared_v4(addr);
        const uint32_t wv[4] = {x.x, x.y, x.z, x.w};
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
        for (int off = kLanes / 2; off > 0; off >>= 1) ss += __shfl_xor_sync(gmask, ss, off, kLanes);
        const float inv = rsqrtf(fmaf(ss, inv_d, eps));
        uint32_t out[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float a = v[2 * i] * inv * (which ? w_k[2 * i] : w_q[2 * i]);
          const float b = v[2 * i + 1] * inv * (which ? w_k[2 * i + 1] : w_q[2 * i + 1]);
          out[i] = pack_bf16(a * cs[i] - b * sn[i], a * sn[i] + b * cs[i]);
        }
        st_shared_v4(addr, out[0], out[1], out[2], out[3]);
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (threadIdx.x == 0) {
      bulk_store(q_out + r0 * D, stage_q(st), rows * D * 2);
      bulk_store(k_out + r0 * D, stage_q(st) + kUnitBytes, rows * D * 2);
      bulk_commit_group();
      const long long nu = u + (long long)(kStages - 1) * gridDim.x;
      if (nu < n_units) {
        bulk_wait_read_all_but_one();  // the stage about to be refilled has been stored
        issue(nu, (it + kStages - 1) % kStages);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0) {
    // after a wait that gave up, loads still in flight must land before the CTA exits
    for (int j = it; j < issued; ++j) wait_bounded(full(j % kStages), (j / kStages) & 1);
    bulk_wait_all();
  }
}

template <int D>
cudaError_t launch_typed(const void *q, const void *k, void *q_out, void *k_out, const float *wq, const float *wk,
                         const float *cos_tab, const float *sin_tab, int S, int H, float eps, long long n_rows,
                         cudaStream_t stream) {
  static std::atomic<bool> configured[64];  // set once the attribute is (other host threads may launch too)
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(qk_norm_rope_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  constexpr int kRows = kUnitBytes / (D * 2);
  const long long n_units = (n_rows + kRows - 1) / kRows;
  const long long grid = n_units < 4LL * sms ? n_units : 4LL * sms;
  return launch_kernel(qk_norm_rope_kernel<D>, dim3((unsigned)grid), dim3(kThreads), kSmem, stream,
                       static_cast<const __nv_bfloat16 *>(q), static_cast<const __nv_bfloat16 *>(k),
                       static_cast<__nv_bfloat16 *>(q_out), static_cast<__nv_bfloat16 *>(k_out), wq, wk,
                       reinterpret_cast<const float4 *>(cos_tab), reinterpret_cast<const float4 *>(sin_tab), S, H, eps,
                       n_rows, n_units);
}

}  // namespace

cudaError_t launch_qk_norm_rope(const void *q, const void *k, void *q_out, void *k_out, const float *wq,
                                const float *wk, const float *cos_tab, const float *sin_tab, int B, int S, int H,
                                int D, float eps, cudaStream_t stream) {
  const long long n_rows = (long long)B * S * H;
  if (D == 64) return launch_typed<64>(q, k, q_out, k_out, wq, wk, cos_tab, sin_tab, S, H, eps, n_rows, stream);
  return launch_typed<128>(q, k, q_out, k_out, wq, wk, cos_tab, sin_tab, S, H, eps, n_rows, stream);
}

cudaError_t read_and_clear_prologue_error(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_prologue_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_prologue_error, &zero, sizeof(unsigned int));
}

}  // namespace ditattn
