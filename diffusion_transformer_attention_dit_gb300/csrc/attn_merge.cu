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
#include <atomic>

#include "internal.h"
#include "sm100_ptx.cuh"

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

// Hardware base-2 exponential / logarithm (ex2.approx / lg2.approx, ~2 ulp): the
// merge weights exp(L_c - L) and L = m + ln(sum) are formed in base 2.
__device__ __forceinline__ float fast_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
__device__ __forceinline__ float fast_lg2(float x) {
  float y;
  asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.69314718055994531f;

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
  griddep_wait();
  griddep_launch_dependents();

  float mx = -INFINITY;
  for (int c = 0; c < C; ++c) mx = fmaxf(mx, lse_parts[c * psl + li]);
  float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (mx == -INFINITY) {  // no block holds any key for this row
    store_vec<N>(o + off, acc);
    if (lane == 0) lse[li] = -INFINITY;
    return;
  }
  float sum = 0.f;
  for (int c = 0; c < C; ++c) sum += fast_ex2((lse_parts[c * psl + li] - mx) * kLog2e);
  const float L = mx + fast_lg2(sum) * kLn2;
  for (int c0 = 0; c0 < C; c0 += kGroup) {
    float v[kGroup][N], w[kGroup];
#pragma unroll
    for (int u = 0; u < kGroup; ++u) {
      if (c0 + u < C) {
        load_vec(o_parts + (c0 + u) * pso + off, v[u]);
        w[u] = fast_ex2((lse_parts[(c0 + u) * psl + li] - L) * kLog2e);
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

// ---------------------------------------------------------------- bulk-copy path
// For D = 128 and C in {2, 4, 8}: a unit is 32 KB / (C * D * size) consecutive rows; each
// of the C partial slabs of a unit is one 1-D bulk copy (TMA) into a 2-stage
// shared-memory ring, three persistent CTAs per SM, so up to 192 KB per SM is
// in flight (swept on GB300 over stage size, ring depth, CTAs per SM and
// threads: 7.2 TB/s on the 7.1 GB Wan2.2-720p merge, against 5.6 TB/s with
// two 3-stage CTAs).  The C partial LSEs of each of a thread's rows (rows x C =
// 8) are held in registers, loaded before the slab wait.

__device__ unsigned int g_merge_error = 0;

constexpr int kStages = 2;
constexpr int kStageBytes = 32768;
constexpr int kBulkSmem = kStages * kStageBytes + 8 * kStages;
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
      atomicOr(&g_merge_error, 1u);
      return false;
    }
  }
}

template <typename Tin>
__device__ __forceinline__ void load_vec_smem(uint32_t addr, float (&v)[16 / sizeof(Tin)]);
template <>
__device__ __forceinline__ void load_vec_smem<float>(uint32_t addr, float (&v)[4]) {
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v[0]), "=f"(v[1]), "=f"(v[2]), "=f"(v[3]) : "r"(addr));
}
template <>
__device__ __forceinline__ void load_vec_smem<__nv_bfloat16>(uint32_t addr, float (&v)[8]) {
  uint32_t w[4];
  asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];" : "=r"(w[0]), "=r"(w[1]), "=r"(w[2]), "=r"(w[3]) : "r"(addr));
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    v[2 * i] = __uint_as_float(w[i] << 16);
    v[2 * i + 1] = __uint_as_float(w[i] & 0xFFFF0000u);
  }
}

template <typename Tin, typename Tout, int D, int C>
__global__ void __launch_bounds__(kThreads, 3)
    merge_lse_bulk_kernel(const Tin *o_parts, const float *__restrict__ lse_parts, int H, int Sq, long long n_rows,
                          long long pso, long long psl, Tout *o, float *lse, long long n_units) {
  constexpr int N = 16 / sizeof(Tin);  // elements per 16-byte vector
  constexpr int kLanes = D / N;        // lanes per row
  constexpr int kRowsPerPass = kThreads / kLanes;
  constexpr int kUnitRows = kStageBytes / (C * D * (int)sizeof(Tin));
  constexpr int kRowsPerThread = kUnitRows / kRowsPerPass;
  constexpr int kSlab = kUnitRows * D * (int)sizeof(Tin);  // bytes of one partial's rows in a unit
  static_assert(kRowsPerThread >= 1 && kRowsPerThread * kRowsPerPass == kUnitRows, "unit shape");
  extern __shared__ __align__(128) uint8_t smem[];
  const uint32_t base = smem_u32(smem);
  const uint32_t bars = base + kStages * kStageBytes;
  auto full = [&](int st) { return bars + 8u * st; };
  const int g = threadIdx.x / kLanes, lane = threadIdx.x % kLanes;
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int st = 0; st < kStages; ++st) mbar_init(full(st), 1);
    mbar_fence_init();
  }
  __syncthreads();
  auto issue = [&](long long u, int st) {
    const long long r0 = u * kUnitRows;
    const long long rows = n_rows - r0 < kUnitRows ? n_rows - r0 : kUnitRows;
    const uint32_t bytes = static_cast<uint32_t>(rows * D * sizeof(Tin));
    mbar_arrive_expect_tx(full(st), bytes * C);
#pragma unroll
    for (int c = 0; c < C; ++c) bulk_load(base + st * kStageBytes + c * kSlab, o_parts + c * pso + r0 * D, bytes, full(st));
  };
  int issued = 0;
  if (threadIdx.x == 0)
    for (int i = 0; i < kStages; ++i) {
      const long long u = blockIdx.x + (long long)i * gridDim.x;
      if (u < n_units) {
        issue(u, i);
        ++issued;
      }
    }
  int it = 0;
  for (long long u = blockIdx.x; u < n_units; u += gridDim.x, ++it) {
    const int st = it % kStages;
    const long long r0 = u * kUnitRows;
    const int rows = static_cast<int>(n_rows - r0 < kUnitRows ? n_rows - r0 : kUnitRows);
    // the partial LSEs of this thread's rows are fetched before waiting for the slabs
    long long li[kRowsPerThread];
    float lv[kRowsPerThread][C];
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      const int row = g + k * kRowsPerPass;
      const long long gr = r0 + row, bq = gr / H;
      li[k] = (bq / Sq * H + gr % H) * Sq + bq % Sq;
#pragma unroll
      for (int c = 0; c < C; ++c) lv[k][c] = row < rows ? lse_parts[c * psl + li[k]] : -INFINITY;
    }
    const bool ok = wait_bounded(full(st), (it / kStages) & 1);
    if (!__syncthreads_and(ok)) break;
#pragma unroll
    for (int k = 0; k < kRowsPerThread; ++k) {
      const int row = g + k * kRowsPerPass;
      if (row >= rows) continue;
      float mx = lv[k][0];
#pragma unroll
      for (int c = 1; c < C; ++c) mx = fmaxf(mx, lv[k][c]);
      float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
      float L = -INFINITY;
      if (mx != -INFINITY) {
        float sum = 0.f;
#pragma unroll
        for (int c = 0; c < C; ++c) sum += fast_ex2((lv[k][c] - mx) * kLog2e);
        L = mx + fast_lg2(sum) * kLn2;
        const uint32_t src = base + st * kStageBytes + row * (D * (int)sizeof(Tin)) + lane * 16;
#pragma unroll
        for (int c = 0; c < C; ++c) {
          const float w = fast_ex2((lv[k][c] - L) * kLog2e);
          float v[N];
          load_vec_smem<Tin>(src + c * kSlab, v);
#pragma unroll
          for (int i = 0; i < N; ++i) acc[i] = fmaf(w, v[i], acc[i]);
        }
      }
      store_vec<N>(o + (r0 + row) * D + lane * N, acc);
      if (lane == 0) lse[li[k]] = L;
    }
    __syncthreads();  // every thread is done with this stage
    if (threadIdx.x == 0) {
      const long long nu = u + (long long)kStages * gridDim.x;
      if (nu < n_units) {
        issue(nu, st);
        ++issued;
      }
    }
  }
  if (threadIdx.x == 0)
    for (int j = it; j < issued; ++j) wait_bounded(full(j % kStages), (j / kStages) & 1);
}

template <typename Tin, typename Tout, int C>
cudaError_t launch_bulk(const void *o_parts, const float *lse_parts, int B, int H, int Sq, long long pso,
                        long long psl, void *o, float *lse, cudaStream_t stream) {
  constexpr int D = 128;
  static std::atomic<bool> configured[64];  // set once the attribute is (other host threads may launch too)
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(merge_lse_bulk_kernel<Tin, Tout, D, C>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kBulkSmem);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return e;
  const long long n_rows = (long long)B * Sq * H;
  constexpr int kUnitRows = kStageBytes / (C * D * (int)sizeof(Tin));
  const long long n_units = (n_rows + kUnitRows - 1) / kUnitRows;
  const long long grid = n_units < 3LL * sms ? n_units : 3LL * sms;
  return launch_kernel(merge_lse_bulk_kernel<Tin, Tout, D, C>, dim3((unsigned)grid), dim3(kThreads), kBulkSmem, stream,
                       static_cast<const Tin *>(o_parts), lse_parts, H, Sq, n_rows, pso, psl, static_cast<Tout *>(o),
                       lse, n_units);
}

template <typename Tin, typename Tout, int D>
cudaError_t launch_typed(const void *o_parts, const float *lse_parts, int C, int B, int H, int Sq, long long pso,
                         long long psl, void *o, float *lse, cudaStream_t stream) {
  constexpr int kRows = kThreads / (D / (16 / sizeof(Tin)));
  const long long n_rows = (long long)B * Sq * H;
  const long long blocks = (n_rows + kRows - 1) / kRows;
  if (blocks > 0x7fffffffLL) return cudaErrorInvalidConfiguration;
  return launch_kernel(merge_lse_kernel<Tin, Tout, D>, dim3((unsigned)blocks), dim3(kThreads), 0, stream,
                       static_cast<const Tin *>(o_parts), lse_parts, C, H, Sq, n_rows, pso, psl,
                       static_cast<Tout *>(o), lse);
}

template <typename Tin, typename Tout>
cudaError_t launch_d(const void *o_parts, const float *lse_parts, int C, int B, int H, int Sq, int D, long long pso,
                     long long psl, void *o, float *lse, cudaStream_t stream) {
  // bulk-copy path for the common chunk counts at D = 128; everything else row-parallel
  if (D == 128 && C == 2) return launch_bulk<Tin, Tout, 2>(o_parts, lse_parts, B, H, Sq, pso, psl, o, lse, stream);
  if (D == 128 && C == 4) return launch_bulk<Tin, Tout, 4>(o_parts, lse_parts, B, H, Sq, pso, psl, o, lse, stream);
  if (D == 128 && C == 8) return launch_bulk<Tin, Tout, 8>(o_parts, lse_parts, B, H, Sq, pso, psl, o, lse, stream);
  if (D == 64) return launch_typed<Tin, Tout, 64>(o_parts, lse_parts, C, B, H, Sq, pso, psl, o, lse, stream);
  return launch_typed<Tin, Tout, 128>(o_parts, lse_parts, C, B, H, Sq, pso, psl, o, lse, stream);
}

}  // namespace

int merge_max_parts() { return kMaxC; }

cudaError_t read_and_clear_merge_error(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_merge_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_merge_error, &zero, sizeof(unsigned int));
}

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
