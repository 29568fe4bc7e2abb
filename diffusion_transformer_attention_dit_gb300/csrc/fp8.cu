// W8A8 fp8 (e4m3) projection for GB300 (sm_103a): per-token dynamic
// quantisation and the scaled fp8 GEMM that consumes it.
//
// Operation ("feat: support Ascend NPU backend (torch_npu) for Qwen-Image
// pipelines - #274", item 4, npu_quant_linear: per-token dynamic activation
// quantisation, per-channel weight scales, quantised matmul to bf16):
//   quantise:  scale_m = max_k |x_mk| / 448 (1 for an all-zero row),
//              code_mk = e4m3(x_mk / scale_m)   (round to nearest even, saturating)
//   GEMM:      out_mn = a_scale_m * b_scale_n * sum_k A_mk B_nk
//
// Quantiser: HBM-bound; a row is spread over 128 threads as 16-byte vectors
// held in registers, one CTA max-reduction per row; persistent CTAs issue the
// next row's loads before reducing the current one; the quotient x / scale is
// formed by Markstein's division (one correctly rounded reciprocal per row,
// then per element a product, its exact FMA residual and one FMA correction,
// on packed fp32 pairs) and converted with cvt.rn.satfinite.e4m3x2.  The codes
// equal those of the IEEE quotient on every bf16 input (checked exhaustively).
//
// GEMM: persistent CTA pairs (clusters of 2, one CTA per SM) over 256 x 256
// output tiles.  Each CTA's TMA warp streams 128-byte K blocks of its 128 A
// rows and of its half of the tile's 256 B rows into a 6-stage ring (128-byte
// swizzle) across tile boundaries; one thread of the pair issues
// tcgen05.mma.cta_group::2 kind::f8f6f4 (M 256, N 256, K 32 per instruction)
// into one of two 256-column fp32 TMEM accumulators in each CTA; four epilogue
// warps per CTA drain the other: read it back, apply the two scales, convert to
// bf16, stage 64-column boxes in two alternating swizzled buffers and store
// them with TMA.  Sharing B across the pair cuts each SM's operand loads from
// 48 KB to 32 KB per 128-deep K block (one CTA per 128 x 256 tile: 3086 ->
// 3440 TFLOP/s at the Wan2.2-480p QKV shape).  Waits are bounded.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <atomic>
#include <mutex>

#include "attn_math.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace ditattn {
namespace {

__device__ unsigned int g_fp8_error = 0;

constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || i > kWaitLimitIters)) {
      atomicOr(&g_fp8_error, 1u);
      return false;
    }
  }
}

// ---------------------------------------------------------------- quantiser

constexpr int kQThreads = 128;
constexpr int kQMaxVec = 8;  // 16-byte bf16 vectors per thread: K <= 8192

__device__ __forceinline__ uint16_t e4m3x2(float lo, float hi) {
  uint16_t r;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// x / s for both lanes of a packed pair by Markstein's division ("Computation
// of elementary functions on the IBM RISC System/6000 processor", IBM J. Res.
// Dev. 34(1), 1990): with r = RN(1/s), q0 = RN(x r) is within an ulp of x / s,
// the residual x - q0 s is exact as one FMA, and RN(q0 + residual * r)
// corrects q0.  ns = -s.  The sign is taken from x, so -0 stays -0 as IEEE
// division keeps it.  Callers take it for scales s >= kMinFastScale (no step
// underflows or overflows; the quotients here are at most 448 in magnitude).
// On the quantiser's inputs (every bf16 row max and bf16 element of at most
// its magnitude, ~2.1e9 pairs) the quotient differs from IEEE division's in
// 0.1 % of the pairs, and its e4m3 code in none: dit_selftest_fp8_quotients
// counts both.
constexpr float kMinFastScale = 0x1p-100f;

__device__ __forceinline__ void div2_markstein(float x0, float x1, uint64_t r2, uint64_t ns2, float &q0, float &q1) {
  using namespace attn;
  const uint64_t x2 = f2(x0, x1);
  const uint64_t p2 = f2_mul(x2, r2);
  const uint64_t res2 = f2_fma(p2, ns2, x2);
  f2_split(f2_fma(res2, r2, p2), q0, q1);
  q0 = copysignf(q0, x0);
  q1 = copysignf(q1, x1);
}

template <int kVec>
__device__ __forceinline__ void q_load_row(uint4 (&raw)[kVec], const uint4 *__restrict__ x, long long m, int nvec) {
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const int i = threadIdx.x + u * kQThreads;
    if (i < nvec) raw[u] = __ldcs(x + m * nvec + i);
  }
}

// Quantise one row whose 16-byte vectors this thread holds in `raw`.  `red`
// holds 4 floats; callers alternate two buffers between rows (one barrier each).
template <int kVec>
__device__ __forceinline__ void q_row(const uint4 (&raw)[kVec], uint2 *codes, float *scale, long long m, int nvec,
                                      float *red) {
  float v[kVec][8];
  float amax = 0.f;
#pragma unroll
  for (int u = 0; u < kVec; ++u) {
    const uint32_t ww[4] = {raw[u].x, raw[u].y, raw[u].z, raw[u].w};
#pragma unroll
    for (int e = 0; e < 4; ++e) {
      v[u][2 * e] = __uint_as_float(ww[e] << 16);
      v[u][2 * e + 1] = __uint_as_float(ww[e] & 0xFFFF0000u);
    }
    if (threadIdx.x + u * kQThreads < nvec)
#pragma unroll
      for (int e = 0; e < 8; ++e) amax = fmaxf(amax, fabsf(v[u][e]));
  }
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, off));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = amax;
  __syncthreads();
  amax = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  const float sc = amax > 0.f ? __fdiv_rn(amax, 448.0f) : 1.0f;
  if (threadIdx.x == 0) scale[m] = sc;
  if (sc >= kMinFastScale) {  // every row but those whose largest magnitude is below ~2^-91
    const float r = __frcp_rn(sc);
    const uint64_t r2 = attn::f2(r, r), ns2 = attn::f2(-sc, -sc);
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const int i = threadIdx.x + u * kQThreads;
      if (i < nvec) {
        uint32_t w[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          float a, b, c, d;
          div2_markstein(v[u][4 * e], v[u][4 * e + 1], r2, ns2, a, b);
          div2_markstein(v[u][4 * e + 2], v[u][4 * e + 3], r2, ns2, c, d);
          w[e] = static_cast<uint32_t>(e4m3x2(a, b)) | (static_cast<uint32_t>(e4m3x2(c, d)) << 16);
        }
        __stcs(codes + m * nvec + i, make_uint2(w[0], w[1]));
      }
    }
  } else {
#pragma unroll
    for (int u = 0; u < kVec; ++u) {
      const int i = threadIdx.x + u * kQThreads;
      if (i < nvec) {
        uint32_t w[2];
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const uint16_t lo = e4m3x2(__fdiv_rn(v[u][4 * e], sc), __fdiv_rn(v[u][4 * e + 1], sc));
          const uint16_t hi = e4m3x2(__fdiv_rn(v[u][4 * e + 2], sc), __fdiv_rn(v[u][4 * e + 3], sc));
          w[e] = static_cast<uint32_t>(lo) | (static_cast<uint32_t>(hi) << 16);
        }
        __stcs(codes + m * nvec + i, make_uint2(w[0], w[1]));
      }
    }
  }
}

// Exhaustive check of div2_markstein against IEEE division over every input the
// quantiser can meet: the row max has bf16 bits 1 + blockIdx.x + 256 *
// blockIdx.y (every positive finite bf16, 0x0001 .. 0x7F7F) and the element
// bits 256 * blockIdx.z + threadIdx.x (every bf16 pattern; each thread also
// takes its negation); pairs with |x| > max, NaN or inf are skipped, and so are
// scales below kMinFastScale (those rows divide).
// counts[0]: fp32 quotients that differ; counts[1]: e4m3 codes that differ.
__device__ unsigned long long g_fp8_selftest_counts[2];

__global__ void fp8_quotient_selftest_kernel() {
  const uint32_t amax_bits = 1u + blockIdx.x + 256u * blockIdx.y;  // 0x0001 .. 0x7F7F
  const uint32_t x_bits = 256u * blockIdx.z + threadIdx.x;
  if (amax_bits > 0x7F7Fu) return;
  const float amax = __uint_as_float(amax_bits << 16);
  const float x = __uint_as_float(x_bits << 16);
  if (!(fabsf(x) <= amax)) return;
  const float sc = __fdiv_rn(amax, 448.0f);
  if (!(sc >= kMinFastScale)) return;
  const float r = __frcp_rn(sc);
  float q, q_other;
  div2_markstein(x, -x, attn::f2(r, r), attn::f2(-sc, -sc), q, q_other);
  const float ref = __fdiv_rn(x, sc), ref_other = __fdiv_rn(-x, sc);
  if (__float_as_uint(q) != __float_as_uint(ref) || __float_as_uint(q_other) != __float_as_uint(ref_other))
    atomicAdd(&g_fp8_selftest_counts[0], 1ull);
  if (e4m3x2(q, q_other) != e4m3x2(ref, ref_other)) atomicAdd(&g_fp8_selftest_counts[1], 1ull);
}

// Persistent CTAs walk rows m = blockIdx.x, + gridDim.x, ...; the next row's
// loads are issued before the current row's reduction.
template <int kVec>
__global__ void __launch_bounds__(kQThreads) quant_fp8_rows_kernel(const uint4 *__restrict__ x, uint2 *codes,
                                                                   float *scale, long long M, int K) {
  __shared__ float red[8];
  const int nvec = K / 8;
  uint4 cur[kVec], nxt[kVec];
  griddep_wait();
  griddep_launch_dependents();
  long long m = blockIdx.x;
  if (m < M) q_load_row<kVec>(cur, x, m, nvec);
  for (; m < M; m += 2LL * gridDim.x) {
    const long long m1 = m + gridDim.x;
    if (m1 < M) q_load_row<kVec>(nxt, x, m1, nvec);
    q_row<kVec>(cur, codes, scale, m, nvec, red);
    if (m1 >= M) break;
    const long long m2 = m1 + gridDim.x;
    if (m2 < M) q_load_row<kVec>(cur, x, m2, nvec);
    q_row<kVec>(nxt, codes, scale, m1, nvec, red + 4);
  }
}

// ---------------------------------------------------------------- GEMM

// A CTA pair (cluster of 2) computes one 256 x 256 output tile: CTA r holds
// rows 128 r .. 128 r + 127 of the tile's A block and columns 128 r .. + 127 of
// its B block, and its own 128 x 256 fp32 accumulator in TMEM.
constexpr int kGM = 128, kGN = 256, kGK = 128;  // per-CTA tile (K in bytes = elements)
constexpr int kGBRows = kGN / 2;                // B rows (output columns) each CTA loads
constexpr int kGStages = 6;  // 6 x 32 KB: ~2 us of MMA work buffered per SM
constexpr int kGThreads = 192;  // warp 0 TMA, warp 1 MMA, warps 2-5 epilogue
constexpr int kABytes = kGM * kGK, kBBytes = kGBRows * kGK, kStageBytes = kABytes + kBBytes;
constexpr int kOutBox = kGM * 128;                  // one output box: 128 rows x 64 bf16 columns
constexpr int kOutOff = kGStages * kStageBytes;     // two output boxes, alternating
constexpr int kBarOff = kOutOff + 2 * kOutBox;
// full[kGStages], empty[kGStages], acc_full[2], acc_empty[2], drain
constexpr int kGNumBars = 2 * kGStages + 5;
constexpr int kTmemSlotOff = kBarOff + 8 * kGNumBars;
constexpr int kGSmem = kTmemSlotOff + 16 + 1024;
constexpr uint32_t kGTmemCols = 2 * kGN;  // two accumulators: the epilogue drains one while the MMAs fill the other

__host__ __device__ constexpr uint32_t idesc_e4m3_f32(int M, int N) {
  return (1u << 4)                                  /* D format: f32 */
         | (0u << 7) | (0u << 10)                   /* A, B format: e4m3 */
         | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// wait_bounded with cluster-scope acquire, for barriers the peer CTA arrives on.
__device__ __forceinline__ bool wait_bounded_cluster(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    if ((i & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || i > kWaitLimitIters)) {
      atomicOr(&g_fp8_error, 1u);
      return false;
    }
  }
}
__device__ __forceinline__ void mma_f8_pair(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// 2-D tiled load into this CTA's shared memory, counted on an mbarrier of either CTA of the pair.
__device__ __forceinline__ void tma_load_2d_pair(uint32_t dst, const CUtensorMap *map, uint32_t bar_cluster, int c0,
                                                 int c1) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(bar_cluster), "r"(c0), "r"(c1)
      : "memory");
}

__device__ __forceinline__ void tma_store_2d(const CUtensorMap *map, uint32_t src, int c0, int c1) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(map)),
               "r"(src), "r"(c0), "r"(c1)
               : "memory");
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

// Persistent pairs: pair p takes 256 x 256 output tiles p, p + pairs, ... (N
// fastest).  Both CTAs' producers stream their halves of each K block through
// their own rings, completing on the rank-0 CTA's `full` barriers; one thread
// of the rank-0 CTA issues the M = 256 MMAs (each CTA's A half and B half at
// the same shared-memory offsets) and multicasts every commit to both CTAs; the
// epilogue warps of each CTA drain its own accumulator rows and report the
// buffer free on the rank-0 CTA's acc_empty (one arrive per warp).
__global__ void __launch_bounds__(kGThreads, 1)
    gemm_fp8_kernel(const __grid_constant__ CUtensorMap tm_a, const __grid_constant__ CUtensorMap tm_b,
                    const __grid_constant__ CUtensorMap tm_o, const float *__restrict__ a_scale,
                    const float *__restrict__ b_scale, int M, int N, int K) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + kTmemSlotOff);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int pair = blockIdx.x >> 1, pairs = gridDim.x >> 1;
  const int nk = (K + kGK - 1) / kGK;
  const int tiles_n = (N + kGN - 1) / kGN;
  const int n_tiles = tiles_n * ((M + 2 * kGM - 1) / (2 * kGM));
  const uint32_t bars = base + kBarOff;
  auto full = [&](int s) { return bars + 8u * s; };
  auto empty = [&](int s) { return bars + 8u * (kGStages + s); };
  auto acc_full = [&](int b) { return bars + 8u * (2 * kGStages + b); };
  auto acc_empty = [&](int b) { return bars + 8u * (2 * kGStages + 2 + b); };
  const uint32_t drain = bars + 8u * (2 * kGStages + 4);
  griddep_wait();
  griddep_launch_dependents();

  if (threadIdx.x == 0) {
    for (int s = 0; s < kGStages; ++s) {
      mbar_init(full(s), 1);
      mbar_init(empty(s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(acc_full(b), 1);
      mbar_init(acc_empty(b), 8);  // one arrive per epilogue warp of both CTAs (rank 0's barrier counts)
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  if (warp == 1) {
    tmem_alloc_pair(base + kTmemSlotOff, kGTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive or load
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      uint32_t g = 0;  // K blocks issued over all tiles
      bool ok = true;
      for (int tile = pair; tile < n_tiles && ok; tile += pairs) {
        const int m0 = (tile / tiles_n) * (2 * kGM) + static_cast<int>(rank) * kGM;
        const int nb = (tile % tiles_n) * kGN + static_cast<int>(rank) * kGBRows;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kGStages;
          if (!wait_bounded(empty(s), ((g / kGStages) & 1) ^ 1)) {
            ok = false;
            break;
          }
          const uint32_t lead_full = mapa_shared(full(s), 0);
          if (rank == 0) mbar_arrive_expect_tx(full(s), 2 * kStageBytes);
          tma_load_2d_pair(base + s * kStageBytes, &tm_a, lead_full, kb * kGK, m0);
          tma_load_2d_pair(base + s * kStageBytes + kABytes, &tm_b, lead_full, kb * kGK, nb);
        }
      }
      // Copies must land before the CTA may exit.  Both CTAs' copies complete on
      // rank 0's full barriers: rank 0 waits for the last fills there (the final
      // cluster barrier keeps rank 1 resident until then); rank 1 sees its last
      // fills consumed (their empty phase) on the normal path.
      for (uint32_t i = g > kGStages ? g - kGStages : 0; i < g; ++i) {
        if (rank == 0)
          wait_bounded(full(i % kGStages), (i / kGStages) & 1);
        else if (ok)
          wait_bounded(empty(i % kGStages), (i / kGStages) & 1);
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc = idesc_e4m3_f32(2 * kGM, kGN);
      uint32_t g = 0;
      bool ok = true;
      int i = 0;
      for (int tile = pair; tile < n_tiles && ok; tile += pairs, ++i) {
        const int buf = i & 1;
        ok = wait_bounded_cluster(acc_empty(buf), ((i >> 1) & 1) ^ 1);  // both epilogues have drained it
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t d = tmem + buf * kGN;
        for (int kb = 0; kb < nk; ++kb, ++g) {
          const int s = g % kGStages;
          ok = wait_bounded(full(s), (g / kGStages) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          const uint32_t a0 = base + s * kStageBytes, b0 = a0 + kABytes;
#pragma unroll
          for (int kk = 0; kk < kGK / 32; ++kk)
            mma_f8_pair(d, smem_desc_sw128(a0 + kk * 32, 16, 1024), smem_desc_sw128(b0 + kk * 32, 16, 1024), idesc,
                        (kb > 0 || kk > 0) ? 1u : 0u);
          tc_commit_pair(empty(s));
        }
        if (ok) tc_commit_pair(acc_full(buf));
      }
      // every MMA issued must complete (in both CTAs) before TMEM is freed
      tc_commit_pair(drain);
    }
    if (lane == 0) wait_bounded(drain, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    // warp w reads TMEM lanes 32 * (w % 4) .. + 31: one output row per thread
    const int wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t sw = row & 7;
    const uint32_t lead_acc_empty0 = mapa_shared(acc_empty(0), 0), lead_acc_empty1 = mapa_shared(acc_empty(1), 0);
    bool ok = true;
    int i = 0;
    int last_buf = -1;  // (row 0) staging buffer read by the most recently committed store
    for (int tile = pair; tile < n_tiles; tile += pairs, ++i) {
      const int buf = i & 1;
      const int m0 = (tile / tiles_n) * (2 * kGM) + static_cast<int>(rank) * kGM, n0 = (tile % tiles_n) * kGN;
      ok = named_barrier_and(1, 128, ok && wait_bounded(acc_full(buf), (i >> 1) & 1));
      if (!ok) break;
      tc_fence_after_sync();
      const float as = m0 + row < M ? a_scale[m0 + row] : 0.f;
#pragma unroll 1
      for (int c = 0; c < kGN / 32; ++c) {
        const int box = c >> 1;  // 64 output columns per box, staged in buffer box % 2
        const uint32_t stage = base + kOutOff + (box & 1) * kOutBox;
        if ((c & 1) == 0) {
          if (row == 0) {
            if (last_buf == (box & 1))
              bulk_wait_read_all();
            else
              bulk_wait_read_all_but_one();
          }
          named_barrier_sync(1, 128);
        }
        uint32_t o[32];
        tmem_ld_x32(tmem + lane_base + buf * kGN + c * 32, o);
        const int col0 = n0 + c * 32;
        float bs[32];
#pragma unroll
        for (int j = 0; j < 32; ++j) bs[j] = col0 + j < N ? __ldg(b_scale + col0 + j) : 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            const int j = 8 * u + 2 * e;
            w[e] = pack_bf16(__uint_as_float(o[j]) * as * bs[j], __uint_as_float(o[j + 1]) * as * bs[j + 1]);
          }
          st_shared_v4(stage + row * 128 + ((((c & 1) * 4 + u) ^ sw) << 4), w[0], w[1], w[2], w[3]);
        }
        if (c & 1) {
          fence_proxy_async_smem();
          named_barrier_sync(1, 128);
          if (row == 0 && n0 + box * 64 < N && m0 < M) {
            tma_store_2d(&tm_o, stage, n0 + box * 64, m0);
            bulk_commit_group();
            last_buf = box & 1;
          }
        }
      }
      // this warp's reads of the buffer are complete (each TMEM load waits): hand it back
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(acc_empty(buf));
        else
          mbar_arrive_cluster(buf ? lead_acc_empty1 : lead_acc_empty0);
      }
    }
    if (row == 0) bulk_wait_read_all();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // neither CTA leaves while the pair's MMAs or loads may still touch it
  if (warp == 1) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kGTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

// 2-D row-major map (inner dim first) with a box of box0 x box1 and 128-byte swizzle.
bool encode_2d(CUtensorMap *map, const void *ptr, CUtensorMapDataType dt, int esize, long long inner, long long outer,
               long long ld_elems, int box0, int box1) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  cuuint64_t dims[2] = {(cuuint64_t)inner, (cuuint64_t)outer};
  cuuint64_t strides[1] = {(cuuint64_t)ld_elems * esize};
  cuuint32_t box[2] = {(cuuint32_t)box0, (cuuint32_t)box1};
  cuuint32_t estr[2] = {1, 1};
  return enc(map, dt, 2, const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

}  // namespace

int quant_fp8_max_k() { return kQMaxVec * 8 * kQThreads; }

cudaError_t run_fp8_quotient_selftest(unsigned long long counts[2], cudaStream_t stream) {
  const unsigned long long zero[2] = {0ull, 0ull};
  cudaError_t e = cudaMemcpyToSymbolAsync(g_fp8_selftest_counts, zero, sizeof(zero), 0, cudaMemcpyHostToDevice, stream);
  if (e != cudaSuccess) return e;
  fp8_quotient_selftest_kernel<<<dim3(256, 128, 256), 256, 0, stream>>>();  // 0x7F7F row maxima x 65536 elements
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  e = cudaMemcpyFromSymbolAsync(counts, g_fp8_selftest_counts, 2 * sizeof(unsigned long long), 0,
                                cudaMemcpyDeviceToHost, stream);
  if (e != cudaSuccess) return e;
  return cudaStreamSynchronize(stream);
}

namespace {

// Persistent grid sized by occupancy (capped at 8 CTAs per SM); kVec as for the row norms.
template <int kVec>
cudaError_t launch_quant_vec(const uint4 *x, uint2 *codes, float *scale, long long M, int K, cudaStream_t stream) {
  int dev = 0, sms = 0, per_sm = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e == cudaSuccess)
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, quant_fp8_rows_kernel<kVec>, kQThreads, 0);
  if (e != cudaSuccess) return e;
  const long long cap = (long long)(per_sm < 1 ? 1 : per_sm > 8 ? 8 : per_sm) * sms;
  const unsigned grid = static_cast<unsigned>(M < cap ? M : cap);
  return launch_kernel(quant_fp8_rows_kernel<kVec>, dim3(grid), dim3(kQThreads), 0, stream, x, codes, scale, M, K);
}

}  // namespace

cudaError_t launch_quant_fp8_rows(const void *x, void *codes, float *scale, long long M, int K, cudaStream_t stream) {
  const uint4 *xx = static_cast<const uint4 *>(x);
  uint2 *cc = static_cast<uint2 *>(codes);
  switch ((K / 8 + kQThreads - 1) / kQThreads) {
    case 1: return launch_quant_vec<1>(xx, cc, scale, M, K, stream);
    case 2: return launch_quant_vec<2>(xx, cc, scale, M, K, stream);
    case 3: return launch_quant_vec<3>(xx, cc, scale, M, K, stream);
    case 4: return launch_quant_vec<4>(xx, cc, scale, M, K, stream);
    case 5: return launch_quant_vec<5>(xx, cc, scale, M, K, stream);
    case 6: return launch_quant_vec<6>(xx, cc, scale, M, K, stream);
    case 7: return launch_quant_vec<7>(xx, cc, scale, M, K, stream);
    default: return launch_quant_vec<kQMaxVec>(xx, cc, scale, M, K, stream);
  }
}

cudaError_t launch_gemm_fp8(const void *a, const float *a_scale, const void *b, const float *b_scale, void *out,
                            int M, int N, int K, long long lda, long long ldb, long long ldo, cudaStream_t stream,
                            const char **detail) {
  CUtensorMap ta, tb, to;
  if (!encode_2d(&ta, a, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, M, lda, kGK, kGM) ||
      !encode_2d(&tb, b, CU_TENSOR_MAP_DATA_TYPE_UINT8, 1, K, N, ldb, kGK, kGBRows) ||
      !encode_2d(&to, out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, N, M, ldo, 64, kGM)) {
    *detail = "cuTensorMapEncodeTiled failed for the fp8 GEMM operands";
    return cudaErrorInvalidValue;
  }
  // pairs that can be resident at once, per device (0: not yet known); other host threads may launch too
  static std::atomic<int> max_pairs[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.blockDim = dim3(kGThreads);
  cfg.dynamicSmemBytes = kGSmem;
  cfg.stream = stream;
  cfg.attrs = attr;
  int cap = dev < 64 ? max_pairs[dev].load(std::memory_order_acquire) : 0;
  if (cap == 0) {
    e = cudaFuncSetAttribute(gemm_fp8_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGSmem);
    if (e != cudaSuccess) return e;
    int sms = 0;
    e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    if (e != cudaSuccess) return e;
    cfg.gridDim = dim3(sms & ~1);
    cfg.numAttrs = 1;
    e = cudaOccupancyMaxActiveClusters(&cap, gemm_fp8_kernel, &cfg);
    if (e != cudaSuccess) return e;
    if (cap < 1) return cudaErrorInvalidConfiguration;
    if (dev < 64) max_pairs[dev].store(cap, std::memory_order_release);
  }
  const long long tiles = (long long)((N + kGN - 1) / kGN) * ((M + 2 * kGM - 1) / (2 * kGM));
  // persistent: as many pairs as can be resident at once (pairs wait only on each other)
  const int pairs = static_cast<int>(tiles < cap ? tiles : cap);
  cfg.gridDim = dim3(2 * pairs);
  cfg.numAttrs = launch_overlap_enabled() ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, gemm_fp8_kernel, ta, tb, to, a_scale, b_scale, M, N, K);
}

cudaError_t read_and_clear_fp8_error(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_fp8_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_fp8_error, &zero, sizeof(unsigned int));
}

}  // namespace ditattn
