// Non-causal flash attention forward for GB300 (sm_103a): O and fp32 LSE over a key range.
//
// Operation (the DiT attention of "NPU Wan2.2-I2V model inference optimisation
// practice", section "NPU npu_fused_infer_attention_score operator adaptation",
// non-causal, whose second output is the log-sum-exp; the key-range form is the
// per-block attention of the ring / gather sequence-parallel paths in "feat:
// support Ascend NPU backend (torch_npu) for Qwen-Image pipelines - #274", item 2):
//   s_j = scale * q . k_j  for j in [kv_begin, kv_end)
//   O   = sum_j softmax(s)_j v_j,   LSE = ln sum_j exp(s_j)
//
// Design (one CTA = 256 query rows of one (b, h), warp specialised):
//   warp 8      TMA producer: Q tiles once, then K_j / V_j blocks of 128 keys
//               into a ring of shared-memory slots (128-byte swizzle).
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (SS form),
//               O_t += P_t V_j with P read from TMEM (TS form).  Two query
//               tiles t = 0, 1 alternate so the tensor core always has one
//               tile's work while the other tile's softmax runs.
//   warps 0-7   two softmax warpgroups, one per query tile; thread = one query
//               row (TMEM lane), so row max / row sum need no shuffles.  Online
//               softmax in base 2 with the scale folded into one FFMA; the O
//               rescale is lazy (only when a row max grows by more than 2^8),
//               exact after the final 1/l.  P is written back over S in TMEM
//               as bf16.  Epilogue: O / l from TMEM to global, LSE = (m + log2 l) ln 2.
// TMEM (512 columns): S/P of tile 0 | S/P of tile 1 | O of tile 0 | O of tile 1.
// Every mbarrier wait is bounded (about 2 s); a wait that gives up sets the
// library's device error word and the CTA drains its in-flight copies and MMAs,
// frees TMEM and exits.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "internal.h"
#include "sm100_ptx.cuh"

namespace ditattn {

__device__ unsigned int g_device_error = 0;

namespace {

constexpr int kBM = 128;            // query rows per tile (MMA M)
constexpr int kBN = 128;            // keys per block (MMA N of S, K of PV)
constexpr int kNQ = 2;              // query tiles per CTA
constexpr int kSlots = 4;           // K/V shared-memory ring slots
constexpr int kThreads = 320;       // 8 softmax warps + TMA warp + MMA warp
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;  // lazy-rescale threshold on the running max (base-2 units)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr unsigned int kErrWaitTimeout = 1u;

template <int D>
struct Layout {
  static constexpr int kBox = 128 * 128;     // one TMA box: 128 rows x 128 bytes (64 bf16)
  static constexpr int kTile = 128 * D * 2;  // one Q tile or one K / V block
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kNQ * kTile;
  static constexpr int kBar = kKV + kSlots * kTile;
  // q_full, slot_full[kSlots], slot_empty[kSlots], s_full[kNQ], p_full[kNQ], o_done[kNQ], drain
  static constexpr int kNumBars = 1 + 2 * kSlots + 3 * kNQ + 1;
  static constexpr int kTmemSlot = kBar + 8 * kNumBars;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
  static constexpr uint32_t kTmemO = 2 * kBN;   // first O column
};

struct AttnArgs {
  int H, Sq, n_kv;
  float scale_log2;
  void *o;
  long long o_sb, o_ss, o_sh;
  int o_f32;
  float *lse;
};

// Bounded wait; false (and the device error word set) if the phase did not complete in time.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && global_timer_ns() - t0 > kWaitLimitNs) {
      atomicOr(&g_device_error, kErrWaitTimeout);
      return false;
    }
  }
}

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float lo, float hi) {
  __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t *>(&v);
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const AttnArgs args) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + L::kTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = blockIdx.x * (kBM * kNQ);
  const int nblk = (args.n_kv + kBN - 1) / kBN;

  const uint32_t bars = base + L::kBar;
  const uint32_t q_full = bars;
  auto slot_full = [&](int s) { return bars + 8u * (1 + s); };
  auto slot_empty = [&](int s) { return bars + 8u * (1 + kSlots + s); };
  auto s_full = [&](int t) { return bars + 8u * (1 + 2 * kSlots + t); };
  auto p_full = [&](int t) { return bars + 8u * (1 + 2 * kSlots + kNQ + t); };
  auto o_done = [&](int t) { return bars + 8u * (1 + 2 * kSlots + 2 * kNQ + t); };
  const uint32_t drain = bars + 8u * (1 + 2 * kSlots + 3 * kNQ);

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int t = 0; t < kNQ; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 128);
      mbar_init(o_done(t), 1);
    }
    mbar_init(drain, 1);
    mbar_fence_init();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
  }
  if (warp == kWarpMma) {
    tmem_alloc(base + L::kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, kNQ * L::kTile);
      for (int t = 0; t < kNQ; ++t)
        for (int hf = 0; hf < D / 64; ++hf)
          tma_load_4d(base + L::kQ + t * L::kTile + hf * L::kBox, &tm_q, q_full, hf * 64, h, q0 + t * kBM, b);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        for (int which = 0; which < 2; ++which) {  // 0: K_j, 1: V_j
          const int i = 2 * j + which, slot = i % kSlots;
          if (!wait_bounded(slot_empty(slot), ((i / kSlots) & 1) ^ 1)) {
            ok = false;
            break;
          }
          mbar_arrive_expect_tx(slot_full(slot), L::kTile);
          const uint32_t dst = base + L::kKV + slot * L::kTile;
          for (int hf = 0; hf < D / 64; ++hf)
            tma_load_4d(dst + hf * L::kBox, which ? &tm_v : &tm_k, slot_full(slot), hf * 64, h, j * kBN, b);
          ++issued;
        }
      }
      // Every copy issued must land before the CTA may exit.
      wait_bounded(q_full, 0);
      for (int i = issued > kSlots ? issued - kSlots : 0; i < issued; ++i)
        wait_bounded(slot_full(i % kSlots), (i / kSlots) & 1);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 1);
      auto issue_s = [&](int t, int slot) {  // S_t = Q_t K^T, K-major A and B
        const uint32_t a0 = base + L::kQ + t * L::kTile, b0 = base + L::kKV + slot * L::kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * L::kBox + (kk & 3) * 32;
          mma_ss(tmem + t * kBN, smem_desc_sw128(a0 + off, 16, 1024), smem_desc_sw128(b0 + off, 16, 1024), idesc_s,
                 kk > 0);
        }
      };
      auto issue_o = [&](int t, int slot, bool acc) {  // O_t += P_t V, P in TMEM, V MN-major
        const uint32_t v0 = base + L::kKV + slot * L::kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts(tmem + L::kTmemO + t * D, tmem + t * kBN + kk * 8, smem_desc_sw128(v0 + kk * 2048, L::kBox, 1024),
                 idesc_o, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_bounded(q_full, 0) && wait_bounded(slot_full(0), 0);
      if (ok) {
        tc_fence_after_sync();
        for (int t = 0; t < kNQ; ++t) {
          issue_s(t, 0);
          tc_commit(s_full(t));
        }
        tc_commit(slot_empty(0));
      }
      for (int j = 0; j < nblk && ok; ++j) {
        const int iv = 2 * j + 1, ik = 2 * j + 2;
        const bool next = j + 1 < nblk;
        ok = wait_bounded(slot_full(iv % kSlots), (iv / kSlots) & 1);
        if (ok && next) ok = wait_bounded(slot_full(ik % kSlots), (ik / kSlots) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        for (int t = 0; t < kNQ && ok; ++t) {
          ok = wait_bounded(p_full(t), j & 1);
          if (!ok) break;
          tc_fence_after_sync();
          issue_o(t, iv % kSlots, j > 0);
          if (next) {
            issue_s(t, ik % kSlots);
            tc_commit(s_full(t));
          }
        }
        if (!ok) break;
        tc_commit(slot_empty(iv % kSlots));
        if (next) tc_commit(slot_empty(ik % kSlots));
      }
      if (ok)
        for (int t = 0; t < kNQ; ++t) tc_commit(o_done(t));
      // Every MMA issued must complete before TMEM is freed.
      tc_commit(drain);
      wait_bounded(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * kBN;
    const uint32_t tO = tmem + lane_base + L::kTmemO + t * D;
    const float sl2 = args.scale_log2;
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(s_full(t), j & 1));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sr[128];
      tmem_ld_x128(tS, sr);
      float s[128];
#pragma unroll
      for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(sr[i]);
      const int valid = args.n_kv - j * kBN;
      if (valid < kBN) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      // row max as 8 independent chains and a tree (a single chain is ~127 dependent fmax)
      float mp[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) mp[u] = s[u];
#pragma unroll
      for (int i = 8; i < kBN; i += 8)
#pragma unroll
        for (int u = 0; u < 8; ++u) mp[u] = fmaxf(mp[u], s[i + u]);
      float mx = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])), fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      mx *= sl2;
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, mx > m + kRescaleLog2)) {
        // The previous PV product of this tile is complete: S_t for block j was
        // issued after it and its commit covers every earlier MMA.
        const float m_new = fmaxf(m, mx);
        const float alpha = ex2(m - m_new);
        m = m_new;
        l *= alpha;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(tO + c * 32, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_x32(tO + c * 32, o);
        }
        tmem_st_wait();
      }
      const float nm = -m;
      float rp[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};  // row-sum partials (independent chains)
      uint32_t p0[32], p1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float a = ex2(fmaf(s[2 * i], sl2, nm)), c = ex2(fmaf(s[2 * i + 1], sl2, nm));
        rp[i & 7] += a + c;
        p0[i] = pack_bf16(a, c);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float a = ex2(fmaf(s[64 + 2 * i], sl2, nm)), c = ex2(fmaf(s[64 + 2 * i + 1], sl2, nm));
        rp[i & 7] += a + c;
        p1[i] = pack_bf16(a, c);
      }
      l += ((rp[0] + rp[1]) + (rp[2] + rp[3])) + ((rp[4] + rp[5]) + (rp[6] + rp[7]));
      tmem_st_x32(tS, p0);
      tmem_st_x32(tS + 32, p1);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(p_full(t));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(o_done(t), 0));
    if (ok) {
      tc_fence_after_sync();
      const int q = q0 + t * kBM + row;
      const bool live = q < args.Sq;
      const float inv_l = 1.0f / l;
      const long long off = (long long)b * args.o_sb + (long long)q * args.o_ss + (long long)h * args.o_sh;
#pragma unroll
      for (int c = 0; c < D / 32; ++c) {
        uint32_t o[32];
        tmem_ld_x32(tO + c * 32, o);
        if (live) {
          if (args.o_f32) {
            float4 *dst = reinterpret_cast<float4 *>(static_cast<float *>(args.o) + off + c * 32);
#pragma unroll
            for (int i = 0; i < 8; ++i)
              dst[i] = make_float4(__uint_as_float(o[4 * i]) * inv_l, __uint_as_float(o[4 * i + 1]) * inv_l,
                                   __uint_as_float(o[4 * i + 2]) * inv_l, __uint_as_float(o[4 * i + 3]) * inv_l);
          } else {
            uint4 *dst = reinterpret_cast<uint4 *>(static_cast<__nv_bfloat16 *>(args.o) + off + c * 32);
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              uint4 v;
              v.x = pack_bf16(__uint_as_float(o[8 * i + 0]) * inv_l, __uint_as_float(o[8 * i + 1]) * inv_l);
              v.y = pack_bf16(__uint_as_float(o[8 * i + 2]) * inv_l, __uint_as_float(o[8 * i + 3]) * inv_l);
              v.z = pack_bf16(__uint_as_float(o[8 * i + 4]) * inv_l, __uint_as_float(o[8 * i + 5]) * inv_l);
              v.w = pack_bf16(__uint_as_float(o[8 * i + 6]) * inv_l, __uint_as_float(o[8 * i + 7]) * inv_l);
              dst[i] = v;
            }
          }
        }
      }
      if (live) args.lse[((long long)b * args.H + h) * args.Sq + q] = (m + log2f(l)) * 0.69314718055994531f;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

// bf16 [B, S, H, D] with element strides {b, s, h}, as a 4-D map (d, h, s, b),
// box 64 x 1 x 128 x 1, 128-byte swizzle; rows past S read as zero.
bool encode_bshd(CUtensorMap *map, const void *ptr, int B, int S, int H, int D, const int64_t st[3]) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * 2, (cuuint64_t)st[1] * 2, (cuuint64_t)st[0] * 2};
  cuuint32_t box[4] = {64, 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void *>(ptr), dims, strides, box, estr,
                   CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                   CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const AttnArgs &a,
                         int B, cudaStream_t stream) {
  using Lay = Layout<D>;
  static_assert(Lay::kAlloc <= 232448, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, Lay::kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  dim3 grid((a.Sq + kBM * kNQ - 1) / (kBM * kNQ), a.H, B);
  attn_fwd_kernel<D><<<grid, kThreads, Lay::kAlloc, stream>>>(tq, tk, tv, a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                            const int64_t q_st[3], const int64_t kv_st[3], float scale, int kv_begin, int kv_end,
                            void *o, bool o_f32, const int64_t o_st[3], float *lse, cudaStream_t stream,
                            const char **detail) {
  (void)Skv;
  CUtensorMap tq, tk, tv;
  const int n_kv = kv_end - kv_begin;
  const char *k0 = static_cast<const char *>(k) + (int64_t)kv_begin * kv_st[1] * 2;
  const char *v0 = static_cast<const char *>(v) + (int64_t)kv_begin * kv_st[1] * 2;
  if (!encode_bshd(&tq, q, B, Sq, H, D, q_st) || !encode_bshd(&tk, k0, B, n_kv, H, D, kv_st) ||
      !encode_bshd(&tv, v0, B, n_kv, H, D, kv_st)) {
    *detail = "cuTensorMapEncodeTiled failed (driver entry point missing or strides/extents unsupported)";
    return cudaErrorInvalidValue;
  }
  AttnArgs a;
  a.H = H;
  a.Sq = Sq;
  a.n_kv = n_kv;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.o = o;
  a.o_sb = o_st[0];
  a.o_ss = o_st[1];
  a.o_sh = o_st[2];
  a.o_f32 = o_f32 ? 1 : 0;
  a.lse = lse;
  if (D == 64) return launch_typed<64>(tq, tk, tv, a, B, stream);
  return launch_typed<128>(tq, tk, tv, a, B, stream);
}

cudaError_t read_and_clear_device_error(cudaStream_t stream, unsigned int *value) {
  cudaError_t e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return e;
  unsigned int zero = 0;
  e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace ditattn
