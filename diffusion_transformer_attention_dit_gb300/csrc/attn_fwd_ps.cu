// Flash attention forward for GB300, head dim 128, with P in shared memory: the
// same operation, outputs, causal mask, key-range and update forms as
// attn_fwd.cu (see there for the definition and its sources).
//
// Why: in attn_fwd.cu, P is written back over S in TMEM, so S of block j + 1
// can only be computed after block j's O += P V has read P.  Each query tile
// then runs S (512 tensor cycles) -> softmax (~1300 cycles) -> P V (512) -> S
// in series, and two interleaved tiles keep the tensor core ~70 % busy.  Here
// the softmax writes P (bf16, 128-byte swizzled) to shared memory and O += P V
// takes both operands from shared memory, so S of block j + 1 is issued as soon
// as the softmax has read S of block j into registers: the next S overlaps the
// softmax instead of following the product.
//
// Shared memory (224 KB): Q tiles 2 x 32 KB | P tiles 2 x 32 KB | K/V ring of
// three 32 KB slots, filled K_0, K_1, V_0, K_2, V_1, ... V_(n-1): each K is
// needed one step before its V (S of block j + 1 is issued before P V of block
// j), so the K a step needs was requested two steps earlier.  TMEM: S0 S1 O0 O1.
// Barriers per tile t: s_full (S_t ready), s_free (the softmax has read S_t),
// p_full (P_t written), pv_done (O_t += P_t V complete: P_t may be rewritten and
// O_t rescaled), o_done.  Each completes once per block and is waited for one
// phase behind at most, so every parity wait has a single pending phase.
// Roles: warps 0-7 softmax (tile t = w / 4, thread = query row = TMEM lane),
// warp 8 TMA producer, warp 9 MMA issuer.  Every wait is bounded.

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <mutex>

#include "attn_math.cuh"
#include "internal.h"
#include "sm100_ptx.cuh"

namespace ditattn {
namespace {

using namespace attn;

__device__ unsigned int g_ps_error = 0;

constexpr int D = 128;
constexpr int kBM = 128;
constexpr int kBN = 128;
constexpr int kNQ = 2;
constexpr int kSlots = 3;
constexpr int kThreads = 320;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;

constexpr int kBox = 128 * 128;  // TMA box: 128 rows x 128 bytes
constexpr int kTile = kBM * D * 2;  // 32 KB: a Q tile, a P tile or a K / V block
constexpr int kQ = 0;
constexpr int kP = kQ + kNQ * kTile;
constexpr int kKV = kP + kNQ * kTile;
constexpr int kBar = kKV + kSlots * kTile;
// q_full, slot_full[3], slot_empty[3], s_full[2], s_free[2], p_full[2], pv_done[2], o_done[2], drain, acc_full
constexpr int kNumBars = 1 + 2 * kSlots + 5 * kNQ + 2;
constexpr int kTmemSlot = kBar + 8 * kNumBars;
constexpr int kAlloc = kTmemSlot + 16 + 1024;
constexpr uint32_t kTmemO = 2 * kBN;
static_assert(kAlloc <= 232448, "shared memory budget");

// Ring fill index of K_m and V_m (n blocks): K_0, K_1, V_0, K_2, V_1, ..., K_(n-1), V_(n-2), V_(n-1).
__host__ __device__ __forceinline__ int fill_k(int m) { return m == 0 ? 0 : 2 * m - 1; }
__host__ __device__ __forceinline__ int fill_v(int m, int n) { return m <= n - 2 ? 2 * m + 2 : 2 * n - 1; }

struct PsArgs {
  int H, Sq, n_kv;
  int kv_begin;
  float scale_log2;
  int o_f32;
  float *lse;
  const float *lse_acc;
  int acc_f32;
};

__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || i > kWaitLimitIters)) {
      atomicOr(&g_ps_error, 1u);
      return false;
    }
  }
}

template <bool kCausal, bool kUpdate>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_ps_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                       const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                       const __grid_constant__ CUtensorMap tm_acc, const PsArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + kTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = blockIdx.x * (kBM * kNQ);
  int nblk = (args.n_kv + kBN - 1) / kBN;
  if (kCausal) {
    const int q_last = min(q0 + kBM * kNQ, args.Sq) - 1;
    const int reach = q_last - args.kv_begin + 1;  // keys of the range visible to the last row
    nblk = max(1, min(nblk, (reach + kBN - 1) / kBN));
  }
  // update form: query tile t's running O (32 KB bf16 or 64 KB fp32) is loaded, once the last products are
  // done, into the P tiles and ring slots, which form one contiguous region from kP
  const int acc_tile = kUpdate ? (args.acc_f32 ? 2 * kTile : kTile) : 0;
  griddep_wait();
  griddep_launch_dependents();

  const uint32_t bars = base + kBar;
  const uint32_t q_full = bars;
  auto slot_full = [&](int s) { return bars + 8u * (1 + s); };
  auto slot_empty = [&](int s) { return bars + 8u * (1 + kSlots + s); };
  auto s_full = [&](int t) { return bars + 8u * (1 + 2 * kSlots + t); };
  auto s_free = [&](int t) { return bars + 8u * (1 + 2 * kSlots + kNQ + t); };
  auto p_full = [&](int t) { return bars + 8u * (1 + 2 * kSlots + 2 * kNQ + t); };
  auto pv_done = [&](int t) { return bars + 8u * (1 + 2 * kSlots + 3 * kNQ + t); };
  auto o_done = [&](int t) { return bars + 8u * (1 + 2 * kSlots + 4 * kNQ + t); };
  const uint32_t drain = bars + 8u * (1 + 2 * kSlots + 5 * kNQ);
  const uint32_t acc_full = drain + 8;

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int t = 0; t < kNQ; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(s_free(t), 4);  // one arrive per softmax warp of the tile
      mbar_init(p_full(t), 4);
      mbar_init(pv_done(t), 1);
      mbar_init(o_done(t), 1);
    }
    mbar_init(drain, 1);
    mbar_init(acc_full, 1);
    mbar_fence_init();
  }
  if (warp == kWarpTma && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    tma_prefetch_map(&tm_o);
    if (kUpdate) tma_prefetch_map(&tm_acc);
  }
  if (warp == kWarpMma) {
    tmem_alloc(base + kTmemSlot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      mbar_arrive_expect_tx(q_full, kNQ * kTile);
      for (int t = 0; t < kNQ; ++t)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_4d(base + kQ + t * kTile + hf * kBox, &tm_q, q_full, hf * 64, h, q0 + t * kBM, b);
      int issued = 0;
      bool ok = true;
      for (int i = 0; i < 2 * nblk && ok; ++i) {
        // fill i: K_0, then K_(i+1)/2 for odd i, V_(i/2 - 1) for even i, and V_(n-1) last
        bool is_v;
        int blk;
        if (i == 0) {
          is_v = false, blk = 0;
        } else if (i == 2 * nblk - 1) {
          is_v = true, blk = nblk - 1;
        } else if (i & 1) {
          is_v = false, blk = (i + 1) / 2;
        } else {
          is_v = true, blk = i / 2 - 1;
        }
        const int slot = i % kSlots;
        if (!wait_bounded(slot_empty(slot), ((i / kSlots) & 1) ^ 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(slot_full(slot), kTile);
        const uint32_t dst = base + kKV + slot * kTile;
        for (int hf = 0; hf < 2; ++hf)
          tma_load_4d(dst + hf * kBox, is_v ? &tm_v : &tm_k, slot_full(slot), hf * 64, h, blk * kBN, b);
        ++issued;
      }
      bool acc_issued = false;
      if (kUpdate && ok) {
        // every product is done with the P tiles and the ring once both tiles' last P V has completed
        ok = wait_bounded(o_done(0), 0) && wait_bounded(o_done(1), 0);
        if (ok) {
          const int per_box = args.acc_f32 ? 32 : 64;  // columns per 16 KB box
          const int boxes = acc_tile / kBox;
          mbar_arrive_expect_tx(acc_full, kNQ * acc_tile);
          for (int t = 0; t < kNQ; ++t)
            for (int bx = 0; bx < boxes; ++bx)
              tma_load_4d(base + kP + t * acc_tile + bx * kBox, &tm_acc, acc_full, bx * per_box, h, q0 + t * kBM,
                          b);
          acc_issued = true;
        }
      }
      // every copy issued must land before the CTA may exit
      wait_bounded(q_full, 0);
      for (int i = issued > kSlots ? issued - kSlots : 0; i < issued; ++i)
        wait_bounded(slot_full(i % kSlots), (i / kSlots) & 1);
      if (acc_issued) wait_bounded(acc_full, 0);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(kBM, kBN, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(kBM, D, 1);
      auto issue_s = [&](int t, int slot) {  // S_t = Q_t K^T: both K-major in shared memory
        const uint32_t a0 = base + kQ + t * kTile, b0 = base + kKV + slot * kTile;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kBox + (kk & 3) * 32;
          mma_ss(tmem + t * kBN, smem_desc_sw128(a0 + off, 16, 1024), smem_desc_sw128(b0 + off, 16, 1024), idesc_s,
                 kk > 0);
        }
      };
      auto issue_o = [&](int t, int slot, bool acc) {  // O_t += P_t V: P K-major, V MN-major, both in shared memory
        const uint32_t p0 = base + kP + t * kTile, v0 = base + kKV + slot * kTile;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ss(tmem + kTmemO + t * D, smem_desc_sw128(p0 + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                 smem_desc_sw128(v0 + kk * 2048, kBox, 1024), idesc_o, (acc || kk > 0) ? 1u : 0u);
      };
      auto next_k_fill = [&](int j) { return fill_k(j + 1); };
      bool ok = wait_bounded(q_full, 0) && wait_bounded(slot_full(0), 0);  // K_0 is fill 0
      if (ok) {
        tc_fence_after_sync();
        for (int t = 0; t < kNQ; ++t) {
          issue_s(t, 0);
          tc_commit(s_full(t));
        }
        tc_commit(slot_empty(0));
      }
      for (int j = 0; j < nblk && ok; ++j) {
        const int iv = fill_v(j, nblk), ik = next_k_fill(j);
        const bool next = j + 1 < nblk;
        if (next) ok = wait_bounded(slot_full(ik % kSlots), (ik / kSlots) & 1);
        if (!ok) break;
        // S of block j + 1 as soon as each tile's softmax has read S of block j
        for (int t = 0; t < kNQ && next && ok; ++t) {
          ok = wait_bounded(s_free(t), j & 1);
          if (!ok) break;
          tc_fence_after_sync();
          issue_s(t, ik % kSlots);
          tc_commit(s_full(t));
        }
        if (!ok) break;
        if (next) tc_commit(slot_empty(ik % kSlots));
        ok = wait_bounded(slot_full(iv % kSlots), (iv / kSlots) & 1);
        // O += P V of block j once each tile's P is in shared memory
        for (int t = 0; t < kNQ && ok; ++t) {
          ok = wait_bounded(p_full(t), j & 1);
          if (!ok) break;
          tc_fence_after_sync();
          issue_o(t, iv % kSlots, j > 0);
          tc_commit(pv_done(t));
        }
        if (!ok) break;
        tc_commit(slot_empty(iv % kSlots));
      }
      if (ok)
        for (int t = 0; t < kNQ; ++t) tc_commit(o_done(t));
      tc_commit(drain);  // every MMA issued must complete before TMEM is freed
      wait_bounded(drain, 0);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * kBN;
    const uint32_t tO = tmem + lane_base + kTmemO + t * D;
    const uint32_t p_row = base + kP + t * kTile + row * 128;  // this row of P_t (two boxes of 64 keys)
    const uint32_t sw = row & 7;
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(s_full(t), j & 1));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t sr[128];
      tmem_ld_x128(tS, sr);  // (waits for the load)
      // S_t is in registers: the next block's S may be written over it
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) mbar_arrive(s_free(t));
      float s[128];
#pragma unroll
      for (int i = 0; i < kBN; ++i) s[i] = __uint_as_float(sr[i]);
      int valid = args.n_kv - j * kBN;
      if (kCausal) valid = min(valid, q0 + t * kBM + row - args.kv_begin - j * kBN + 1);
      if (valid < kBN) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      float mp[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i < kBN - 4; i += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u) mp[u] = max3(mp[u], s[i + u], s[i + 4 + u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) mp[u] = fmaxf(mp[u], s[kBN - 4 + u]);
      const float mx = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])) * sl2;
      // block j - 1's product must be done before P_t is rewritten or O_t rescaled
      if (j > 0) {
        ok = __all_sync(0xffffffffu, wait_bounded(pv_done(t), (j - 1) & 1));
        if (!ok) break;
        tc_fence_after_sync();
      }
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, mx > m + kRescaleLog2)) {
        const float m_new = fmaxf(m, mx);
        const float alpha = (kCausal && m_new == -INFINITY) ? 1.f : ex2(m - m_new);
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
        tc_fence_before_sync();  // (ordered before the next P V by the P-ready arrive below)
      }
      const float m_use = (kCausal && m == -INFINITY) ? 0.f : m;
      const uint64_t nm2 = f2(-m_use, -m_use);
      uint64_t rs[4] = {0ull, 0ull, 0ull, 0ull};
      // P in 16-byte chunks of 8 keys: chunk c of the row goes to box c / 8, swizzled position (c % 8) ^ (row % 8)
#pragma unroll
      for (int c = 0; c < 16; ++c) {
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          float a, x;
          f2_split(f2_fma(f2(s[8 * c + 2 * e], s[8 * c + 2 * e + 1]), sl2x2, nm2), a, x);
          a = ex2(a);
          x = ex2(x);
          rs[e] = f2_add(rs[e], f2(a, x));
          w[e] = pack_bf16(a, x);
        }
        st_shared_v4(p_row + (c >> 3) * kBox + (((c & 7) ^ sw) << 4), w[0], w[1], w[2], w[3]);
      }
      float r0, r1;
      f2_split(f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3])), r0, r1);
      l += r0 + r1;
      fence_proxy_async_smem();  // P written by this thread, visible to the tensor core
      __syncwarp();
      if (lane == 0) mbar_arrive(p_full(t));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(o_done(t), 0));
    if (kUpdate && ok) ok = __all_sync(0xffffffffu, wait_bounded(acc_full, 0));
    ok = named_barrier_and(1 + t, 128, ok);
    if (ok) {
      tc_fence_after_sync();
      const int tile_q0 = q0 + t * kBM;
      float wc = l > 0.f ? 1.0f / l : 0.f, wa = 0.f;
      float lse_out = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (kUpdate) {
        const int q = tile_q0 + row;
        const float la = q < args.Sq ? args.lse_acc[((long long)b * args.H + h) * args.Sq + q] * 1.4426950408889634f
                                     : -INFINITY;
        const float lc = l > 0.f ? m + log2f(l) : -INFINITY;
        const float mx = fmaxf(la, lc);
        if (mx == -INFINITY) {
          wa = 0.f;
          wc = 0.f;
          lse_out = -INFINITY;
        } else {
          const float L2 = mx + log2f(ex2(la - mx) + ex2(lc - mx));
          wa = ex2(la - L2);
          wc = l > 0.f ? ex2(m - L2) : 0.f;
          lse_out = L2 * 0.69314718055994531f;
        }
      }
      const uint64_t wc2 = f2(wc, wc), wa2 = f2(wa, wa);
      const uint32_t stage = base + kQ + t * kTile;
      const bool f32 = args.o_f32 != 0;
      const int W = f32 ? 32 : 64;
      const int n_boxes = D / W;
      constexpr int kPerRound = D / 64;
      const uint32_t row_addr = stage + row * 128;
      for (int r0 = 0; r0 < n_boxes; r0 += kPerRound) {
        if (r0 > 0) {
          if (row == 0) bulk_wait_read_all();
          named_barrier_sync(1 + t, 128);
        }
        for (int c = r0 * W / 32; c < (r0 + kPerRound) * W / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(tO + c * 32, o);
          if (kUpdate) {
            // this row's columns 32c .. 32c + 31 of O_acc: box c (fp32) or c / 2 (bf16) of tile t's running O
            float a[32];
            const uint32_t src = base + kP + t * acc_tile + (args.acc_f32 ? c : c / 2) * kBox + row * 128;
            if (args.acc_f32) {
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                uint32_t x0, x1, x2, x3;
                ld_shared_v4(src + ((u ^ sw) << 4), x0, x1, x2, x3);
                a[4 * u] = __uint_as_float(x0), a[4 * u + 1] = __uint_as_float(x1);
                a[4 * u + 2] = __uint_as_float(x2), a[4 * u + 3] = __uint_as_float(x3);
              }
            } else {
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                uint32_t x[4];
                ld_shared_v4(src + (((4 * (c & 1) + u) ^ sw) << 4), x[0], x[1], x[2], x[3]);
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                  a[8 * u + 2 * e] = __uint_as_float(x[e] << 16);
                  a[8 * u + 2 * e + 1] = __uint_as_float(x[e] & 0xFFFF0000u);
                }
              }
            }
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2) {
              float y0, y1;
              f2_split(f2_fma(f2(__uint_as_float(o[2 * i2]), __uint_as_float(o[2 * i2 + 1])), wc2,
                              f2_mul(f2(a[2 * i2], a[2 * i2 + 1]), wa2)),
                       y0, y1);
              o[2 * i2] = __float_as_uint(y0), o[2 * i2 + 1] = __float_as_uint(y1);
            }
          }
          const uint64_t il2 = kUpdate ? f2(1.f, 1.f) : wc2;
          const int col0 = c * 32;
          const uint32_t dst = row_addr + (col0 / W - r0) * kBox;
          const int chunk0 = (col0 % W) / (f32 ? 4 : 8);
          if (f32) {
#pragma unroll
            for (int u = 0; u < 8; ++u) {
              float x0, x1, x2, x3;
              f2_split(f2_mul(f2(__uint_as_float(o[4 * u]), __uint_as_float(o[4 * u + 1])), il2), x0, x1);
              f2_split(f2_mul(f2(__uint_as_float(o[4 * u + 2]), __uint_as_float(o[4 * u + 3])), il2), x2, x3);
              st_shared_v4(dst + (((chunk0 + u) ^ sw) << 4), __float_as_uint(x0), __float_as_uint(x1),
                           __float_as_uint(x2), __float_as_uint(x3));
            }
          } else {
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              uint32_t w[4];
#pragma unroll
              for (int e = 0; e < 4; ++e) {
                float x0, x1;
                f2_split(f2_mul(f2(__uint_as_float(o[8 * u + 2 * e]), __uint_as_float(o[8 * u + 2 * e + 1])), il2),
                         x0, x1);
                w[e] = pack_bf16(x0, x1);
              }
              st_shared_v4(dst + (((chunk0 + u) ^ sw) << 4), w[0], w[1], w[2], w[3]);
            }
          }
        }
        fence_proxy_async_smem();
        named_barrier_sync(1 + t, 128);
        if (row == 0 && tile_q0 < args.Sq) {
          for (int bx = 0; bx < kPerRound && r0 + bx < n_boxes; ++bx)
            tma_store_4d(&tm_o, stage + bx * kBox, (r0 + bx) * W, h, tile_q0, b);
          bulk_commit_group();
        }
      }
      if (row == 0) bulk_wait_read_all();
      const int q = tile_q0 + row;
      if (q < args.Sq) args.lse[((long long)b * args.H + h) * args.Sq + q] = lse_out;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
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

// [B, S, H, D] with element strides {b, s, h} as a 4-D map (d, h, s, b), box of
// 128 bytes x 1 x 128 rows x 1, 128-byte swizzle; rows past S read as zero.
bool encode(CUtensorMap *map, const void *ptr, int B, int S, int H, const int64_t st[3], bool f32) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * es, (cuuint64_t)st[1] * es, (cuuint64_t)st[0] * es};
  cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kCausal, bool kUpdate>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to,
                         const CUtensorMap &tacc, const PsArgs &a, int B, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64] = {};
  if (dev < 64 && !configured[dev]) {
    e = cudaFuncSetAttribute(attn_fwd_ps_kernel<kCausal, kUpdate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return launch_kernel(attn_fwd_ps_kernel<kCausal, kUpdate>, dim3((a.Sq + kBM * kNQ - 1) / (kBM * kNQ), a.H, B),
                       dim3(kThreads), kAlloc, stream, tq, tk, tv, to, tacc, a);
}

}  // namespace

cudaError_t launch_attn_fwd_ps(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv,
                               const int64_t q_st[3], const int64_t kv_st[3], float scale, int kv_begin, int kv_end,
                               bool causal, void *o, bool o_f32, const int64_t o_st[3], float *lse, const void *o_acc,
                               bool acc_f32, const int64_t acc_st[3], const float *lse_acc, cudaStream_t stream,
                               const char **detail) {
  (void)Skv;
  CUtensorMap tq, tk, tv, to, tacc;
  const int n_kv = kv_end - kv_begin;
  const char *k0 = static_cast<const char *>(k) + (int64_t)kv_begin * kv_st[1] * 2;
  const char *v0 = static_cast<const char *>(v) + (int64_t)kv_begin * kv_st[1] * 2;
  if (!encode(&tq, q, B, Sq, H, q_st, false) || !encode(&tk, k0, B, n_kv, H, kv_st, false) ||
      !encode(&tv, v0, B, n_kv, H, kv_st, false) || !encode(&to, o, B, Sq, H, o_st, o_f32)) {
    *detail = "cuTensorMapEncodeTiled failed (driver entry point missing or strides/extents unsupported)";
    return cudaErrorInvalidValue;
  }
  const bool update = o_acc != nullptr;
  if (update && !encode(&tacc, o_acc, B, Sq, H, acc_st, acc_f32)) {
    *detail = "cuTensorMapEncodeTiled failed for the running output";
    return cudaErrorInvalidValue;
  }
  if (!update) tacc = to;
  PsArgs a;
  a.H = H;
  a.Sq = Sq;
  a.n_kv = n_kv;
  a.kv_begin = kv_begin;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.o_f32 = o_f32 ? 1 : 0;
  a.lse = lse;
  a.lse_acc = lse_acc;
  a.acc_f32 = acc_f32 ? 1 : 0;
  if (causal)
    return update ? launch_typed<true, true>(tq, tk, tv, to, tacc, a, B, stream)
                  : launch_typed<true, false>(tq, tk, tv, to, tacc, a, B, stream);
  return update ? launch_typed<false, true>(tq, tk, tv, to, tacc, a, B, stream)
                : launch_typed<false, false>(tq, tk, tv, to, tacc, a, B, stream);
}

cudaError_t read_and_clear_ps_error(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_ps_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_ps_error, &zero, sizeof(unsigned int));
}

}  // namespace ditattn
