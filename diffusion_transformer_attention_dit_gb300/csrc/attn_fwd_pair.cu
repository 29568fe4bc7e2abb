// Non-causal flash attention forward on CTA pairs (cluster of 2, tcgen05
// cta_group::2) for GB300, head dim 128: the same operation, outputs and update
// form as attn_fwd.cu (see there for the definition and its sources).
//
// Why pairs: in one CTA, every 128-key block costs the SM 256 KB of
// shared-memory traffic (the S = Q K^T MMAs read Q and K, the O += P V MMAs
// read V, TMA writes K and V) against 2048 tensor cycles of work, so shared
// memory, not the tensor core, sets the pace.  Two CTAs on two SMs run the
// block as M = 256 MMAs: each CTA keeps its own query rows (A operand) but holds
// only half of the block's K (64 keys) and half of its V (64 head-dim columns);
// the tensor cores of the pair exchange the halves.  Per SM that is 160 KB per
// block for the same tensor work.
//
// Roles, per CTA (320 threads): warps 0-7 softmax (two warpgroups, one per
// query tile; thread = query row = TMEM lane), warp 8 TMA producer, warp 9 MMA
// issuer (rank 0 only).  A pair covers 512 query rows: CTA r holds tiles
// [q0 + 256 r + 128 t, + 128) for t = 0, 1, and the MMA of tile t spans both
// CTAs' tile t.
//   - Loads: each CTA loads its own Q tiles, its K half (keys 64 r .. 64 r + 63
//     of the block) and its V half (columns 64 r .. 64 r + 63) with TMA
//     cta_group::2, completing on the rank-0 CTA's barriers (which expect both
//     CTAs' bytes).
//   - MMAs (rank 0, one thread): S_t = Q_t K^T and O_t += P_t V as M = 256 MMAs;
//     each commit is multicast to the same barrier in both CTAs.
//   - Softmax: as attn_fwd.cu; P-ready is one arrive per warp on the rank-0
//     CTA's barrier (remote for rank 1).
//   - Epilogue: each CTA normalises and stores its own rows; the update form
//     loads each CTA's running O tiles into its own freed ring slots.
// Every wait is bounded; a wait that gives up sets the device error word, and
// both CTAs still meet at the final cluster barrier before TMEM is freed.

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

__device__ unsigned int g_pair_error = 0;

constexpr int D = 128;
constexpr int kBM = 128;            // query rows per tile (per CTA; M = 256 over the pair)
constexpr int kBN = 128;            // keys per block
constexpr int kNQ = 2;              // query tiles per CTA
constexpr int kSlots = 8;           // ring slots of 16 KB: a K half or a V half each
constexpr int kThreads = 320;
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 8.0f;
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;

constexpr int kBox = 128 * 128;        // TMA box of 128 rows x 128 bytes (16 KB)
constexpr int kKHalfBox = 64 * 128;    // K half: 64 keys x 64 head-dim columns (8 KB), two per slot
constexpr int kTile = kBM * D * 2;     // one Q tile: 32 KB (two boxes)
constexpr int kSlotBytes = 16384;
constexpr int kQ = 0;
constexpr int kKV = kQ + kNQ * kTile;
constexpr int kBar = kKV + kSlots * kSlotBytes;
// q_full, slot_full[8], slot_empty[8], s_full[2], p_full[2], o_done[2], drain, acc_full[8]
constexpr int kNumBars = 1 + 2 * kSlots + 3 * kNQ + 1 + 8;
constexpr int kTmemSlot = kBar + 8 * kNumBars;
constexpr int kBytes = kTmemSlot + 16;
constexpr int kAlloc = kBytes + 1024;
constexpr uint32_t kTmemO = 2 * kBN;
static_assert(kAlloc <= 232448, "shared memory budget");

struct PairArgs {
  int H, Sq, n_kv;
  float scale_log2;
  int o_f32;
  float *lse;
  const float *lse_acc;
  int acc_f32;
};

// Bounded wait; kCluster: cluster-scope acquire, for barriers the other CTA arrives on.
template <bool kCluster = false>
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  auto try_wait = [&]() { return kCluster ? mbar_try_wait_cluster(bar, parity) : mbar_try_wait(bar, parity); };
  if (try_wait()) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (try_wait()) return true;
    if ((i & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || i > kWaitLimitIters)) {
      atomicOr(&g_pair_error, 1u);
      return false;
    }
  }
}

template <bool kUpdate>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_pair_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                         const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                         const __grid_constant__ CUtensorMap tm_acc, const PairArgs args) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + kTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = (blockIdx.x >> 1) * (2 * kBM * kNQ) + static_cast<int>(rank) * (kBM * kNQ);
  const int nblk = (args.n_kv + kBN - 1) / kBN;
  // update form: box bx (16 KB) of query tile t's running O is piece bx * kNQ + t, ring fill 2 * nblk + piece
  const int acc_boxes = kUpdate ? (args.acc_f32 ? 4 : 2) : 0;
  griddep_wait();
  griddep_launch_dependents();

  const uint32_t bars = base + kBar;
  const uint32_t q_full = bars;
  auto slot_full = [&](int s) { return bars + 8u * (1 + s); };
  auto slot_empty = [&](int s) { return bars + 8u * (1 + kSlots + s); };
  auto s_full = [&](int t) { return bars + 8u * (1 + 2 * kSlots + t); };
  auto p_full = [&](int t) { return bars + 8u * (1 + 2 * kSlots + kNQ + t); };
  auto o_done = [&](int t) { return bars + 8u * (1 + 2 * kSlots + 2 * kNQ + t); };
  const uint32_t drain = bars + 8u * (1 + 2 * kSlots + 3 * kNQ);
  auto acc_full = [&](int p) { return bars + 8u * (2 + 2 * kSlots + 3 * kNQ + p); };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int t = 0; t < kNQ; ++t) {
      mbar_init(s_full(t), 1);
      mbar_init(p_full(t), 8);  // one arrive per softmax warp of the tile, in both CTAs
      mbar_init(o_done(t), 1);
    }
    mbar_init(drain, 1);
    for (int p = 0; p < 8; ++p) mbar_init(acc_full(p), 1);
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
    tmem_alloc_pair(base + kTmemSlot, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();  // both CTAs' barriers exist before any cross-CTA arrive or load
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      const uint32_t lead_q_full = mapa_shared(q_full, 0);
      if (rank == 0) mbar_arrive_expect_tx(q_full, 2 * kNQ * kTile);
      for (int t = 0; t < kNQ; ++t)
        for (int hf = 0; hf < 2; ++hf)
          tma_load_4d_pair(base + kQ + t * kTile + hf * kBox, &tm_q, lead_q_full, hf * 64, h, q0 + t * kBM, b);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        for (int which = 0; which < 2; ++which) {  // 0: K half of block j, 1: V half
          const int i = 2 * j + which, slot = i % kSlots;
          if (!wait_bounded(slot_empty(slot), ((i / kSlots) & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(slot_full(slot), 2 * kSlotBytes);
          const uint32_t dst = base + kKV + slot * kSlotBytes, bar = mapa_shared(slot_full(slot), 0);
          if (which == 0) {  // keys j*128 + 64 r .. + 63, both head-dim halves
            for (int hf = 0; hf < 2; ++hf)
              tma_load_4d_pair(dst + hf * kKHalfBox, &tm_k, bar, hf * 64, h, j * kBN + 64 * static_cast<int>(rank), b);
          } else {  // all 128 keys, head-dim columns 64 r .. 64 r + 63
            tma_load_4d_pair(dst, &tm_v, bar, 64 * static_cast<int>(rank), h, j * kBN, b);
          }
          ++issued;
        }
      }
      // update form: this CTA's running O tiles, box by box, into the slots the last blocks free
      int pieces = 0;
      for (int p = 0; p < acc_boxes * kNQ && ok; ++p) {
        const int i = 2 * nblk + p, slot = i % kSlots, t = p % kNQ, bx = p / kNQ;
        if (!wait_bounded(slot_empty(slot), ((i / kSlots) & 1) ^ 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(acc_full(p), kSlotBytes);
        tma_load_4d(base + kKV + slot * kSlotBytes, &tm_acc, acc_full(p), bx * (args.acc_f32 ? 32 : 64), h,
                    q0 + t * kBM, b);
        ++pieces;
      }
      // Copies must land before the CTA may exit.  K/V halves of both CTAs complete
      // on rank 0's slot barriers: rank 0 waits for the last fills there (the final
      // cluster barrier keeps rank 1 resident until then); rank 1 additionally sees
      // its last fills consumed (their slot_empty) on the normal path.
      if (rank == 0) wait_bounded(q_full, 0);
      for (int i = issued > kSlots ? issued - kSlots : 0; i < issued; ++i) {
        if (rank == 0)
          wait_bounded(slot_full(i % kSlots), (i / kSlots) & 1);
        else if (ok)
          wait_bounded(slot_empty(i % kSlots), (i / kSlots) & 1);
      }
      for (int p = 0; p < pieces; ++p) wait_bounded(acc_full(p), 0);
    }
    __syncwarp();
  } else if (warp == kWarpMma) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(2 * kBM, kBN, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(2 * kBM, D, 1);
      auto issue_s = [&](int t, int slot) {  // S_t = Q_t K^T: A = own Q tile, B = K half (64 keys), K-major
        const uint32_t a0 = base + kQ + t * kTile, b0 = base + kKV + slot * kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_pair(tmem + t * kBN, smem_desc_sw128(a0 + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                      smem_desc_sw128(b0 + (kk >> 2) * kKHalfBox + (kk & 3) * 32, 16, 1024), idesc_s, kk > 0);
      };
      auto issue_o = [&](int t, int slot, bool acc) {  // O_t += P_t V: P in TMEM, B = V half (64 columns), MN-major
        const uint32_t v0 = base + kKV + slot * kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)
          mma_ts_pair(tmem + kTmemO + t * D, tmem + t * kBN + kk * 8, smem_desc_sw128(v0 + kk * 2048, kBox, 1024),
                      idesc_o, (acc || kk > 0) ? 1u : 0u);
      };
      bool ok = wait_bounded(q_full, 0) && wait_bounded(slot_full(0), 0);
      if (ok) {
        tc_fence_after_sync();
        for (int t = 0; t < kNQ; ++t) {
          issue_s(t, 0);
          tc_commit_pair(s_full(t));
        }
        tc_commit_pair(slot_empty(0));
      }
      for (int j = 0; j < nblk && ok; ++j) {
        const int iv = 2 * j + 1, ik = 2 * j + 2;
        const bool next = j + 1 < nblk;
        ok = wait_bounded(slot_full(iv % kSlots), (iv / kSlots) & 1);
        if (ok && next) ok = wait_bounded(slot_full(ik % kSlots), (ik / kSlots) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        for (int t = 0; t < kNQ && ok; ++t) {
          ok = wait_bounded<true>(p_full(t), j & 1);
          if (!ok) break;
          tc_fence_after_sync();
          issue_o(t, iv % kSlots, j > 0);
          if (next) {
            issue_s(t, ik % kSlots);
            tc_commit_pair(s_full(t));
          }
        }
        if (!ok) break;
        tc_commit_pair(slot_empty(iv % kSlots));
        if (next) tc_commit_pair(slot_empty(ik % kSlots));
      }
      if (ok)
        for (int t = 0; t < kNQ; ++t) tc_commit_pair(o_done(t));
      tc_commit_pair(drain);  // every pair MMA issued has completed in both CTAs when this fires
    }
    // both CTAs: no TMEM release before the pair's MMAs are done with it
    if (lane == 0) wait_bounded(drain, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warpgroups (both CTAs)
    const int t = warp >> 2, wq = warp & 3;
    const int row = wq * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem + lane_base + t * kBN;
    const uint32_t tO = tmem + lane_base + kTmemO + t * D;
    const uint32_t p_ready = rank == 0 ? p_full(t) : mapa_shared(p_full(t), 0);
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
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
      const int valid = args.n_kv - j * kBN;  // columns past the range end are masked
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
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, mx > m + kRescaleLog2)) {
        // the previous PV product of this tile is complete: S_t for block j was
        // issued after it, and its commit covers every earlier pair MMA
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
      const uint64_t nm2 = f2(-m, -m);
      uint64_t rs[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t p0[32], p1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a, c;
        f2_split(f2_fma(f2(s[2 * i], s[2 * i + 1]), sl2x2, nm2), a, c);
        a = ex2(a);
        c = ex2(c);
        rs[i & 3] = f2_add(rs[i & 3], f2(a, c));
        p0[i] = pack_bf16(a, c);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a, c;
        f2_split(f2_fma(f2(s[64 + 2 * i], s[64 + 2 * i + 1]), sl2x2, nm2), a, c);
        a = ex2(a);
        c = ex2(c);
        rs[i & 3] = f2_add(rs[i & 3], f2(a, c));
        p1[i] = pack_bf16(a, c);
      }
      tmem_st_x32(tS, p0);
      tmem_st_x32(tS + 32, p1);
      float r0, r1;
      f2_split(f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3])), r0, r1);
      l += r0 + r1;
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(p_ready);
        else
          mbar_arrive_cluster(p_ready);
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(o_done(t), 0));
    if (kUpdate && ok) {
      bool got = true;
      for (int bx = 0; bx < acc_boxes; ++bx) got = got && wait_bounded(acc_full(bx * kNQ + t), 0);
      ok = __all_sync(0xffffffffu, got);
    }
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
      const uint32_t sw = row & 7;
      for (int r0 = 0; r0 < n_boxes; r0 += kPerRound) {
        if (r0 > 0) {
          if (row == 0) bulk_wait_read_all();
          named_barrier_sync(1 + t, 128);
        }
        for (int c = r0 * W / 32; c < (r0 + kPerRound) * W / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(tO + c * 32, o);
          if (kUpdate) {
            // the same 32 columns of this row of O_acc: box c (fp32, 32 columns) or box c / 2 (bf16)
            float a[32];
            const int bx = args.acc_f32 ? c : c / 2;
            const int i = 2 * nblk + bx * kNQ + t;
            const uint32_t src = base + kKV + (i % kSlots) * kSlotBytes + row * 128;
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
  cluster_sync();  // neither CTA leaves while the pair's MMAs or loads may still touch it
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kTmemCols);
  }
}

// ---------------------------------------------------------------------------
// Pair kernel with one query tile per CTA and three S buffers in TMEM
// (S0 S1 S2 O = 512 columns).  The MMA thread issues S for block j + 3 as soon
// as P of block j is in (into the buffer P_j frees), so S is computed three
// blocks ahead of the softmax and the cross-SM signals of a block are off the
// softmax's critical path.  O += P_j V_j is committed to pv_done[j % 3]; the
// (rare) O rescale of block j waits there for block j - 1's product.
// Roles: warps 0-3 softmax (thread = query row), warp 4 TMA, warp 5 MMA (rank 0).

namespace p3 {

constexpr int kNS = 3;               // S buffers
constexpr int kSlots3 = 10;          // ring slots of 16 KB (five blocks of K/V halves)
constexpr int kThreads3 = 192;
constexpr int kWarpTma3 = 4;
constexpr int kWarpMma3 = 5;
constexpr int kQ3 = 0;
constexpr int kKV3 = kQ3 + kTile;
constexpr int kBar3 = kKV3 + kSlots3 * kSlotBytes;
// q_full, slot_full[10], slot_empty[10], s_full[3], p_full[3], pv_done[3], o_done, drain, acc_full[4]
constexpr int kNumBars3 = 1 + 2 * kSlots3 + 3 * kNS + 2 + 4;
constexpr int kTmemSlot3 = kBar3 + 8 * kNumBars3;
constexpr int kAlloc3 = kTmemSlot3 + 16 + 1024;
constexpr uint32_t kTmemO3 = kNS * kBN;
static_assert(kAlloc3 <= 232448, "shared memory budget");

}  // namespace p3

template <bool kUpdate>
__global__ void __launch_bounds__(p3::kThreads3, 1)
    attn_fwd_pair3_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                          const __grid_constant__ CUtensorMap tm_acc, const PairArgs args) {
  using namespace p3;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + kTmemSlot3);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = (blockIdx.x >> 1) * (2 * kBM) + static_cast<int>(rank) * kBM;
  const int nblk = (args.n_kv + kBN - 1) / kBN;
  const int acc_boxes = kUpdate ? (args.acc_f32 ? 4 : 2) : 0;  // running-O box p is ring fill 2 * nblk + p
  griddep_wait();
  griddep_launch_dependents();

  const uint32_t bars = base + kBar3;
  const uint32_t q_full = bars;
  auto slot_full = [&](int s) { return bars + 8u * (1 + s); };
  auto slot_empty = [&](int s) { return bars + 8u * (1 + kSlots3 + s); };
  // one P-ready barrier per S buffer: the softmax runs up to three blocks ahead of the PV products, and
  // block j + 3 (same buffer) cannot start before the MMA has taken block j's phase
  auto s_full = [&](int x) { return bars + 8u * (1 + 2 * kSlots3 + x); };
  auto p_full = [&](int x) { return bars + 8u * (1 + 2 * kSlots3 + kNS + x); };
  // PV of block j completes on pv_done[j % 3], so block j - 1's product is the only phase that can be
  // pending there when block j's softmax asks (block j - 4's is done, block j + 2's cannot exist yet)
  auto pv_done = [&](int x) { return bars + 8u * (1 + 2 * kSlots3 + 2 * kNS + x); };
  const uint32_t o_done = bars + 8u * (1 + 2 * kSlots3 + 3 * kNS), drain = o_done + 8;
  auto acc_full = [&](int p) { return o_done + 16 + 8u * p; };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSlots3; ++s) {
      mbar_init(slot_full(s), 1);
      mbar_init(slot_empty(s), 1);
    }
    for (int x = 0; x < kNS; ++x) {
      mbar_init(s_full(x), 1);
      mbar_init(p_full(x), 8);  // one arrive per softmax warp, in both CTAs
    }
    for (int x = 0; x < kNS; ++x) mbar_init(pv_done(x), 1);
    mbar_init(o_done, 1);
    mbar_init(drain, 1);
    for (int p = 0; p < 4; ++p) mbar_init(acc_full(p), 1);
    mbar_fence_init();
  }
  if (warp == kWarpTma3 && lane == 0) {
    tma_prefetch_map(&tm_q);
    tma_prefetch_map(&tm_k);
    tma_prefetch_map(&tm_v);
    tma_prefetch_map(&tm_o);
    if (kUpdate) tma_prefetch_map(&tm_acc);
  }
  if (warp == kWarpMma3) {
    tmem_alloc_pair(base + kTmemSlot3, kTmemCols);
    tmem_relinquish_pair();
  }
  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;

  if (warp == kWarpTma3) {
    // ------------------------------------------------------------ producer (both CTAs)
    if (lane == 0) {
      if (rank == 0) mbar_arrive_expect_tx(q_full, 2 * kTile);
      for (int hf = 0; hf < 2; ++hf)
        tma_load_4d_pair(base + kQ3 + hf * kBox, &tm_q, mapa_shared(q_full, 0), hf * 64, h, q0, b);
      int issued = 0;
      bool ok = true;
      for (int j = 0; j < nblk && ok; ++j) {
        for (int which = 0; which < 2; ++which) {  // fill 2j: K half of block j; 2j + 1: V half
          const int i = 2 * j + which, slot = i % kSlots3;
          if (!wait_bounded(slot_empty(slot), ((i / kSlots3) & 1) ^ 1)) {
            ok = false;
            break;
          }
          if (rank == 0) mbar_arrive_expect_tx(slot_full(slot), 2 * kSlotBytes);
          const uint32_t dst = base + kKV3 + slot * kSlotBytes, bar = mapa_shared(slot_full(slot), 0);
          if (which == 0) {
            for (int hf = 0; hf < 2; ++hf)
              tma_load_4d_pair(dst + hf * kKHalfBox, &tm_k, bar, hf * 64, h, j * kBN + 64 * static_cast<int>(rank), b);
          } else {
            tma_load_4d_pair(dst, &tm_v, bar, 64 * static_cast<int>(rank), h, j * kBN, b);
          }
          ++issued;
        }
      }
      int pieces = 0;
      for (int p = 0; p < acc_boxes && ok; ++p) {
        const int i = 2 * nblk + p, slot = i % kSlots3;
        if (!wait_bounded(slot_empty(slot), ((i / kSlots3) & 1) ^ 1)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(acc_full(p), kSlotBytes);
        tma_load_4d(base + kKV3 + slot * kSlotBytes, &tm_acc, acc_full(p), p * (args.acc_f32 ? 32 : 64), h, q0, b);
        ++pieces;
      }
      if (rank == 0) wait_bounded(q_full, 0);
      for (int i = issued > kSlots3 ? issued - kSlots3 : 0; i < issued; ++i) {
        if (rank == 0)
          wait_bounded(slot_full(i % kSlots3), (i / kSlots3) & 1);
        else if (ok)
          wait_bounded(slot_empty(i % kSlots3), (i / kSlots3) & 1);
      }
      for (int p = 0; p < pieces; ++p) wait_bounded(acc_full(p), 0);
    }
    __syncwarp();
  } else if (warp == kWarpMma3) {
    // ------------------------------------------------------------ MMA issuer (rank 0)
    if (lane == 0 && rank == 0) {
      constexpr uint32_t idesc_s = idesc_bf16_f32(2 * kBM, kBN, 0);
      constexpr uint32_t idesc_o = idesc_bf16_f32(2 * kBM, D, 1);
      auto issue_s = [&](int j) {  // S_j = Q K_j^T into buffer j % 3 (K half: fill 2j)
        const int slot = (2 * j) % kSlots3;
        const uint32_t a0 = base + kQ3, b0 = base + kKV3 + slot * kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ss_pair(tmem + (j % kNS) * kBN, smem_desc_sw128(a0 + (kk >> 2) * kBox + (kk & 3) * 32, 16, 1024),
                      smem_desc_sw128(b0 + (kk >> 2) * kKHalfBox + (kk & 3) * 32, 16, 1024), idesc_s, kk > 0);
        tc_commit_pair(s_full(j % kNS));
        tc_commit_pair(slot_empty(slot));
      };
      bool ok = wait_bounded(q_full, 0);
      for (int j = 0; j < kNS && j < nblk && ok; ++j) {
        ok = wait_bounded(slot_full((2 * j) % kSlots3), ((2 * j) / kSlots3) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        issue_s(j);
      }
      for (int j = 0; j < nblk && ok; ++j) {
        const int iv = 2 * j + 1;
        ok = wait_bounded(slot_full(iv % kSlots3), (iv / kSlots3) & 1) &&
             wait_bounded<true>(p_full(j % kNS), (j / kNS) & 1);
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t v0 = base + kKV3 + (iv % kSlots3) * kSlotBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk)  // O += P_j V_j, P_j in buffer j % 3
          mma_ts_pair(tmem + kTmemO3, tmem + (j % kNS) * kBN + kk * 8, smem_desc_sw128(v0 + kk * 2048, kBox, 1024),
                      idesc_o, (j > 0 || kk > 0) ? 1u : 0u);
        tc_commit_pair(pv_done(j % kNS));
        tc_commit_pair(slot_empty(iv % kSlots3));
        const int jn = j + kNS;  // S of block j + 3 into the buffer P_j leaves (after the product above, in order)
        if (jn < nblk) {
          const int ik = 2 * jn;
          ok = wait_bounded(slot_full(ik % kSlots3), (ik / kSlots3) & 1);
          if (!ok) break;
          tc_fence_after_sync();
          issue_s(jn);
        }
      }
      if (ok) tc_commit_pair(o_done);
      tc_commit_pair(drain);
    }
    if (lane == 0) wait_bounded(drain, 0);
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax (both CTAs): warps 0-3, thread = row
    const int row = warp * 32 + lane;
    const uint32_t lane_base = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem + lane_base + kTmemO3;
    const float sl2 = args.scale_log2;
    const uint64_t sl2x2 = f2(sl2, sl2);
    float m = -INFINITY, l = 0.f;
    bool ok = true;
    for (int j = 0; j < nblk; ++j) {
      const uint32_t tS = tmem + lane_base + (j % kNS) * kBN;
      const uint32_t p_ready = rank == 0 ? p_full(j % kNS) : mapa_shared(p_full(j % kNS), 0);
      ok = __all_sync(0xffffffffu, wait_bounded(s_full(j % kNS), (j / kNS) & 1));
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
      float mp[4] = {s[0], s[1], s[2], s[3]};
#pragma unroll
      for (int i = 4; i < kBN - 4; i += 8)
#pragma unroll
        for (int u = 0; u < 4; ++u) mp[u] = max3(mp[u], s[i + u], s[i + 4 + u]);
#pragma unroll
      for (int u = 0; u < 4; ++u) mp[u] = fmaxf(mp[u], s[kBN - 4 + u]);
      const float mx = fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])) * sl2;
      if (j == 0) {
        m = mx;
      } else if (__any_sync(0xffffffffu, mx > m + kRescaleLog2)) {
        // O holds the products up to block j - 1 once that product is done (in order, so
        // are all earlier ones)
        ok = __all_sync(0xffffffffu, wait_bounded(pv_done((j - 1) % kNS), ((j - 1) / kNS) & 1));
        if (!ok) break;
        tc_fence_after_sync();
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
      const uint64_t nm2 = f2(-m, -m);
      uint64_t rs[4] = {0ull, 0ull, 0ull, 0ull};
      uint32_t p0[32], p1[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a, c;
        f2_split(f2_fma(f2(s[2 * i], s[2 * i + 1]), sl2x2, nm2), a, c);
        a = ex2(a);
        c = ex2(c);
        rs[i & 3] = f2_add(rs[i & 3], f2(a, c));
        p0[i] = pack_bf16(a, c);
      }
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        float a, c;
        f2_split(f2_fma(f2(s[64 + 2 * i], s[64 + 2 * i + 1]), sl2x2, nm2), a, c);
        a = ex2(a);
        c = ex2(c);
        rs[i & 3] = f2_add(rs[i & 3], f2(a, c));
        p1[i] = pack_bf16(a, c);
      }
      tmem_st_x32(tS, p0);
      tmem_st_x32(tS + 32, p1);
      float r0, r1;
      f2_split(f2_add(f2_add(rs[0], rs[1]), f2_add(rs[2], rs[3])), r0, r1);
      l += r0 + r1;
      tmem_st_wait();
      tc_fence_before_sync();
      __syncwarp();
      if (lane == 0) {
        if (rank == 0)
          mbar_arrive(p_ready);
        else
          mbar_arrive_cluster(p_ready);
      }
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(o_done, 0));
    if (kUpdate && ok) {
      bool got = true;
      for (int p = 0; p < acc_boxes; ++p) got = got && wait_bounded(acc_full(p), 0);
      ok = __all_sync(0xffffffffu, got);
    }
    ok = named_barrier_and(1, 128, ok);
    if (ok) {
      tc_fence_after_sync();
      float wc = l > 0.f ? 1.0f / l : 0.f, wa = 0.f;
      float lse_out = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (kUpdate) {
        const int q = q0 + row;
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
      const uint32_t stage = base + kQ3;
      const bool f32 = args.o_f32 != 0;
      const int W = f32 ? 32 : 64;
      const int n_boxes = D / W;
      constexpr int kPerRound = D / 64;
      const uint32_t row_addr = stage + row * 128;
      const uint32_t sw = row & 7;
      for (int r0 = 0; r0 < n_boxes; r0 += kPerRound) {
        if (r0 > 0) {
          if (row == 0) bulk_wait_read_all();
          named_barrier_sync(1, 128);
        }
        for (int c = r0 * W / 32; c < (r0 + kPerRound) * W / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(tO + c * 32, o);
          if (kUpdate) {
            float a[32];
            const int bx = args.acc_f32 ? c : c / 2;
            const uint32_t src = base + kKV3 + ((2 * nblk + bx) % kSlots3) * kSlotBytes + row * 128;
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
        named_barrier_sync(1, 128);
        if (row == 0 && q0 < args.Sq) {
          for (int bx = 0; bx < kPerRound && r0 + bx < n_boxes; ++bx)
            tma_store_4d(&tm_o, stage + bx * kBox, (r0 + bx) * W, h, q0, b);
          bulk_commit_group();
        }
      }
      if (row == 0) bulk_wait_read_all();
      const int q = q0 + row;
      if (q < args.Sq) args.lse[((long long)b * args.H + h) * args.Sq + q] = lse_out;
    }
  }

  tc_fence_before_sync();
  __syncthreads();
  cluster_sync();
  if (warp == kWarpMma3) {
    tc_fence_after_sync();
    tmem_dealloc_pair(tmem, kTmemCols);
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
// 128 bytes x 1 x box_rows x 1, 128-byte swizzle; rows past S read as zero.
bool encode(CUtensorMap *map, const void *ptr, int B, int S, int H, const int64_t st[3], bool f32, int box_rows) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (!enc) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * es, (cuuint64_t)st[1] * es, (cuuint64_t)st[0] * es};
  cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, (cuuint32_t)box_rows, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  return enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
             const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
             CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
             CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

template <bool kUpdate>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to,
                         const CUtensorMap &tacc, const PairArgs &a, int B, bool one_tile, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static bool configured[64][2] = {};
  if (dev < 64 && !configured[dev][one_tile]) {
    e = one_tile ? cudaFuncSetAttribute(attn_fwd_pair3_kernel<kUpdate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        p3::kAlloc3)
                 : cudaFuncSetAttribute(attn_fwd_pair_kernel<kUpdate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                        kAlloc);
    if (e != cudaSuccess) return e;
    configured[dev][one_tile] = true;
  }
  if (one_tile) {
    const int pairs = (a.Sq + 2 * kBM - 1) / (2 * kBM);
    return launch_kernel_cluster(attn_fwd_pair3_kernel<kUpdate>, dim3(2 * pairs, a.H, B), dim3(p3::kThreads3),
                                 p3::kAlloc3, stream, 2u, tq, tk, tv, to, tacc, a);
  }
  const int pairs = (a.Sq + 2 * kBM * kNQ - 1) / (2 * kBM * kNQ);
  return launch_kernel_cluster(attn_fwd_pair_kernel<kUpdate>, dim3(2 * pairs, a.H, B), dim3(kThreads), kAlloc,
                               stream, 2u, tq, tk, tv, to, tacc, a);
}

}  // namespace

cudaError_t launch_attn_fwd_pair(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv,
                                 const int64_t q_st[3], const int64_t kv_st[3], float scale, int kv_begin, int kv_end,
                                 void *o, bool o_f32, const int64_t o_st[3], float *lse, const void *o_acc,
                                 bool acc_f32, const int64_t acc_st[3], const float *lse_acc, bool one_tile,
                                 cudaStream_t stream, const char **detail) {
  (void)Skv;
  CUtensorMap tq, tk, tv, to, tacc;
  const int n_kv = kv_end - kv_begin;
  const char *k0 = static_cast<const char *>(k) + (int64_t)kv_begin * kv_st[1] * 2;
  const char *v0 = static_cast<const char *>(v) + (int64_t)kv_begin * kv_st[1] * 2;
  if (!encode(&tq, q, B, Sq, H, q_st, false, 128) || !encode(&tk, k0, B, n_kv, H, kv_st, false, 64) ||
      !encode(&tv, v0, B, n_kv, H, kv_st, false, 128) || !encode(&to, o, B, Sq, H, o_st, o_f32, 128)) {
    *detail = "cuTensorMapEncodeTiled failed (driver entry point missing or strides/extents unsupported)";
    return cudaErrorInvalidValue;
  }
  const bool update = o_acc != nullptr;
  if (update && !encode(&tacc, o_acc, B, Sq, H, acc_st, acc_f32, 128)) {
    *detail = "cuTensorMapEncodeTiled failed for the running output";
    return cudaErrorInvalidValue;
  }
  if (!update) tacc = to;
  PairArgs a;
  a.H = H;
  a.Sq = Sq;
  a.n_kv = n_kv;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.o_f32 = o_f32 ? 1 : 0;
  a.lse = lse;
  a.lse_acc = lse_acc;
  a.acc_f32 = acc_f32 ? 1 : 0;
  return update ? launch_typed<true>(tq, tk, tv, to, tacc, a, B, one_tile, stream)
                : launch_typed<false>(tq, tk, tv, to, tacc, a, B, one_tile, stream);
}

cudaError_t read_and_clear_pair_error(unsigned int *value) {
  unsigned int zero = 0;
  cudaError_t e = cudaMemcpyFromSymbol(value, g_pair_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_pair_error, &zero, sizeof(unsigned int));
}

}  // namespace ditattn
