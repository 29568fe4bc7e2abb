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
//               into a ring of shared-memory slots (128-byte swizzle); a slot
//               is refilled when the S-ready barrier of the second tile shows
//               that its last reader has completed.
//   warp 9      MMA issuer (one thread): S_t = Q_t K_j^T into TMEM (SS form),
//               O_t += P_t V_j with P read from TMEM (TS form).  Two query
//               tiles t = 0, 1 alternate so the tensor core always has one
//               tile's work while the other tile's softmax runs.
//   warps 0-7   two softmax warpgroups, one per query tile; thread = one query
//               row (TMEM lane), so row max / row sum need no shuffles.  Online
//               softmax in base 2: the scale is folded into one packed FFMA2 per
//               pair of scores, row sums use packed FADD2 and the row max a
//               3-input max; the O rescale is lazy (only when a row max grows by
//               more than a factor 2^10, so weights stay below 1024), exact
//               after the final 1/l.  On K x 3 scores 2^8 rescaled ~5 % of the
//               warp-blocks and ran 1.2 % slower; 2^12 and 2^16 ran ~2 % faster
//               but their merged bf16 partials strayed further from the exact
//               result (0.03 max abs at 2^16 against 0.022 at 2^8 and 2^10).
//               P is written back
//               over S in TMEM as bf16.  Epilogue: O / l from TMEM, staged in
//               the idle Q buffer in swizzled layout and written by TMA;
//               LSE = (m + log2 l) ln 2.
// TMEM (512 columns): S/P of tile 0 | S/P of tile 1 | O of tile 0 | O of tile 1.
//
// Update form (same PR, item 2: update_out_and_lse after each ring step): with a
// running result (O_acc, LSE_acc) of earlier key ranges, the epilogue writes
//   L = ln(e^LSE_acc + e^LSE_c),  O = e^(LSE_acc - L) O_acc + e^(LSE_c - L) O_c
// so the block's own O never reaches memory.  The O_acc tiles are loaded by TMA
// into K/V ring slots freed by the last blocks, as further fills of the ring.
// Every mbarrier wait is bounded (about 2 s); a wait that gives up sets the
// library's device error word and the CTA drains its in-flight copies and MMAs,
// frees TMEM and exits.
//
// Deferred dependency wait (a later chunk of one attention, launched right
// after the previous chunk on the same stream): Q, K and V were complete before
// the previous chunk started, so the kernel starts its blocks at once, beside
// the previous launch's last wave, and calls griddepcontrol.wait only where it
// needs that launch's results -- the update form before it loads O_acc (TMA
// producer) and reads LSE_acc (epilogue threads), the plain form before its
// CTAs exit.  Either way no CTA ends before the previous launch has, so the
// launches still complete in stream order.

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

__device__ unsigned int g_device_error = 0;

namespace {

using namespace attn;

constexpr int kBM = 128;            // query rows per tile (MMA M)
constexpr int kBN = 128;            // keys per block (MMA N of S, K of PV)
constexpr int kNQ = 2;              // query tiles per CTA
constexpr int kSlots = 4;           // K/V shared-memory ring slots
constexpr int kThreads = 320;       // 8 softmax warps + TMA warp + MMA warp
constexpr int kWarpTma = 8;
constexpr int kWarpMma = 9;
constexpr uint32_t kTmemCols = 512;
constexpr float kRescaleLog2 = 10.0f;  // lazy-rescale threshold on the running max (base-2 units)
constexpr uint64_t kWaitLimitNs = 2000000000ull;
constexpr uint32_t kWaitLimitIters = 1u << 26;
constexpr unsigned int kErrWaitTimeout = 1u;

template <int D>
struct Layout {
  static constexpr int kBox = 128 * 128;     // one TMA box: 128 rows x 128 bytes (64 bf16)
  static constexpr int kTile = 128 * D * 2;  // one Q tile or one K / V block
  static constexpr int kQ = 0;
  static constexpr int kKV = kQ + kNQ * kTile;
  static constexpr int kBar = kKV + kSlots * kTile;
  // q_full, slot_full[kSlots], s_full[kNQ], p_full[kNQ], o_done[kNQ], drain
  static constexpr int kNumBars = 1 + kSlots + 3 * kNQ + 1;
  static constexpr int kTmemSlot = kBar + 8 * kNumBars;
  static constexpr int kBytes = kTmemSlot + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 bytes
  static constexpr uint32_t kTmemO = 2 * kBN;   // first O column
};

struct AttnArgs {
  int H, Sq, n_kv;
  int kv_begin;  // absolute index of the first key of the range
  float scale_log2;
  void *o;
  long long o_sb, o_ss, o_sh;
  int o_f32;
  float *lse;
  const float *lse_acc;  // update form: running LSE [B, H, Sq] (may equal lse)
  int acc_f32;           // update form: O_acc is fp32 (else bf16)
  int defer_wait;        // wait for the previous launch only where its results are needed (see above)
};

// Bounded wait; false (and the device error word set) if the phase did not complete in time.
__device__ __forceinline__ bool wait_bounded(uint32_t bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = global_timer_ns();
  for (uint32_t i = 1;; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    // two bounds: elapsed time, and an iteration count that ends the wait even if
    // the global timer were not advancing
    if ((i & 63u) == 0 && (global_timer_ns() - t0 > kWaitLimitNs || i > kWaitLimitIters)) {
      atomicOr(&g_device_error, kErrWaitTimeout);
      return false;
    }
  }
}

template <int D, bool kCausal, bool kUpdate>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                    const __grid_constant__ CUtensorMap tm_v, const __grid_constant__ CUtensorMap tm_o,
                    const __grid_constant__ CUtensorMap tm_acc, const AttnArgs args) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw = smem_u32(smem_raw);
  const uint32_t base = (raw + 1023u) & ~1023u;
  uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem_raw + (base - raw) + L::kTmemSlot);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int h = blockIdx.y, b = blockIdx.z;
  const int q0 = blockIdx.x * (kBM * kNQ);
  // key blocks this CTA visits: all of the range, or (causal) those up to its last query row
  int nblk = (args.n_kv + kBN - 1) / kBN;
  if (kCausal) {
    const int q_last = min(q0 + kBM * kNQ, args.Sq) - 1;
    const int reach = q_last - args.kv_begin + 1;  // keys of the range visible to the last row
    nblk = max(1, min(nblk, (reach + kBN - 1) / kBN));
  }
  // Update form: the O_acc tile of query tile t, half hf, is ring fill 2 * nblk + hf * kNQ + t
  // (one 128 x D bf16 tile, or two halves of an fp32 tile, per ring slot).
  const int acc_halves = kUpdate ? (args.acc_f32 ? 2 : 1) : 0;
  if (!args.defer_wait) griddep_wait();
  griddep_launch_dependents();

  const uint32_t bars = base + L::kBar;
  const uint32_t q_full = bars;
  auto slot_full = [&](int s) { return bars + 8u * (1 + s); };
  auto s_full = [&](int t) { return bars + 8u * (1 + kSlots + t); };
  auto p_full = [&](int t) { return bars + 8u * (1 + kSlots + kNQ + t); };
  auto o_done = [&](int t) { return bars + 8u * (1 + kSlots + 2 * kNQ + t); };
  const uint32_t drain = bars + 8u * (1 + kSlots + 3 * kNQ);
  // K/V fill i (i < 2 * nblk) reuses the slot of fill i - kSlots, which may be
  // overwritten once the last MMA reading it has completed.  K_b is read last by
  // S_1(b), the last MMA issued for block b; V_b by P V_1(b), which S_1(b + 1)
  // follows (for the last block, the o_done commits).  The s_full(1) / o_done(1)
  // arrivals therefore also release the ring, and the MMA thread commits nothing
  // for it.  A parity wait is exact while the barrier is at most one phase past
  // the awaited one.  The producer waits for each s_full(1) phase (two fills per
  // phase) as soon as it has issued the fill before, and the next phase needs a
  // whole softmax pass of tile 1 after that one, so it sees every phase it waits
  // for before the following one completes.  Were it ever two phases late, the
  // wait would not return until a phase that needs this very fill: it times out
  // and the launch reports an error; no slot is overwritten early.  Fills after
  // the last K/V block (the update form's running O) wait for o_done(1) instead,
  // which completes once.
  auto wait_slot_free = [&](int i) -> bool {
    const int prev = i - kSlots;
    if (prev < 0) return true;
    const int blk = prev >> 1;
    if ((prev & 1) == 0) return wait_bounded(s_full(kNQ - 1), blk & 1);
    if (blk + 1 < nblk) return wait_bounded(s_full(kNQ - 1), (blk + 1) & 1);
    return wait_bounded(o_done(kNQ - 1), 0);
  };

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < kSlots; ++s) mbar_init(slot_full(s), 1);
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
    tma_prefetch_map(&tm_o);
    if (kUpdate) tma_prefetch_map(&tm_acc);
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
          if (!wait_slot_free(i)) {
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
      if (kUpdate && args.defer_wait) griddep_wait();  // O_acc is the previous launch's output
      // Update form: the O_acc tiles follow the last K/V block through the ring.
      // A slot holds D / 64 boxes of 128 rows x 128 bytes: a whole bf16 tile, or
      // half of an fp32 tile (boxes of 32 columns).
      for (int p = 0; p < acc_halves * kNQ && ok; ++p) {
        const int i = 2 * nblk + p, slot = i % kSlots, t = p % kNQ, hf = p / kNQ;
        if (!wait_bounded(o_done(kNQ - 1), 0)) {  // every MMA has completed: every slot is free
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(slot_full(slot), L::kTile);
        const uint32_t dst = base + L::kKV + slot * L::kTile;
        const int cols = args.acc_f32 ? 32 : 64;  // columns per box
        for (int bx = 0; bx < D / 64; ++bx)
          tma_load_4d(dst + bx * L::kBox, &tm_acc, slot_full(slot), (hf * (D / 64) + bx) * cols, h,
                      q0 + t * kBM, b);
        ++issued;
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
          } else {
            // tile t's O is final once this P V is: its epilogue need not wait for the other tile's
            tc_commit(o_done(t));
          }
        }
        if (!ok) break;
      }
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
      // columns past the range end, and (causal) keys after this row, are masked
      int valid = args.n_kv - j * kBN;
      if (kCausal) valid = min(valid, q0 + t * kBM + row - args.kv_begin - j * kBN + 1);
      if (valid < kBN) {
#pragma unroll
        for (int i = 0; i < kBN; ++i)
          if (i >= valid) s[i] = -INFINITY;
      }
      // row max: 3-input max over 4 independent chains, then a tree
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
        // The previous PV product of this tile is complete: S_t for block j was
        // issued after it and its commit covers every earlier MMA.
        const float m_new = fmaxf(m, mx);
        // (causal) rows that have seen no key yet keep m = -inf and O = 0
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
      }
      // (causal) a row that has seen no key yet keeps m = -inf: its weights are all zero
      const float m_use = (kCausal && m == -INFINITY) ? 0.f : m;
      const uint64_t nm2 = f2(-m_use, -m_use);
      uint64_t rs[4] = {0ull, 0ull, 0ull, 0ull};  // packed row-sum partials (0.0f bit patterns)
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
      mbar_arrive(p_full(t));
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(o_done(t), 0));
    if (kUpdate && ok) {  // this tile's O_acc halves have landed
      bool got = true;
      for (int hf = 0; hf < acc_halves; ++hf) {
        const int i = 2 * nblk + hf * kNQ + t;
        got = got && wait_bounded(slot_full(i % kSlots), (i / kSlots) & 1);
      }
      ok = __all_sync(0xffffffffu, got);
    }
    // Every warp of the warpgroup gets here (all waits above are bounded); the
    // epilogue's named barriers run only if all four warps are on the normal path.
    ok = named_barrier_and(1 + t, 128, ok);
    if (ok) {
      // Epilogue: O / l, converted, is written into this tile's Q buffer (no MMA
      // reads it any more) in the 128-byte-swizzled box layout of the O tensor
      // map, then stored by TMA as whole 128-byte rows.  fp32 output is twice the
      // buffer, so it goes in two rounds.
      tc_fence_after_sync();
      const int tile_q0 = q0 + t * kBM;
      // Output row = wc * (unnormalised O in TMEM) + wa * O_acc row.  Plain form:
      // wc = 1 / l, wa = 0 (a row with no visible key outputs zeros).
      float wc = l > 0.f ? 1.0f / l : 0.f, wa = 0.f;
      float lse_out = l > 0.f ? (m + log2f(l)) * 0.69314718055994531f : -INFINITY;
      if (kUpdate) {
        if (args.defer_wait) griddep_wait();  // LSE_acc is the previous launch's output
        // base 2: this range's LSE is m + log2 l; O_c = acc / l, so its weight
        // e^(LSE_c - L) / l is 2^(m - L2)
        const int q = tile_q0 + row;
        const float la = q < args.Sq ? args.lse_acc[((long long)b * args.H + h) * args.Sq + q] * 1.4426950408889634f
                                     : -INFINITY;
        const float lc = l > 0.f ? m + log2f(l) : -INFINITY;
        const float mx = fmaxf(la, lc);
        if (mx == -INFINITY) {  // neither part has seen a key: O = 0, LSE = -inf
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
      const uint32_t stage = base + L::kQ + t * L::kTile;
      const bool f32 = args.o_f32 != 0;
      const int W = f32 ? 32 : 64;          // output columns per 128-byte box row
      const int n_boxes = D / W;            // boxes of 128 rows x 128 bytes per tile
      constexpr int kPerRound = D / 64;     // boxes that fit in the staging buffer
      const uint32_t row_addr = stage + row * 128;
      const uint32_t sw = row & 7;          // 128-byte swizzle: chunk index XOR row % 8
      for (int r0 = 0; r0 < n_boxes; r0 += kPerRound) {
        if (r0 > 0) {  // the previous round's boxes must have been read before reuse
          if (row == 0) bulk_wait_read_all();
          named_barrier_sync(1 + t, 128);
        }
        for (int c = r0 * W / 32; c < (r0 + kPerRound) * W / 32; ++c) {
          uint32_t o[32];
          tmem_ld_x32(tO + c * 32, o);
          if (kUpdate) {
            // the same 32 columns of this row of O_acc, from its ring slot
            float a[32];
            if (args.acc_f32) {  // box c of the tile, in half c / (D / 64)
              const int i = 2 * nblk + (c / (D / 64)) * kNQ + t;
              const uint32_t src = base + L::kKV + (i % kSlots) * L::kTile + (c % (D / 64)) * L::kBox + row * 128;
#pragma unroll
              for (int u = 0; u < 8; ++u) {
                uint32_t x0, x1, x2, x3;
                ld_shared_v4(src + ((u ^ sw) << 4), x0, x1, x2, x3);
                a[4 * u] = __uint_as_float(x0), a[4 * u + 1] = __uint_as_float(x1);
                a[4 * u + 2] = __uint_as_float(x2), a[4 * u + 3] = __uint_as_float(x3);
              }
            } else {  // box c / 2 (64 bf16 columns), 16-byte chunks 4 * (c % 2) ..
              const int i = 2 * nblk + t;
              const uint32_t src = base + L::kKV + (i % kSlots) * L::kTile + (c / 2) * L::kBox + row * 128;
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
            for (int i = 0; i < 16; ++i) {
              float y0, y1;
              f2_split(f2_fma(f2(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1])), wc2,
                              f2_mul(f2(a[2 * i], a[2 * i + 1]), wa2)),
                       y0, y1);
              o[2 * i] = __float_as_uint(y0), o[2 * i + 1] = __float_as_uint(y1);
            }
          }
          const uint64_t il2 = kUpdate ? f2(1.f, 1.f) : wc2;
          const int col0 = c * 32;
          const uint32_t dst = row_addr + (col0 / W - r0) * L::kBox;
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
            tma_store_4d(&tm_o, stage + bx * L::kBox, (r0 + bx) * W, h, tile_q0, b);
          bulk_commit_group();
        }
      }
      if (row == 0) bulk_wait_read_all();
      const int q = tile_q0 + row;
      if (q < args.Sq) args.lse[((long long)b * args.H + h) * args.Sq + q] = lse_out;
    }
  }

  // plain form, deferred: the CTA may not end before the previous launch has
  if (!kUpdate && args.defer_wait && threadIdx.x == 0) griddep_wait();
  tc_fence_before_sync();
  __syncthreads();
  if (warp == kWarpMma) {
    tc_fence_after_sync();
    tmem_dealloc(tmem, kTmemCols);
  }
}

// One thread waits, with the same bounded wait as the attention kernel, on an
// mbarrier that nothing ever arrives at: the wait must give up, record the
// timeout in the error word and let the kernel return.
__global__ void wait_timeout_selftest_kernel() {
  __shared__ __align__(8) uint64_t bar;
  const uint32_t addr = smem_u32(&bar);
  mbar_init(addr, 1);
  mbar_fence_init();
  wait_bounded(addr, 0);
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

// [B, S, H, D] with element strides {b, s, h} (bf16 or fp32) as a 4-D map
// (d, h, s, b) with a box of 128 bytes x 1 x 128 rows x 1 and 128-byte swizzle;
// rows past S read as zero and are not written.
bool encode_bshd(CUtensorMap *map, const void *ptr, int B, int S, int H, int D, const int64_t st[3], bool f32) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (!enc) return false;
  const cuuint64_t es = f32 ? 4 : 2;
  cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)S, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)st[2] * es, (cuuint64_t)st[1] * es, (cuuint64_t)st[0] * es};
  cuuint32_t box[4] = {(cuuint32_t)(128 / es), 1, 128, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  CUresult r = enc(map, f32 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4,
                   const_cast<void *>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                   CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

template <int D, bool kCausal, bool kUpdate>
cudaError_t launch_typed(const CUtensorMap &tq, const CUtensorMap &tk, const CUtensorMap &tv, const CUtensorMap &to,
                         const CUtensorMap &tacc, const AttnArgs &a, int B, cudaStream_t stream) {
  using Lay = Layout<D>;
  static_assert(Lay::kAlloc <= 232448, "shared memory budget");
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  static std::atomic<bool> configured[64];  // set once the attribute is (other host threads may launch too)
  if (dev >= 64 || !configured[dev].load(std::memory_order_acquire)) {
    e = cudaFuncSetAttribute(attn_fwd_kernel<D, kCausal, kUpdate>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             Lay::kAlloc);
    if (e != cudaSuccess) return e;
    if (dev < 64) configured[dev].store(true, std::memory_order_release);
  }
  dim3 grid((a.Sq + kBM * kNQ - 1) / (kBM * kNQ), a.H, B);
  return launch_kernel(attn_fwd_kernel<D, kCausal, kUpdate>, grid, dim3(kThreads), Lay::kAlloc, stream, tq, tk, tv,
                       to, tacc, a);
}

}  // namespace

cudaError_t launch_attn_fwd(const void *q, const void *k, const void *v, int B, int H, int Sq, int Skv, int D,
                            const int64_t q_st[3], const int64_t kv_st[3], float scale, int kv_begin, int kv_end,
                            bool causal, void *o, bool o_f32, const int64_t o_st[3], float *lse, const void *o_acc,
                            bool acc_f32, const int64_t acc_st[3], const float *lse_acc, bool defer_wait,
                            cudaStream_t stream, const char **detail) {
  (void)Skv;
  CUtensorMap tq, tk, tv, to, tacc;
  const int n_kv = kv_end - kv_begin;
  const char *k0 = static_cast<const char *>(k) + (int64_t)kv_begin * kv_st[1] * 2;
  const char *v0 = static_cast<const char *>(v) + (int64_t)kv_begin * kv_st[1] * 2;
  if (!encode_bshd(&tq, q, B, Sq, H, D, q_st, false) || !encode_bshd(&tk, k0, B, n_kv, H, D, kv_st, false) ||
      !encode_bshd(&tv, v0, B, n_kv, H, D, kv_st, false) || !encode_bshd(&to, o, B, Sq, H, D, o_st, o_f32)) {
    *detail = "cuTensorMapEncodeTiled failed (driver entry point missing or strides/extents unsupported)";
    return cudaErrorInvalidValue;
  }
  const bool update = o_acc != nullptr;
  if (update && !encode_bshd(&tacc, o_acc, B, Sq, H, D, acc_st, acc_f32)) {
    *detail = "cuTensorMapEncodeTiled failed for the running output";
    return cudaErrorInvalidValue;
  }
  if (!update) tacc = to;
  AttnArgs a;
  a.H = H;
  a.Sq = Sq;
  a.n_kv = n_kv;
  a.kv_begin = kv_begin;
  a.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  a.o = o;
  a.o_sb = o_st[0];
  a.o_ss = o_st[1];
  a.o_sh = o_st[2];
  a.o_f32 = o_f32 ? 1 : 0;
  a.lse = lse;
  a.lse_acc = lse_acc;
  a.acc_f32 = acc_f32 ? 1 : 0;
  a.defer_wait = defer_wait ? 1 : 0;
  if (update) {
    if (causal)
      return D == 64 ? launch_typed<64, true, true>(tq, tk, tv, to, tacc, a, B, stream)
                     : launch_typed<128, true, true>(tq, tk, tv, to, tacc, a, B, stream);
    return D == 64 ? launch_typed<64, false, true>(tq, tk, tv, to, tacc, a, B, stream)
                   : launch_typed<128, false, true>(tq, tk, tv, to, tacc, a, B, stream);
  }
  if (causal)
    return D == 64 ? launch_typed<64, true, false>(tq, tk, tv, to, tacc, a, B, stream)
                   : launch_typed<128, true, false>(tq, tk, tv, to, tacc, a, B, stream);
  return D == 64 ? launch_typed<64, false, false>(tq, tk, tv, to, tacc, a, B, stream)
                 : launch_typed<128, false, false>(tq, tk, tv, to, tacc, a, B, stream);
}

cudaError_t launch_wait_timeout_selftest(cudaStream_t stream) {
  wait_timeout_selftest_kernel<<<1, 1, 0, stream>>>();
  return cudaGetLastError();
}

cudaError_t read_and_clear_attn_error(unsigned int *value) {
  cudaError_t e;
  unsigned int zero = 0;
  e = cudaMemcpyFromSymbol(value, g_device_error, sizeof(unsigned int));
  if (e != cudaSuccess) return e;
  return cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
}

}  // namespace ditattn
