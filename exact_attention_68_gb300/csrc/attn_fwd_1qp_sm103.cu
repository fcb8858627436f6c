// attn_fwd_1qp_sm103.cu — the one-Q-tile forward run persistently on GB300
// (sm_103a): one CTA per SM walks Q tiles one after another.
//
// Same computation as the other forward kernels: out = softmax(scale·q·kᵀ +
// causal mask)·v per (batch, head) with the row logsumexp, the five steps of
// "Profiling in PyTorch (Part 3): Attention is all you profile", section
// "Naive attention", walked K/V tile by K/V tile with a running softmax so
// the [S, S] scores never leave the chip (same page, "Why flash attention
// exists"; FlashAttention-2 blog, "FlashAttention-2 Optimizations" §1-§3: few
// non-matmul operations, causal tiles skipped, work split over the sequence).
//
// Why persistent.  With one CTA per Q tile, every tile pays its own start
// (barrier and TMEM set-up, Q load, first S product, first softmax) and its
// own end (last P·V, output store, CTA exit and the launch of the next CTA on
// the SM): about 10^4 cycles, as much as 7 K/V steps of the loop.  Here the
// CTA resident on an SM keeps going: while tile k drains, tile k+1's Q is
// already in tensor memory and its first two S products are queued behind
// tile k's last P·V.
//
// Which tile comes next.  The grid still has one CTA per Q tile, in the order
// of the schedule (schedule.h); a CTA that is running asks the hardware for
// the next CTA of the grid that has not been launched (cluster launch
// control).  If granted, that CTA is never launched and its tile is done here;
// once refused, the CTA ends after its current tile.  So tiles run in the
// schedule's order and an SM that finishes early takes more of them, as with
// a grid of one CTA per tile, without a counter in global memory.
//
// L2: K and V are loaded with an evict-last policy, Q rows and the output,
// each touched once, with evict-first, so that the heads in flight keep their
// K/V in L2 (the grid order of schedule.h groups heads for that).
//
// Layout (D = 128; D = 64 halves the tiles): K and V rings of 128-row tiles
// (3 + 3 stages of 32 KB), a 32 KB staging buffer for the output, and a ring
// of four tile slots that the producer fills.  TMEM columns: S buffers
// [0, 128) and [128, 256) (P, 16-bit, over the first 64 columns of its S),
// two Q slots of D/2 columns from 256 (the tile's Q rows as the A operand of
// every S product; two 16-bit values per column), O in the last D.  K/V steps
// are counted over the whole run of the CTA: step g uses S buffer g & 1 and
// ring stage g mod stages, so phases carry over from one tile to the next.
//
// Roles (192 threads): warps 0-3 softmax, correction and epilogue, one thread
// per query row (TMEM lane); warp 4 issues tcgen05.mma and owns TMEM; warp 5
// (one lane) feeds the K and V rings with TMA, asks for the next tile and
// publishes it in the tile ring.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_fwd.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace ea {
namespace {

constexpr int kRowsP = 128;  // rows of a Q tile and of a K/V tile
constexpr int kThreadsP = 192;
constexpr float kLn2P = 0.6931471805599453f;
constexpr uint64_t kDrainLimitNsP = 1000000000ull;
constexpr int kSlots = 4;  // tile ring
// The producer asks for the next tile after issuing the loads of the step
// this many steps before its current tile's last one, and settles it after
// the last: late enough that the choice of the next tile is made when this SM
// is about to be free (as the hardware would launch a CTA), early enough that
// the answer is back before the other roles need it.
constexpr int kAskAhead = 2;

template <int D>
struct LayoutP {
  static constexpr int kChunkBytes = kRowsP * 128;  // 64 columns of a 128-row tile
  static constexpr int kTile = kRowsP * D * 2;
  static constexpr int kKStages = (kTile >= 32768) ? 3 : 5;
  static constexpr int kVStages = (kTile >= 32768) ? 3 : 5;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKStages * kTile;
  static constexpr int kStageOff = kVOff + kVStages * kTile;  // output staging
  static constexpr int kRespOff = kStageOff + kTile;          // launch-control response, 16 B
  static constexpr int kInfoOff = kRespOff + 16;              // tile ring: kSlots ints (16 B each)
  static constexpr int kBarOff = kInfoOff + kSlots * 16;
  static constexpr int kKFull = 0, kKEmpty = kKFull + kKStages, kVFull = kKEmpty + kKStages,
                       kVEmpty = kVFull + kVStages,
                       kSFull = kVEmpty + kVStages,  // [2]
                       kPFull = kSFull + 2,          // [2], 128 arrivals
                       kQTmem = kPFull + 2,          // [2] Q slots, 128 arrivals
                       kPvDone = kQTmem + 2, kOFull = kPvDone + 1,
                       kInfoFull = kOFull + 1,         // [kSlots]
                       kInfoEmpty = kInfoFull + kSlots,  // [kSlots], 5 arrivals
                       kClc = kInfoEmpty + kSlots, kDrain = kClc + 1, kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  static_assert((kStageOff & 1023) == 0, "staging buffer must be 1024-byte aligned");
  static constexpr uint32_t kTmemCols = 512, kQCol = 256, kOCol = kTmemCols - D;
  static_assert(kQCol + 2 * (D / 2) <= kOCol, "TMEM budget exceeded");
};

// Arrivals on a tile slot's empty barrier: the MMA warp and the four softmax warps.
constexpr uint32_t kInfoReaders = 5;

enum : int { kSitePProdK = 0x4100, kSitePProdV = 0x4200, kSitePProdInfo = 0x4300,
             kSitePClc = 0x4400, kSitePMmaQ = 0x4500, kSitePMmaK = 0x4600, kSitePMmaV = 0x4700,
             kSitePMmaP = 0x4800, kSitePMmaInfo = 0x4900, kSitePSoftS = 0x4a00,
             kSitePSoftPv = 0x4b00, kSitePSoftO = 0x4c00, kSitePSoftInfo = 0x4d00 };
// debug-check sites (-DATTN_DEBUG)
enum : int { kChkPQLoad = 0x5301, kChkPQTmem, kChkPSTmem, kChkPPTmem, kChkPOTmem, kChkPStage,
             kChkPStore, kChkPLse, kChkPLoadK, kChkPLoadV, kChkPMmaK, kChkPMmaV, kChkPMmaTmem,
             kChkPTile };

// K/V tiles Q tile i meets.
template <bool CAUSAL>
__device__ __forceinline__ int kv_steps(int i, int n_kt) {
  return CAUSAL ? (i + 1 < n_kt ? i + 1 : n_kt) : n_kt;
}

// QCP selects how a tile's Q rows reach tensor memory.  false: the softmax
// warps load them (the next tile's while the current one drains) and store
// them with tcgen05.st.  true: the producer brings them into the K ring with
// TMA, ahead of the tile's K tiles, and the MMA warp copies them in with
// tcgen05.cp, so the softmax warps go straight from a tile's last step to its
// epilogue; that shortens every tile hand-over, and pays off for short tiles
// (fwd1qp_launch chooses).
template <int D, bool CAUSAL, bool F16, bool QCP>
__global__ void __launch_bounds__(kThreadsP, 1) attn_fwd_1qp_kernel(const __grid_constant__ Fwd1QParams p) {
  using L = LayoutP<D>;
  constexpr int kTile = L::kTile, kChunkBytes = L::kChunkBytes;
  constexpr int kKStages = L::kKStages, kVStages = L::kVStages;
  constexpr uint32_t kQCol = L::kQCol, kOCol = L::kOCol;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint8_t* smem_gen = smem_raw + (sb - smem_u32(smem_raw));  // same window, generic
  auto bar = [sb](int idx) -> uint32_t { return sb + L::kBarOff + 8u * idx; };
  const uint32_t tmem_slot = sb + L::kMiscOff;
  const uint32_t abort_addr = sb + L::kMiscOff + 4;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const DbgBounds dbb{p.status, sb, smem_u32(smem_raw) + static_cast<uint32_t>(L::kAlloc), p.S,
                      p.d_cols, p.BH};
  const int n_units = p.BH * p.n_qt;  // CTAs of the grid, one per Q tile

  // The first tile is this CTA's own.  A softmax thread's row of its Q is
  // requested before the set-up below, so that the load's latency overlaps it.
  uint32_t qw[D / 2];
  if (!QCP && warp < 4) {
    int bh0, i0;
    schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh0, &i0);
    const int grow = i0 * kRowsP + warp * 32 + lane;
    const bool valid = grow < p.S;
    const uint16_t* qr = p.q + (valid ? (int64_t)bh0 * p.S + grow : 0) * p.d_cols;
#pragma unroll
    for (int u = 0; u < D / 8; ++u) {
      const int col = 8 * u;
      const uint4 x = valid && col < p.d_cols && dbg_row(dbb, bh0, grow, col, 8, kChkPQLoad)
                          ? ldg_policy(qr + col, l2_policy_evict_first())
                          : make_uint4(0u, 0u, 0u, 0u);
      qw[4 * u] = x.x, qw[4 * u + 1] = x.y, qw[4 * u + 2] = x.z, qw[4 * u + 3] = x.w;
    }
  }

  // With QCP the producer thread sets up the barriers and at once starts the
  // copy of the first tile's Q rows (K-ring position 0), so that the load's
  // latency overlaps the rest of the set-up.
  if (threadIdx.x == (QCP ? 5 * 32 : 0)) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kSFull + b), 1);
      mbar_init(bar(L::kPFull + b), 128);
      mbar_init(bar(L::kQTmem + b), 128);
    }
    for (int s = 0; s < kSlots; ++s) {
      mbar_init(bar(L::kInfoFull + s), 1);
      mbar_init(bar(L::kInfoEmpty + s), kInfoReaders);
    }
    mbar_init(bar(L::kPvDone), 1);
    mbar_init(bar(L::kOFull), 1);
    mbar_init(bar(L::kClc), 1);
    mbar_init(bar(L::kDrain), 1);
    st_volatile_shared(abort_addr, 0);
    fence_barrier_init();
    if constexpr (QCP) {
      int bh0, i0;
      schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh0, &i0);
      mbar_arrive_expect_tx(bar(L::kKFull + 0), kTile);
#pragma unroll
      for (int c = 0; c < D / 64; ++c) {
        const uint32_t dst = sb + L::kKOff + c * kChunkBytes;
        if (dbg_tma(dbb, dst, kChunkBytes, c * 64, i0 * kRowsP, bh0, false, kChkPLoadK))
          tma_load_3d(dst, &p.tm_q, bar(L::kKFull + 0), c * 64, i0 * kRowsP, bh0,
                      l2_policy_evict_first());
      }
    }
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = static_cast<uint32_t>(ld_volatile_shared(tmem_slot));
  const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};

  // The tile published in ring slot k & 3 (-1: none), after its full barrier.
  auto read_info = [&](int k, int site, bool* ok) -> int {
    *ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kInfoFull + (k & (kSlots - 1))),
                                               (k / kSlots) & 1, ctl, site | (k & 0xff)));
    if (!*ok) return -1;
    const int x = *reinterpret_cast<const volatile int*>(smem_gen + L::kInfoOff +
                                                         16 * (k & (kSlots - 1)));
    __syncwarp();
    if (lane == 0) mbar_arrive(bar(L::kInfoEmpty + (k & (kSlots - 1))));
    return x;
  };

  if (warp < 4) {
    // ======================= softmax / correction / epilogue =======================
    const int row = warp * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem_base + lane_bits + kOCol;
    const float sl2 = p.scale_log2;
    // Q row of tile 0 into Q slot 0, 32 columns (64 values) per store
    if constexpr (!QCP) {
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        if (dbg_warp(dbg_tmem(dbb, tmem_base + lane_bits + kQCol + 32 * c, 32, warp, kChkPQTmem)))
          tmem_st_32x32b_x32(tmem_base + lane_bits + kQCol + 32 * c,
                             *reinterpret_cast<const uint32_t(*)[32]>(&qw[32 * c]));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kQTmem + 0));
    }

    bool ok = true;
    int x = read_info(0, kSitePSoftInfo, &ok);
    int g = 0;  // K/V steps done by this CTA before the current tile
    for (int k = 0; ok && x >= 0; ++k) {
      if (!dbg(x < n_units, dbb, kChkPTile)) {
        ok = false;
        break;
      }
      int bh, i;
      schedule_unit(p.sched, x, &bh, &i);
      const int nkv = kv_steps<CAUSAL>(i, p.n_kt);
      const int grow = i * kRowsP + row;
      const bool valid = grow < p.S;
      float m = -INFINITY;  // reference max (log2 units) of the exponentials in O and l
      float l = 0.f;        // running sum of p: gives the logsumexp
      float lq = 0.f;       // l plus each tile's rounding error of its largest p (normalises O)
      for (int j = 0; j < nkv; ++j) {
        const int gj = g + j;
        const int b = gj & 1;
        ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kSFull + b), (gj >> 1) & 1, ctl,
                                                  kSitePSoftS | (gj & 0xff)));
        if (!ok) break;
        tc_fence_after_sync();
        const uint32_t tS = tmem_base + lane_bits + 128 * b;
        if (!dbg_warp(dbg_tmem(dbb, tS, 128, warp, kChkPSTmem))) {
          ok = false;
          break;
        }
        uint32_t s[4][32];
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) tmem_ld_32x32b_x32(tS + 32 * q4, s[q4]);
        tmem_ld_wait();
#pragma unroll
        for (int q4 = 0; q4 < 4; ++q4) reg_fence(s[q4]);
        // allowed key columns of this tile: 0 .. lim (causal: key <= query; key < S)
        int lim = p.S - 1 - j * kRowsP;
        if (CAUSAL) lim = min(lim, grow - j * kRowsP);
        if (!valid) lim = -1;
        if (lim < kRowsP - 1) {
#pragma unroll
          for (int c = 0; c < kRowsP; ++c)
            if (c > lim) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
        }
        float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
        for (int c = 0; c < kRowsP; ++c)
          m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(s[c >> 5][c & 31]));
        const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
        const float m_tile = mx * sl2;
        // exponentials against the current reference, computed before the
        // reference update is known; redone only when the tile moves it
        const float2 sl2x2 = make_float2(sl2, sl2);
        float2 rs2[4];
        uint32_t pk[2][32];
        auto exps = [&](float neg_m) {
          const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
          for (int a = 0; a < 4; ++a) rs2[a] = make_float2(0.f, 0.f);
#pragma unroll
          for (int hh = 0; hh < 2; ++hh)
#pragma unroll
            for (int e2 = 0; e2 < 32; ++e2) {
              const int h = 2 * hh + (e2 >> 4), e = (2 * e2) & 31;
              const float2 xx = __ffma2_rn(
                  make_float2(__uint_as_float(s[h][e]), __uint_as_float(s[h][e + 1])), sl2x2, nm2);
              const float p0 = ex2_approx(xx.x), p1 = ex2_approx(xx.y);
              rs2[e2 & 3] = __fadd2_rn(rs2[e2 & 3], make_float2(p0, p1));
              pk[hh][e2] = pack_x2<F16>(p0, p1);
            }
        };
        const bool spec = m != -INFINITY;
        if (spec) exps(-m);
        float alpha = 1.f;
        bool moved = false;
        if (m == -INFINITY) {
          m = m_tile;  // first tile with an allowed key sets the reference
        } else if (m_tile > m + kRescaleThreshold<F16>) {
          alpha = ex2_approx(m - m_tile);
          m = m_tile;
          moved = true;
        }
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        const bool any_moved = __any_sync(0xffffffffu, moved);  // every lane, no short-circuit
        if (!spec || any_moved) exps(neg_m);
        if (dbg_warp(dbg_tmem(dbb, tS, 64, warp, kChkPPTmem))) {
          tmem_st_32x32b_x32(tS, pk[0]);
          tmem_st_32x32b_x32(tS + 32, pk[1]);
        }
        const float2 ra = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
        const float rs = ra.x + ra.y;
        const float pmax = ex2_approx(fmaf(mx, sl2, neg_m));
        l = l * alpha + rs;
        lq = lq * alpha + (rs + (round_to_x<F16>(pmax) - pmax));
        // correction: O of a row whose reference moved is rescaled before
        // P·V of this step accumulates into it; the previous step's P·V must
        // have completed first (the first step of a tile starts O afresh)
        if (any_moved && j > 0) {
          ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kPvDone), (gj - 1) & 1, ctl,
                                                    kSitePSoftPv | (gj & 0xff)));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < D / 32 && dbg_warp(dbg_tmem(dbb, tO + 32 * c, 32, warp, kChkPOTmem));
               ++c) {
            uint32_t o[32];
            tmem_ld_32x32b_x32(tO + 32 * c, o);
            tmem_ld_wait();
            reg_fence(o);
#pragma unroll
            for (int t = 0; t < 32; ++t) o[t] = __float_as_uint(__uint_as_float(o[t]) * alpha);
            tmem_st_32x32b_x32(tO + 32 * c, o);
          }
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kPFull + b));
      }
      if (!ok) break;
      g += nkv;

      // ---- the next tile (without QCP: its Q rows into the other Q slot; the
      // producer brought them into L2), so that its first S products can
      // start while this tile's output drains
      const int nx = read_info(k + 1, kSitePSoftInfo, &ok);
      if (!ok) break;
      if (!QCP && nx >= 0 && dbg(nx < n_units, dbb, kChkPTile)) {
        int nbh, ni;
        schedule_unit(p.sched, nx, &nbh, &ni);
        const int ngrow = ni * kRowsP + row;
        const bool nvalid = ngrow < p.S;
        const uint16_t* qr = p.q + (nvalid ? (int64_t)nbh * p.S + ngrow : 0) * p.d_cols;
        const uint32_t tq = tmem_base + lane_bits + kQCol + ((k + 1) & 1) * (D / 2);
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t w[32];
#pragma unroll
          for (int u = 0; u < 8; ++u) {
            const int col = 64 * c + 8 * u;
            const uint4 xq = nvalid && col < p.d_cols && dbg_row(dbb, nbh, ngrow, col, 8, kChkPQLoad)
                                 ? ldg_policy(qr + col, l2_policy_evict_first())
                                 : make_uint4(0u, 0u, 0u, 0u);
            w[4 * u] = xq.x, w[4 * u + 1] = xq.y, w[4 * u + 2] = xq.z, w[4 * u + 3] = xq.w;
          }
          if (dbg_warp(dbg_tmem(dbb, tq + 32 * c, 32, warp, kChkPQTmem)))
            tmem_st_32x32b_x32(tq + 32 * c, w);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(bar(L::kQTmem + ((k + 1) & 1)));
      }

      // ---- epilogue: O / lq → 16-bit → swizzled staging → TMA store; lse
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kOFull), k & 1, ctl, kSitePSoftO | (k & 0xff)));
      if (!ok) break;
      tc_fence_after_sync();
      if (lane == 0) tma_store_wait_read();  // this warp's previous store has read the staging rows
      __syncwarp();
      const float inv_l = lq > 0.f ? 1.f / lq : 0.f;
#pragma unroll 1
      for (int c2 = 0; c2 < D / 64 && dbg_warp(dbg_tmem(dbb, tO + 64 * c2, 64, warp, kChkPOTmem));
           ++c2) {
        uint32_t o[2][32];
        tmem_ld_32x32b_x32(tO + 64 * c2, o[0]);
        tmem_ld_32x32b_x32(tO + 64 * c2 + 32, o[1]);
        tmem_ld_wait();
        reg_fence(o[0]);
        reg_fence(o[1]);
#pragma unroll
        for (int unit = 0; unit < 8; ++unit) {  // 16-byte unit within the 128-byte row
          const uint32_t addr = sb + L::kStageOff + c2 * kChunkBytes + row * 128 +
                                ((unit ^ (row & 7)) << 4);
          const uint32_t* src = &o[unit >> 2][(unit & 3) * 8];
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_x2<F16>(__uint_as_float(src[2 * e]) * inv_l,
                                __uint_as_float(src[2 * e + 1]) * inv_l);
          if (dbg_smem(dbb, addr, 16, 16, kChkPStage)) st_shared_v4(addr, w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      // this warp's 32 rows, if any of them is inside the tensor; a chunk
      // wholly past the tensor's columns is not stored
      const int y0 = i * kRowsP + warp * 32;
      if (lane == 0 && y0 < p.S) {
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          const uint32_t src = sb + L::kStageOff + c * kChunkBytes + warp * 32 * 128;
          if (64 * c < p.d_cols && dbg_tma(dbb, src, 32 * 128, c * 64, y0, bh, true, kChkPStore))
            tma_store_3d_policy(&p.tm_o, src, c * 64, y0, bh, l2_policy_evict_first());
        }
        tma_store_commit();
      }
      if (valid && dbg_row(dbb, bh, grow, 0, 0, kChkPLse))
        p.lse[(int64_t)bh * p.S + grow] = (m + __log2f(l)) * kLn2P;
      x = nx;
    }
    if (lane == 0) tma_store_wait_all();
    tc_fence_before_sync();
  } else if (warp == 5) {
    // ======================= producer: tiles, K and V rings =======================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_o);
      tma_prefetch_desc(&p.tm_q);
      const uint64_t pol = l2_policy_evict_last();
      const uint64_t pol_q = l2_policy_evict_first();
      const uint32_t resp = sb + L::kRespOff;
      // K-ring positions / V steps whose loads were issued (with QCP the K ring
      // also carries each tile's Q rows; tile 0's went out during the set-up)
      int k_issued = QCP ? 1 : 0, v_issued = 0;
      uint32_t clc_n = 0;   // launch-control requests made
      bool clc_wait = false;  // a request is in flight
      bool ok = true;
      // publishes tile x (or -1) in ring slot k
      auto publish = [&](int k, int x) {
        if (!wait_bounded(bar(L::kInfoEmpty + (k & (kSlots - 1))), ((k / kSlots) & 1) ^ 1, ctl,
                          kSitePProdInfo | (k & 0xff)))
          return false;
        *reinterpret_cast<volatile int*>(const_cast<uint8_t*>(smem_gen) + L::kInfoOff +
                                         16 * (k & (kSlots - 1))) = x;
        mbar_arrive(bar(L::kInfoFull + (k & (kSlots - 1))));
        return true;
      };
      auto request = [&]() {
        mbar_arrive_expect_tx(bar(L::kClc), 16);
        clc_try_cancel(resp, bar(L::kClc));
        ++clc_n;
        clc_wait = true;
      };
      int x = static_cast<int>(blockIdx.x);
      ok = publish(0, x);
      int g = 0;
      for (int k = 0; ok && x >= 0; ++k) {
        int bh, i;
        schedule_unit(p.sched, x, &bh, &i);
        const int nkv = kv_steps<CAUSAL>(i, p.n_kt);
        const int jr = nkv > kAskAhead ? nkv - 1 - kAskAhead : 0;  // ask for the next tile
        int nx = -1;
        if (QCP && k > 0) {  // the tile's Q rows, ahead of its K tiles
          const int ks = k_issued % kKStages;
          ok = wait_bounded(bar(L::kKEmpty + ks), ((k_issued / kKStages) & 1) ^ 1, ctl,
                            kSitePProdK | (k_issued & 0xff));
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kKFull + ks), kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            const uint32_t dst = sb + L::kKOff + ks * kTile + c * kChunkBytes;
            if (dbg_tma(dbb, dst, kChunkBytes, c * 64, i * kRowsP, bh, false, kChkPLoadK))
              tma_load_3d(dst, &p.tm_q, bar(L::kKFull + ks), c * 64, i * kRowsP, bh, pol_q);
          }
          ++k_issued;
        }
        for (int j = 0; j < nkv; ++j) {
          const int gj = g + j;
          const int kp = QCP ? k_issued : gj;  // K-ring position of this K tile
          const int ks = kp % kKStages;
          ok = wait_bounded(bar(L::kKEmpty + ks), ((kp / kKStages) & 1) ^ 1, ctl,
                            kSitePProdK | (kp & 0xff));
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kKFull + ks), kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            // a skipped copy leaves the stage's transaction count short: the
            // consumer's bounded wait then ends the kernel
            const uint32_t dst = sb + L::kKOff + ks * kTile + c * kChunkBytes;
            if (dbg_tma(dbb, dst, kChunkBytes, c * 64, j * kRowsP, bh, false, kChkPLoadK))
              tma_load_3d(dst, &p.tm_k, bar(L::kKFull + ks), c * 64, j * kRowsP, bh, pol);
          }
          k_issued = kp + 1;
          const int vs = gj % kVStages;
          ok = wait_bounded(bar(L::kVEmpty + vs), ((gj / kVStages) & 1) ^ 1, ctl,
                            kSitePProdV | (gj & 0xff));
          if (!ok) break;
          mbar_arrive_expect_tx(bar(L::kVFull + vs), kTile);
#pragma unroll
          for (int c = 0; c < D / 64; ++c) {
            const uint32_t dst = sb + L::kVOff + vs * kTile + c * kChunkBytes;
            if (dbg_tma(dbb, dst, kChunkBytes, c * 64, j * kRowsP, bh, false, kChkPLoadV))
              tma_load_3d(dst, &p.tm_v, bar(L::kVFull + vs), c * 64, j * kRowsP, bh, pol);
          }
          v_issued = gj + 1;
          if (j == jr) request();
          if (j == nkv - 1) {
            // settle the next tile: the answer to the request, published for
            // the other roles (without QCP its Q rows are brought into L2)
            if (clc_wait) {
              ok = wait_bounded(bar(L::kClc), (clc_n - 1) & 1, ctl, kSitePClc | (k & 0xff));
              if (!ok) break;
              clc_wait = false;
              int first = -1;
              if (clc_granted(resp, &first) && first >= 0 && first < n_units) nx = first;
            }
            ok = publish(k + 1, nx);
            if (!ok) break;
            if (!QCP && nx >= 0) {
              int nbh, ni;
              schedule_unit(p.sched, nx, &nbh, &ni);
#pragma unroll
              for (int c = 0; c < D / 64; ++c) tma_prefetch_l2_3d(&p.tm_q, c * 64, ni * kRowsP, nbh);
            }
          }
        }
        if (!ok) break;
        g += nkv;
        x = nx;
      }
      if (ok) {
        // every stage released by the tensor core before this CTA may exit
        for (int gj = max(k_issued - kKStages, 0); gj < k_issued && ok; ++gj)
          ok = wait_bounded(bar(L::kKEmpty + gj % kKStages), (gj / kKStages) & 1, ctl,
                            kSitePProdK | 0xff);
        for (int gj = max(v_issued - kVStages, 0); gj < v_issued && ok; ++gj)
          ok = wait_bounded(bar(L::kVEmpty + gj % kVStages), (gj / kVStages) & 1, ctl,
                            kSitePProdV | 0xff);
      }
      if (!ok) {
        // let every copy and request this thread started complete before leaving
        for (int gj = max(k_issued - kKStages, 0); gj < k_issued; ++gj)
          wait_drain(bar(L::kKFull + gj % kKStages), (gj / kKStages) & 1, kDrainLimitNsP);
        for (int gj = max(v_issued - kVStages, 0); gj < v_issued; ++gj)
          wait_drain(bar(L::kVFull + gj % kVStages), (gj / kVStages) & 1, kDrainLimitNsP);
        if (clc_wait) wait_drain(bar(L::kClc), (clc_n - 1) & 1, kDrainLimitNsP);
      }
    }
  } else {
    // ======================= tcgen05 issuer (warp 4) =======================
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = instr_desc_16bit(kRowsP, kRowsP, false, false, F16);
    constexpr uint32_t kIdescO = instr_desc_16bit(kRowsP, D, false, true, F16);
    constexpr uint32_t kTileUnits = kTile >> 4;
    const uint64_t dk = smem_desc_sw128(sb + L::kKOff, 16, 1024);
    const uint64_t dv = smem_desc_sw128(sb + L::kVOff, kChunkBytes, 1024);
    auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
    };
    int kpos = 0;  // with QCP: K-ring positions consumed (each tile's Q, then its K tiles)
    // S of step gh into buffer gh & 1: Q (slot qs, 8 columns per K step) · K_ghᵀ,
    // K in ring position kp
    auto issue_s = [&](int gh, int qs, int kp) {
      const int ks = kp % kKStages;
      if (!dbg_smem(dbb, sb + L::kKOff + ks * kTile, kTile, 1024, kChkPMmaK) ||
          !dbg_tmem_cols(dbb, tmem_base + 128 * (gh & 1), 128, kChkPMmaTmem) ||
          !dbg_tmem_cols(dbb, tmem_base + kQCol + qs * (D / 2), D / 2, kChkPMmaTmem))
        return;  // no commit: the softmax's bounded wait ends the kernel
      const uint64_t db = dk + ks * kTileUnits;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ts(tmem_base + 128 * (gh & 1), tmem_base + kQCol + qs * (D / 2) + kk * 8, db + off,
               kIdescS, kk > 0 ? 1u : 0u);
      }
      mma_commit(bar(L::kSFull + (gh & 1)));
      mma_commit(bar(L::kKEmpty + ks));
    };
    // the first (up to) two S products of a tile starting at step g, Q in slot
    // qs.  With QCP the Q rows are first copied from the K ring into the
    // slot, which was last read by the S products of tile k - 2: complete by
    // now, as the P of tile k - 1's last step, which this warp has waited
    // for, comes after them.
    auto start_tile = [&](int g, int nkv, int qs, int k) {
      bool r;
      if constexpr (QCP) {
        const int ks = kpos % kKStages;
        r = wait_warp(bar(L::kKFull + ks), (kpos / kKStages) & 1, kSitePMmaQ | (k & 0xff));
        if (!r) return false;
        tc_fence_after_sync();
        if (leader && dbg_smem(dbb, sb + L::kKOff + ks * kTile, kTile, 1024, kChkPMmaK) &&
            dbg_tmem_cols(dbb, tmem_base + kQCol + qs * (D / 2), D / 2, kChkPMmaTmem)) {
          const uint64_t db = dk + ks * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk)
            tmem_cp_128x256b(tmem_base + kQCol + qs * (D / 2) + kk * 8,
                             db + (((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4));
          mma_commit(bar(L::kKEmpty + ks));
        }
        __syncwarp();
        ++kpos;
      } else {
        r = wait_warp(bar(L::kQTmem + qs), (k >> 1) & 1, kSitePMmaQ | (k & 0xff));
      }
      for (int j0 = 0; j0 < 2 && j0 < nkv && r; ++j0) {
        const int gh = g + j0;
        const int kp = QCP ? kpos : gh;
        r = wait_warp(bar(L::kKFull + kp % kKStages), (kp / kKStages) & 1, kSitePMmaK | (gh & 0xff));
        if (!r) break;
        tc_fence_after_sync();
        if (leader) issue_s(gh, qs, kp);
        __syncwarp();
        if constexpr (QCP) ++kpos;
      }
      return r;
    };

    bool ok = true;
    int x = read_info(0, kSitePMmaInfo, &ok);
    int g = 0;
    int nkv = 0;
    if (ok && x >= 0) {
      int bh, i;
      schedule_unit(p.sched, x, &bh, &i);
      nkv = kv_steps<CAUSAL>(i, p.n_kt);
      ok = start_tile(0, nkv, 0, 0);
    }
    for (int k = 0; ok && x >= 0; ++k) {
      const int qs = k & 1;
      for (int j = 0; j < nkv && ok; ++j) {
        const int gj = g + j;
        const int b = gj & 1;
        // V of this step has normally landed long before P: waiting for it
        // first keeps that wait off the path from P to its product
        ok = wait_warp(bar(L::kVFull + gj % kVStages), (gj / kVStages) & 1, kSitePMmaV | (gj & 0xff));
        if (ok) ok = wait_warp(bar(L::kPFull + b), (gj >> 1) & 1, kSitePMmaP | (gj & 0xff));
        if (!ok) break;
        tc_fence_after_sync();
        if (leader && dbg_smem(dbb, sb + L::kVOff + (gj % kVStages) * kTile, kTile, 1024, kChkPMmaV) &&
            dbg_tmem_cols(dbb, tmem_base + kOCol, D, kChkPMmaTmem)) {
          const uint64_t db = dv + (gj % kVStages) * kTileUnits;
#pragma unroll
          for (int kk = 0; kk < kRowsP / 16; ++kk)  // O += P_b · V, 16 keys per step
            mma_ts(tmem_base + kOCol, tmem_base + 128 * b + kk * 8, db + kk * (2048 >> 4), kIdescO,
                   (j > 0 || kk > 0) ? 1u : 0u);
          mma_commit(bar(L::kPvDone));
          mma_commit(bar(L::kVEmpty + gj % kVStages));
          if (j == nkv - 1) mma_commit(bar(L::kOFull));
        }
        __syncwarp();
        if (j + 2 < nkv) {
          const int kp = QCP ? kpos : gj + 2;
          ok = wait_warp(bar(L::kKFull + kp % kKStages), (kp / kKStages) & 1,
                         kSitePMmaK | ((gj + 2) & 0xff));
          if (!ok) break;
          tc_fence_after_sync();
          if (leader) issue_s(gj + 2, qs, kp);  // overwrites P_b: P·V of step gj was issued first
          __syncwarp();
          if constexpr (QCP) ++kpos;
        }
      }
      if (!ok) break;
      g += nkv;
      // the next tile: its first S products queue behind this tile's last P·V
      x = read_info(k + 1, kSitePMmaInfo, &ok);
      if (!ok || x < 0 || !dbg(x < n_units, dbb, kChkPTile)) break;
      int bh, i;
      schedule_unit(p.sched, x, &bh, &i);
      nkv = kv_steps<CAUSAL>(i, p.n_kt);
      ok = start_tile(g, nkv, (k + 1) & 1, k + 1);
    }
    if (leader) {
      mma_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, kDrainLimitNsP);
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == 4) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool F16, bool QCP>
cudaError_t launch_1qp(const Fwd1QParams& p, cudaStream_t stream) {
  auto kern = attn_fwd_1qp_kernel<D, CAUSAL, F16, QCP>;
  constexpr int kAlloc = LayoutP<D>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.BH * p.n_qt), 1, 1);
  cfg.blockDim = dim3(kThreadsP, 1, 1);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int D, bool QCP>
cudaError_t launch_1qp_q(const Fwd1QParams& p, bool causal, bool f16, cudaStream_t stream) {
  if (f16)
    return causal ? launch_1qp<D, true, true, QCP>(p, stream) : launch_1qp<D, false, true, QCP>(p, stream);
  return causal ? launch_1qp<D, true, false, QCP>(p, stream) : launch_1qp<D, false, false, QCP>(p, stream);
}

// Q through the K ring and tcgen05.cp (QCP) when a tile meets this many K/V
// steps on average or fewer: it makes each tile hand-over shorter, which
// measured 6 % faster on 2x16x4096x128 causal (16.5 steps a tile) and
// 8x16x2048x128 (16), but 1-2 % slower per step in long tiles.
constexpr int kQcpMaxAvgSteps = 24;

template <int D>
cudaError_t launch_1qp_d(const Fwd1QParams& p, bool causal, bool f16, cudaStream_t stream) {
  const int avg_steps = causal ? (p.n_kt + 1) / 2 : p.n_kt;
  return avg_steps <= kQcpMaxAvgSteps ? launch_1qp_q<D, true>(p, causal, f16, stream)
                                      : launch_1qp_q<D, false>(p, causal, f16, stream);
}

}  // namespace

cudaError_t fwd1qp_launch(const Fwd1QParams& p, int D, bool causal, bool f16, cudaStream_t stream) {
  if (D == 128) return launch_1qp_d<128>(p, causal, f16, stream);
  if (D == 64) return launch_1qp_d<64>(p, causal, f16, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ea
