// attn_fwd_1q_sm103.cu — the fused attention forward with one Q tile per CTA
// on GB300 (sm_103a), for head dimensions 192 and 256 (the persistent kernel
// runs the narrower ones).
//
// Same computation as the D = 64 / 128 kernel: out = softmax(scale·q·kᵀ +
// causal mask)·v per (batch, head) with the row logsumexp, following the five
// steps of "Profiling in PyTorch (Part 3): Attention is all you profile",
// section "Naive attention", walked tile by tile with a running softmax so the
// [S, S] scores never leave the chip (same page, "Why flash attention exists";
// FlashAttention-2 blog, "FlashAttention-2 Optimizations" §1-§3).
//
// Layout: one 128-row Q tile per CTA, K/V tiles of BN rows (64 at D = 192
// and 256), and two BN-column S buffers, so that the next S is computed
// while the softmax of the current one runs: the softmaxes of one tile follow
// each other back to back.  Q is the A operand of every S product of the CTA:
// it is put into TMEM once, so S = Q·Kᵀ is a TS product and shared memory only
// feeds K and V.  TMEM columns: S_b [BN·b, BN·b + BN) (P_b, 16-bit, over its
// first BN/2), Q [2·BN, 2·BN + D/2) (two 16-bit values per column), O in the
// last D.  The softmax computes its exponentials against the running
// reference before the tile's max is known and redoes them only when the tile
// moves the reference by more than the threshold of attn_fwd.h (2^32 for
// bf16, 2^8 for fp16).  At D = 256 two Q tiles' accumulators would fill TMEM
// on their own, and the 64 KB output tile does not fit beside the K/V rings,
// so this kernel is not persistent.
//
// Roles (192 threads): warps 0-3 softmax / correction / epilogue, one thread
// per query row (TMEM lane); warp 4 issues tcgen05.mma and owns TMEM; warp 5
// feeds the K and V rings with TMA.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_fwd.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace ea {
namespace {

constexpr int kQRows = 128;                      // rows of the Q tile
constexpr int kThreads1Q = 192;
constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainLimitNs = 1000000000ull;

// D: head dimension; BN: rows of one K/V tile
template <int D, int BN>
struct Layout1Q {
  static constexpr int kChunkBytes = BN * 128;   // one 64-column block of a K/V tile
  static constexpr int kTile = BN * D * 2;       // one K/V tile
  // ring stages: as many as shared memory holds, up to 5 (32 KB tiles: 3,
  // 24 KB: 4)
  static constexpr int kKStages = (kTile >= 32768) ? 3 : (kTile > 16384) ? 4 : 5;
  static constexpr int kVStages = kKStages;
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKStages * kTile;
  static constexpr int kBarOff = kVOff + kVStages * kTile;
  static constexpr int kKFull = 0, kKEmpty = kKFull + kKStages, kVFull = kKEmpty + kKStages,
                       kVEmpty = kVFull + kVStages, kSFull = kVEmpty + kVStages,  // [2]
                       kPFull = kSFull + 2,                                         // [2], 128
                       kQTmem = kPFull + 2,                                         // 128 arrivals
                       kPvDone = kQTmem + 1, kOFull = kPvDone + 1, kDrain = kOFull + 1,
                       kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  // the epilogue stages O (128 rows x D 16-bit values) in the K ring
  static_assert(kKStages * kTile >= kQRows * D * 2, "O staging must fit the K ring");
  // TMEM: two S buffers of BN columns, then Q (D/2 columns), O in the last D
  static constexpr uint32_t kTmemCols = 512, kQCol = 2 * BN, kOCol = kTmemCols - D;
  static_assert(kQCol + D / 2 <= kOCol && kOCol + D <= kTmemCols, "TMEM budget exceeded");
};

enum : int { kSiteProdK = 0x3100, kSiteProdV = 0x3200, kSiteMmaQ = 0x3300, kSiteMmaK = 0x3400,
             kSiteMmaV = 0x3500, kSiteMmaP = 0x3600, kSiteSoftS = 0x3700, kSiteSoftPv = 0x3800,
             kSiteSoftO = 0x3900 };
// debug-check sites (-DATTN_DEBUG)
enum : int { kChkQLoad = 0x5101, kChkQTmem, kChkSTmem, kChkPTmem, kChkOTmem, kChkStage, kChkStore,
             kChkLse, kChkLoadK, kChkLoadV, kChkMmaK, kChkMmaV, kChkMmaTmem };

template <int D, int BN, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kThreads1Q, 1) attn_fwd_1q_kernel(const __grid_constant__ Fwd1QParams p) {
  using L = Layout1Q<D, BN>;
  constexpr int kKvRows = BN;
  constexpr int kChunkBytes = L::kChunkBytes;
  constexpr int kD = D;
  constexpr int kTile = L::kTile;
  constexpr int kKStages = L::kKStages, kVStages = L::kVStages;
  constexpr int kKOff = L::kKOff, kVOff = L::kVOff, kBarOff = L::kBarOff, kMiscOff = L::kMiscOff;
  constexpr int kKFull = L::kKFull, kKEmpty = L::kKEmpty, kVFull = L::kVFull, kVEmpty = L::kVEmpty;
  constexpr int kSFull = L::kSFull, kPFull = L::kPFull, kQTmem = L::kQTmem, kPvDone = L::kPvDone;
  constexpr int kOFull = L::kOFull, kDrain = L::kDrain;
  constexpr uint32_t kQCol = L::kQCol, kOCol = L::kOCol, kTmemCols = L::kTmemCols;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto bar = [sb](int idx) -> uint32_t { return sb + kBarOff + 8u * idx; };
  const uint32_t tmem_slot = sb + kMiscOff;
  const uint32_t abort_addr = sb + kMiscOff + 4;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const DbgBounds dbb{p.status, sb, smem_u32(smem_raw) + static_cast<uint32_t>(L::kAlloc), p.S,
                      p.d_cols, p.BH};

  // Q tile i of slice bh, in the order of the grid schedule (schedule.h):
  // heavy tiles by L2-sized groups of heads, then the light ones over all heads
  int bh, i;
  schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh, &i);
  int nkv = CAUSAL ? (i + 1) * (kQRows / BN) : p.n_kt;  // K/V tiles this Q tile meets
  if (nkv > p.n_kt) nkv = p.n_kt;

  // A softmax thread's row of Q, requested before the set-up below so that
  // the load's latency overlaps it: all of the row's 16-byte loads are in
  // flight at once (rows past S and columns past d_cols load nothing and
  // hold zero).  It goes into TMEM once the allocation exists.
  uint32_t qw[kD / 2];
  if (warp < 4) {
    const int grow = i * kQRows + warp * 32 + lane;
    const bool valid = grow < p.S;
    const uint16_t* qr = p.q + (valid ? (int64_t)bh * p.S + grow : 0) * p.d_cols;
#pragma unroll
    for (int u = 0; u < kD / 8; ++u) {
      const int col = 8 * u;
      const uint4 x = valid && col < p.d_cols && dbg_row(dbb, bh, grow, col, 8, kChkQLoad)
                          ? __ldg(reinterpret_cast<const uint4*>(qr + col))
                          : make_uint4(0u, 0u, 0u, 0u);
      qw[4 * u] = x.x, qw[4 * u + 1] = x.y, qw[4 * u + 2] = x.z, qw[4 * u + 3] = x.w;
    }
  }

  if (threadIdx.x == 0) {
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(bar(kKFull + s), 1);
      mbar_init(bar(kKEmpty + s), 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(bar(kVFull + s), 1);
      mbar_init(bar(kVEmpty + s), 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(kSFull + b), 1);
      mbar_init(bar(kPFull + b), 128);
    }
    mbar_init(bar(kQTmem), 128);
    mbar_init(bar(kPvDone), 1);
    mbar_init(bar(kOFull), 1);
    mbar_init(bar(kDrain), 1);
    st_volatile_shared(abort_addr, 0);
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = static_cast<uint32_t>(ld_volatile_shared(tmem_slot));
  const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};

  if (warp < 4) {
    // ======================= softmax / correction / epilogue =======================
    const int row = warp * 32 + lane;
    const int grow = i * kQRows + row;
    const bool valid = grow < p.S;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    const uint32_t tO = tmem_base + lane_bits + kOCol;
    {
      // this row of Q into TMEM, 32 columns (64 values) per store
#pragma unroll
      for (int c = 0; c < kD / 64; ++c)
        if (dbg_warp(dbg_tmem(dbb, tmem_base + lane_bits + kQCol + 32 * c, 32, warp, kChkQTmem)))
          tmem_st_32x32b_x32(tmem_base + lane_bits + kQCol + 32 * c,
                             *reinterpret_cast<const uint32_t(*)[32]>(&qw[32 * c]));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(kQTmem));
    }
    const float sl2 = p.scale_log2;
    float m = -INFINITY;  // reference max (log2 units) of the exponentials in O and l
    float l = 0.f;        // running sum of p: gives the logsumexp
    float lq = 0.f;       // l plus each tile's rounding error of its largest p (normalises O)
    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      const int b = j & 1;
      ok = __all_sync(0xffffffffu, wait_bounded(bar(kSFull + b), (j >> 1) & 1, ctl,
                                                kSiteSoftS | (j & 0xff)));
      if (!ok) break;
      tc_fence_after_sync();
      const uint32_t tS = tmem_base + lane_bits + BN * b;
      uint32_t s[BN / 32][32];
      if (!dbg_warp(dbg_tmem(dbb, tS, BN, warp, kChkSTmem))) {
        ok = false;
        break;
      }
#pragma unroll
      for (int g = 0; g < BN / 32; ++g) tmem_ld_32x32b_x32(tS + 32 * g, s[g]);
      tmem_ld_wait();
#pragma unroll
      for (int g = 0; g < BN / 32; ++g) reg_fence(s[g]);
      // allowed key columns of this tile: 0 .. lim (causal: key <= query; key < S)
      int lim = p.S - 1 - j * kKvRows;
      if (CAUSAL) lim = min(lim, grow - j * kKvRows);
      if (!valid) lim = -1;
      if (lim < BN - 1) {
#pragma unroll
        for (int c = 0; c < BN; ++c)
          if (c > lim) s[c >> 5][c & 31] = __float_as_uint(-INFINITY);
      }
      float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // four independent chains
#pragma unroll
      for (int c = 0; c < BN; ++c) m4[c & 3] = fmaxf(m4[c & 3], __uint_as_float(s[c >> 5][c & 31]));
      const float mx = fmaxf(fmaxf(m4[0], m4[1]), fmaxf(m4[2], m4[3]));
      const float m_tile = mx * sl2;
      // exponentials against the current reference, computed before the
      // reference update is known; redone only when the tile moves it
      const float2 sl2x2 = make_float2(sl2, sl2);
      float2 rs2[4];
      uint32_t pk[BN / 64][32];
      auto exps = [&](float neg_m) {
        const float2 nm2 = make_float2(neg_m, neg_m);
#pragma unroll
        for (int a = 0; a < 4; ++a) rs2[a] = make_float2(0.f, 0.f);
#pragma unroll
        for (int g = 0; g < BN / 64; ++g)
#pragma unroll
          for (int e2 = 0; e2 < 32; ++e2) {
            const int h = 2 * g + (e2 >> 4), e = (2 * e2) & 31;
            const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[h][e]), __uint_as_float(s[h][e + 1])),
                                        sl2x2, nm2);
            const float p0 = ex2_approx(x.x), p1 = ex2_approx(x.y);
            rs2[e2 & 3] = __fadd2_rn(rs2[e2 & 3], make_float2(p0, p1));
            pk[g][e2] = pack_x2<F16>(p0, p1);
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
      if (dbg_warp(dbg_tmem(dbb, tS, BN / 2, warp, kChkPTmem))) {
#pragma unroll
        for (int g = 0; g < BN / 64; ++g) tmem_st_32x32b_x32(tS + 32 * g, pk[g]);
      }
      const float2 ra = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
      const float rs0 = ra.x, rs1 = ra.y;
      const float rs = rs0 + rs1;
      const float pmax = ex2_approx(fmaf(mx, sl2, neg_m));
      l = l * alpha + rs;
      lq = lq * alpha + (rs + (round_to_x<F16>(pmax) - pmax));
      // correction: O of a row whose reference moved is rescaled before PV_j
      // accumulates into it; PV_{j-1} must have completed first
      if (any_moved) {
        if (j > 0) {
          ok = __all_sync(0xffffffffu, wait_bounded(bar(kPvDone), (j - 1) & 1, ctl,
                                                    kSiteSoftPv | (j & 0xff)));
          if (!ok) break;
          tc_fence_after_sync();
#pragma unroll 1
          for (int c = 0; c < kD / 32 && dbg_warp(dbg_tmem(dbb, tO + 32 * c, 32, warp, kChkOTmem));
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
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(kPFull + b));
    }

    // ---- epilogue: O / lq → 16-bit → swizzled staging (K ring) → TMA store; lse
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(kOFull), 0, ctl, kSiteSoftO));
    if (ok) {
      tc_fence_after_sync();
      const float inv_l = lq > 0.f ? 1.f / lq : 0.f;
      // column blocks of 64 (128 bytes per row), 128 rows each (16 KB); the
      // two 32-column loads of a block are in flight together
#pragma unroll 1
      for (int c2 = 0; c2 < kD / 64 && dbg_warp(dbg_tmem(dbb, tO + 64 * c2, 64, warp, kChkOTmem));
           ++c2) {
        uint32_t o[2][32];
        tmem_ld_32x32b_x32(tO + 64 * c2, o[0]);
        tmem_ld_32x32b_x32(tO + 64 * c2 + 32, o[1]);
        tmem_ld_wait();
        reg_fence(o[0]);
        reg_fence(o[1]);
#pragma unroll
        for (int unit = 0; unit < 8; ++unit) {  // 16-byte unit within the 128-byte row
          const uint32_t addr = sb + kKOff + c2 * (kQRows * 128) + row * 128 +
                                ((unit ^ (row & 7)) << 4);
          const uint32_t* src = &o[unit >> 2][(unit & 3) * 8];
          uint32_t w[4];
#pragma unroll
          for (int e = 0; e < 4; ++e)
            w[e] = pack_x2<F16>(__uint_as_float(src[2 * e]) * inv_l,
                                __uint_as_float(src[2 * e + 1]) * inv_l);
          if (dbg_smem(dbb, addr, 16, 16, kChkStage)) st_shared_v4(addr, w[0], w[1], w[2], w[3]);
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      // this warp's 32 rows, if any of them is inside the tensor; a chunk
      // wholly past the tensor's columns is not stored either
      const int y0 = i * kQRows + warp * 32;
      if (lane == 0 && y0 < p.S) {
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          const uint32_t src = sb + kKOff + c * (kQRows * 128) + warp * 32 * 128;
          if (64 * c < p.d_cols && dbg_tma(dbb, src, 32 * 128, c * 64, y0, bh, true, kChkStore))
            tma_store_3d(&p.tm_o, src, c * 64, y0, bh);
        }
        tma_store_commit();
      }
      if (valid && dbg_row(dbb, bh, grow, 0, 0, kChkLse))
        p.lse[(int64_t)bh * p.S + grow] = (m + __log2f(l)) * kLn2;
      if (lane == 0) tma_store_wait_all();
    }
    tc_fence_before_sync();
  } else if (warp == 5) {
    // ======================= TMA producer: K and V rings =======================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_o);
      const uint64_t pol = l2_policy_evict_last();
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        const int ks = j % kKStages;
        ok = wait_bounded(bar(kKEmpty + ks), ((j / kKStages) & 1) ^ 1, ctl, kSiteProdK | (j & 0xff));
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kKFull + ks), kTile);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          // a skipped copy leaves the stage's transaction count short: the
          // consumer's bounded wait then ends the kernel
          const uint32_t dst = sb + kKOff + ks * kTile + c * kChunkBytes;
          if (dbg_tma(dbb, dst, kChunkBytes, c * 64, j * kKvRows, bh, false, kChkLoadK))
            tma_load_3d(dst, &p.tm_k, bar(kKFull + ks), c * 64, j * kKvRows, bh, pol);
        }
        k_issued = j + 1;
        const int vs = j % kVStages;
        ok = wait_bounded(bar(kVEmpty + vs), ((j / kVStages) & 1) ^ 1, ctl, kSiteProdV | (j & 0xff));
        if (!ok) break;
        mbar_arrive_expect_tx(bar(kVFull + vs), kTile);
#pragma unroll
        for (int c = 0; c < kD / 64; ++c) {
          const uint32_t dst = sb + kVOff + vs * kTile + c * kChunkBytes;
          if (dbg_tma(dbb, dst, kChunkBytes, c * 64, j * kKvRows, bh, false, kChkLoadV))
            tma_load_3d(dst, &p.tm_v, bar(kVFull + vs), c * 64, j * kKvRows, bh, pol);
        }
        v_issued = j + 1;
      }
      if (ok) {
        for (int j = max(nkv - kKStages, 0); j < nkv && ok; ++j)
          ok = wait_bounded(bar(kKEmpty + j % kKStages), (j / kKStages) & 1, ctl, kSiteProdK | 0xff);
        for (int j = max(nkv - kVStages, 0); j < nkv && ok; ++j)
          ok = wait_bounded(bar(kVEmpty + j % kVStages), (j / kVStages) & 1, ctl, kSiteProdV | 0xff);
      }
      if (!ok) {
        for (int j = max(k_issued - kKStages, 0); j < k_issued; ++j)
          wait_drain(bar(kKFull + j % kKStages), (j / kKStages) & 1, kDrainLimitNs);
        for (int j = max(v_issued - kVStages, 0); j < v_issued; ++j)
          wait_drain(bar(kVFull + j % kVStages), (j / kVStages) & 1, kDrainLimitNs);
      }
    }
  } else {
    // ======================= tcgen05 issuer (warp 4) =======================
    // The whole warp runs the issue code; each product and commit is
    // predicated on the elected lane (mma_ts_p and co.), so that the warp
    // never branches around them: the waits stay warp-wide and converged,
    // which measured faster than a branch around each step's products.
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = instr_desc_16bit(kQRows, kKvRows, false, false, F16);
    constexpr uint32_t kIdescO = instr_desc_16bit(kQRows, kD, false, true, F16);
    constexpr uint32_t kTileUnits = kTile >> 4;
    const uint64_t dk = smem_desc_sw128(sb + kKOff, 16, 1024);
    const uint64_t dv = smem_desc_sw128(sb + kVOff, kChunkBytes, 1024);
    auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
    };
    // S(j) into buffer j & 1: Q (TMEM, 8 columns per K step) · K_jᵀ (K-major)
    auto issue_s = [&](int j) {
      if (!dbg_smem(dbb, sb + kKOff + (j % kKStages) * kTile, kTile, 1024, kChkMmaK) ||
          !dbg_tmem_cols(dbb, tmem_base + BN * (j & 1), BN, kChkMmaTmem) ||
          !dbg_tmem_cols(dbb, tmem_base + kQCol, kD / 2, kChkMmaTmem))
        return;  // no commit: the softmax's bounded wait ends the kernel
      const uint64_t db = dk + (j % kKStages) * kTileUnits;
#pragma unroll
      for (int kk = 0; kk < kD / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ts_p(leader, tmem_base + BN * (j & 1), tmem_base + kQCol + kk * 8, db + off, kIdescS,
                 kk > 0 ? 1u : 0u);
      }
      mma_commit_p(leader, bar(kSFull + (j & 1)));
      mma_commit_p(leader, bar(kKEmpty + j % kKStages));
    };
    bool ok = wait_warp(bar(kQTmem), 0, kSiteMmaQ);
    for (int j0 = 0; j0 < 2 && j0 < nkv && ok; ++j0) {
      ok = wait_warp(bar(kKFull + j0 % kKStages), (j0 / kKStages) & 1, kSiteMmaK | j0);
      if (!ok) break;
      tc_fence_after_sync();
      issue_s(j0);
    }
    for (int j = 0; j < nkv && ok; ++j) {
      const int b = j & 1;
      ok = wait_warp(bar(kPFull + b), (j >> 1) & 1, kSiteMmaP | (j & 0xff));
      if (ok) ok = wait_warp(bar(kVFull + j % kVStages), (j / kVStages) & 1, kSiteMmaV | (j & 0xff));
      if (!ok) break;
      tc_fence_after_sync();
      if (dbg_smem(dbb, sb + kVOff + (j % kVStages) * kTile, kTile, 1024, kChkMmaV) &&
          dbg_tmem_cols(dbb, tmem_base + kOCol, kD, kChkMmaTmem)) {
        const uint64_t db = dv + (j % kVStages) * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < kKvRows / 16; ++kk)  // O += P_b · V_j, 16 keys per step
          mma_ts_p(leader, tmem_base + kOCol, tmem_base + BN * b + kk * 8, db + kk * (2048 >> 4),
                   kIdescO, (j > 0 || kk > 0) ? 1u : 0u);
        mma_commit_p(leader, bar(kPvDone));
        mma_commit_p(leader, bar(kVEmpty + j % kVStages));
      }
      if (j + 2 < nkv) {
        ok = wait_warp(bar(kKFull + (j + 2) % kKStages), ((j + 2) / kKStages) & 1,
                       kSiteMmaK | ((j + 2) & 0xff));
        if (!ok) break;
        tc_fence_after_sync();
        issue_s(j + 2);  // overwrites P_b: PV_j was issued first
      }
    }
    if (leader) {
      if (ok) mma_commit(bar(kOFull));
      mma_commit(bar(kDrain));
      wait_drain(bar(kDrain), 0, kDrainLimitNs);
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == 4) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, kTmemCols);
  }
}

template <int D, int BN, bool CAUSAL, bool F16>
cudaError_t launch_1q(const Fwd1QParams& p, cudaStream_t stream) {
  auto kern = attn_fwd_1q_kernel<D, BN, CAUSAL, F16>;
  constexpr int kAlloc = Layout1Q<D, BN>::kAlloc;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.BH * p.n_qt), 1, 1);
  cfg.blockDim = dim3(kThreads1Q, 1, 1);
  cfg.dynamicSmemBytes = kAlloc;
  cfg.stream = stream;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

template <int D>
cudaError_t launch_1q_d(const Fwd1QParams& p, bool causal, bool f16, cudaStream_t stream) {
  if (f16) return causal ? launch_1q<D, 64, true, true>(p, stream) : launch_1q<D, 64, false, true>(p, stream);
  return causal ? launch_1q<D, 64, true, false>(p, stream) : launch_1q<D, 64, false, false>(p, stream);
}

cudaError_t fwd1q_launch(const Fwd1QParams& p, int D, bool causal, bool f16, cudaStream_t stream) {
  if (D == 192) return launch_1q_d<192>(p, causal, f16, stream);
  if (D == 256) return launch_1q_d<256>(p, causal, f16, stream);
  return cudaErrorInvalidValue;
}

}  // namespace ea
