// attn_fwd_sm103.cu — fused exact attention forward for GB300 (sm_103a).
//
// Computes, per (batch, head), out = softmax(scale·q·kᵀ + causal mask)·v and
// the row logsumexp, as defined step by step in "Profiling in PyTorch (Part 3):
// Attention is all you profile", section "Naive attention", evaluated the way
// that page's "Why flash attention exists" passage describes: K and V are
// walked in tiles with a running (online) softmax and the output accumulates
// tile by tile, so the [S, S] scores never leave the chip.  From the
// FlashAttention-2 blog ("FlashAttention-2 Optimizations"): §2 fully masked
// K/V tiles are skipped under the causal mask, §3 work is split over the
// sequence (one CTA per (b, h, 256 query rows)), §1 the softmax does as few
// non-matmul operations as it can (exp2 with the scale folded in, the 1/l
// normalisation deferred to the end, and the running max only moved when it
// grows by more than the threshold of attn_fwd.h, which bounds every exponent
// by that threshold and is exact because the same reference max scales both
// O and l).
//
// GB300 mapping (one CTA per SM: 225 KB of shared memory, all 512 TMEM columns):
//   warps 0-3   softmax/correction/epilogue for Q tile 0 (rows 0-127 of the unit)
//   warps 4-7   the same for Q tile 1 (rows 128-255).  One thread owns one query
//               row (its TMEM lane): row max and row sums need no shuffles.
//   warp 8      tcgen05 issuer (the warp waits together, one elected lane
//               issues): S_t = Q_t·K_jᵀ (A, B from smem) and
//               O_t += P_t·V_j (A = P from TMEM, B = V from smem, MN-major),
//               fp32 accumulators in TMEM; completion signalled by
//               tcgen05.commit on mbarriers.  Also owns the TMEM allocation.
//   warp 9      TMA producer: Q tiles once, then K_j / V_j through two rings of
//               shared-memory stages guarded by full/empty mbarriers.
//   warps 10-11 idle (they complete the control warpgroup for setmaxnreg).
// The softmax warpgroups run with 200 registers (a whole row of S stays in
// registers), the control warpgroup with 72.  While one softmax warpgroup
// works, the tensor core runs the other tile's MMAs (the two tiles ping-pong).
//
// TMEM columns: S_0 [0,128), S_1 [128,256), O_0 [256,256+D), O_1 [256+D,256+2D).
// P_t (bf16, two per 32-bit column) overwrites columns [0,64) of S_t.
//
// Grid: one CTA per work unit, in the order schedule.h sets out (heavy causal
// levels by L2-sized groups of heads, then the light levels over all heads).
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "attn_fwd.h"
#include "ptx.cuh"
#include "umma.cuh"

namespace ea {
namespace {

constexpr float kLn2 = 0.6931471805599453f;
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // bound on waits while tearing down

template <int D>
struct Layout {
  static constexpr int kTileBytes = kBlockM * D * 2;  // one 128-row bf16 tile
  static constexpr int kChunks = D / 64;              // 64-column (128-byte) swizzle blocks
  static constexpr int kChunkBytes = kBlockM * 128;   // 16 KB
  static constexpr int kKStages = (D == 128) ? 3 : 4;
  static constexpr int kVStages = (D == 128) ? 2 : 4;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + kQTilesPerUnit * kTileBytes;
  static constexpr int kVOff = kKOff + kKStages * kTileBytes;
  static constexpr int kBarOff = kVOff + kVStages * kTileBytes;
  // barrier indices (8 bytes each from kBarOff)
  static constexpr int kQFull = 0;                     // [2]  Q_t landed
  static constexpr int kKFull = kQFull + 2;            // [KS] K stage landed
  static constexpr int kKEmpty = kKFull + kKStages;    // [KS] K stage released by the MMAs
  static constexpr int kVFull = kKEmpty + kKStages;    // [VS]
  static constexpr int kVEmpty = kVFull + kVStages;    // [VS]
  static constexpr int kSFull = kVEmpty + kVStages;    // [2]  S_t computed
  static constexpr int kPFull = kSFull + 2;            // [2]  P_t stored (128 arrivals)
  static constexpr int kOFull = kPFull + 2;            // [2]  O_t final
  static constexpr int kDrain = kOFull + 2;            // MMA drain
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base (u32), abort flag (int)
  static constexpr int kBytes = kMiscOff + 16;
  static constexpr int kAlloc = kBytes + 1024;  // slack to align the base to 1024 B
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  static constexpr uint32_t kTmemCols = 512;
  static_assert(2 * 128 + 2 * D <= 512, "TMEM budget exceeded");
};

// Wait-site tags recorded in status[1] by the first wait that runs out.
enum : int {
  kSiteProducerK = 0x100, kSiteProducerV = 0x200, kSiteMmaQ = 0x300, kSiteMmaK = 0x400,
  kSiteMmaV = 0x500, kSiteMmaP = 0x600, kSiteSoftS = 0x700, kSiteSoftO = 0x800
};
// debug-check sites (-DATTN_DEBUG)
enum : int { kChkSTmem = 0x5001, kChkOTmem, kChkStage, kChkStore, kChkLse, kChkLoadQ, kChkLoadK,
             kChkLoadV, kChkMmaQ, kChkMmaK, kChkMmaV, kChkMmaTmem };

template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ FwdParams p) {
  using L = Layout<D>;
  extern __shared__ uint8_t smem_raw[];
  // 1024-byte aligned base of the shared window (128-byte swizzle atoms)
  const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto bar = [sb](int idx) -> uint32_t { return sb + L::kBarOff + 8u * idx; };
  const uint32_t tmem_slot = sb + L::kMiscOff;
  const uint32_t abort_addr = sb + L::kMiscOff + 4;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const DbgBounds dbb{p.status, sb, smem_u32(smem_raw) + static_cast<uint32_t>(L::kAlloc), p.S,
                      p.d_cols, p.B * p.H};

  // ---- work unit: (b·H + h, pair of Q tiles), from the grid schedule
  int bh, u;
  schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh, &u);
  const int qt0 = 2 * u;
  const int qt1 = 2 * u + 1;
  const int n0 = CAUSAL ? qt0 + 1 : p.n_qt;
  const int n1 = (qt1 < p.n_qt) ? (CAUSAL ? qt1 + 1 : p.n_qt) : 0;
  const int nkv = n0 > n1 ? n0 : n1;

  if (threadIdx.x == 0) {
#pragma unroll
    for (int t = 0; t < 2; ++t) {
      mbar_init(bar(L::kQFull + t), 1);
      mbar_init(bar(L::kSFull + t), 1);
      mbar_init(bar(L::kPFull + t), 128);
      mbar_init(bar(L::kOFull + t), 1);
    }
#pragma unroll
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
#pragma unroll
    for (int s = 0; s < L::kVStages; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    mbar_init(bar(L::kDrain), 1);
    st_volatile_shared(abort_addr, 0);
    fence_barrier_init();
  }
  if (warp == 8) {
    tmem_alloc(tmem_slot, L::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem_base = static_cast<uint32_t>(ld_volatile_shared(tmem_slot));

  if (warp < 8) {
    warpgroup_reg_acquire<kSoftmaxRegs>();
    // ======================= softmax / correction / epilogue =======================
    const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};
    const int t = warp >> 2;  // Q tile of this warpgroup
    const int wq = warp & 3;  // TMEM lane quarter of this warp
    const int row = wq * 32 + lane;
    const int qt = t == 0 ? qt0 : qt1;
    const int nt = t == 0 ? n0 : n1;
    const int grow = qt * kBlockM + row;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_bits + t * 128;
    const uint32_t tO = tmem_base + lane_bits + 256 + t * D;
    const float sl2 = p.scale_log2;

    float m = -INFINITY;  // running max of scale·log2e·s (log2 domain), possibly stale
    float l = 0.f;        // running sum of p = 2^(t - m) in fp32: gives the logsumexp
    float lq = 0.f;       // l plus, for each tile, the bf16 rounding error of the tile's
                          // largest p: normalises the output, so that a row dominated
                          // by one key is weighted exactly as the tensor core weights it
    bool moved_before = false;  // the reference max moved in this warp's previous tile
    bool ok = true;
    for (int j = 0; j < nt; ++j) {
      ok = wait_bounded(bar(L::kSFull + t), j & 1, ctl, kSiteSoftS | (t << 7) | j);
      ok = __all_sync(0xffffffffu, ok);
      if (!ok) break;
      tc_fence_after_sync();

      // S_j arrives in two 64-column halves: the second half's TMEM load is in
      // flight while the first half is processed.
      uint32_t sr[4][32];
      if (!dbg_warp(dbg_tmem(dbb, tS, 128, warp, kChkSTmem))) {  // S_j, then P_j over it
        ok = false;
        break;
      }
      tmem_ld_32x32b_x32(tS + 0, sr[0]);
      tmem_ld_32x32b_x32(tS + 32, sr[1]);
      tmem_ld_wait();
      reg_fence(sr[0]);
      reg_fence(sr[1]);
      tmem_ld_32x32b_x32(tS + 64, sr[2]);
      tmem_ld_32x32b_x32(tS + 96, sr[3]);

      // mask: key column > query row (causal diagonal tile) or column >= S (tail)
      const bool edge = (CAUSAL && j == qt) || ((j + 1) * kBlockN > p.S);
      int lim = p.S - 1 - j * kBlockN;  // last allowed column inside this tile
      if (CAUSAL) lim = min(lim, grow - j * kBlockN);
      auto mask_half = [&](int h) {
#pragma unroll
        for (int c = 2 * h; c < 2 * h + 2; ++c)
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (c * 32 + i > lim) sr[c][i] = __float_as_uint(-INFINITY);
      };
      // max of one 64-column half: 8 independent three-input chains, then a tree
      auto max_half = [&](int h) -> float {
        float cm[8];
#pragma unroll
        for (int g = 0; g < 8; ++g) {
          const uint32_t* e = &sr[2 * h + (g >> 2)][(g & 3) * 8];
          float a = max3f(__uint_as_float(e[0]), __uint_as_float(e[1]), __uint_as_float(e[2]));
          a = max3f(a, __uint_as_float(e[3]), __uint_as_float(e[4]));
          a = max3f(a, __uint_as_float(e[5]), __uint_as_float(e[6]));
          cm[g] = fmaxf(a, __uint_as_float(e[7]));
        }
        return fmaxf(max3f(cm[0], cm[1], cm[2]), max3f(max3f(cm[3], cm[4], cm[5]), cm[6], cm[7]));
      };
      // p = 2^(s·scale·log2e − m) for one half, two scores per packed FMA; P
      // (bf16) goes to TMEM over the consumed S columns; four packed
      // accumulators for the row sum.
      float2 rs2[4];
      auto exp_half = [&](int h, float neg_m) {
        const float2 sl2x2 = make_float2(sl2, sl2);
        const float2 nm2 = make_float2(neg_m, neg_m);
        uint32_t pk[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          const int c = (h * 64 + 2 * i) >> 5;
          const int e = (h * 64 + 2 * i) & 31;
          const float2 x = __ffma2_rn(
              make_float2(__uint_as_float(sr[c][e]), __uint_as_float(sr[c][e + 1])), sl2x2, nm2);
          const float p0 = ex2_approx(x.x);
          const float p1 = ex2_approx(x.y);
          rs2[i & 3] = __fadd2_rn(rs2[i & 3], make_float2(p0, p1));
          pk[i] = pack_x2<F16>(p0, p1);
        }
        tmem_st_32x32b_x32(tS + h * 32, pk);
      };
      auto clear_sums = [&]() {
#pragma unroll
        for (int a = 0; a < 4; ++a) rs2[a] = make_float2(0.f, 0.f);
      };

      // From the second tile on, unless the previous tile moved it, the
      // exponentials are computed against the current reference max right away
      // (it only moves when a row's max grows by more than the threshold); the
      // row max is checked alongside, and a tile that moves it is redone.
      const bool speculate = j > 0 && !moved_before;
      clear_sums();
      if (edge) mask_half(0);
      const float mx0 = max_half(0);
      if (speculate) exp_half(0, -m);
      tmem_ld_wait();
      reg_fence(sr[2]);
      reg_fence(sr[3]);
      if (edge) mask_half(1);
      const float mx = fmaxf(mx0, max_half(1));  // this row's largest raw score in the tile
      const float m_tile = mx * sl2;
      if (speculate) exp_half(1, -m);
      float alpha = 1.f;
      bool moved = false;
      if (j == 0) {
        m = m_tile;  // first tile: the reference is this tile's max
      } else if (m_tile > m + kRescaleThreshold<F16>) {
        alpha = ex2_approx(m - m_tile);
        m = m_tile;
        moved = true;
      }
      moved_before = __any_sync(0xffffffffu, moved);
      if (!speculate || moved_before) {
        const float neg_m = (m == -INFINITY) ? 0.f : -m;
        clear_sums();
        exp_half(0, neg_m);
        exp_half(1, neg_m);
      }
      const float2 rs_a = __fadd2_rn(__fadd2_rn(rs2[0], rs2[1]), __fadd2_rn(rs2[2], rs2[3]));
      const float rs = rs_a.x + rs_a.y;
      // the tile's largest p, computed exactly as in P, and its bf16 value
      const float pmax = ex2_approx(fmaf(mx, sl2, (m == -INFINITY) ? 0.f : -m));
      const float pmax_q = round_to_x<F16>(pmax);
      l = l * alpha + rs;
      lq = lq * alpha + (rs + (pmax_q - pmax));
      // correction: rescale this row of O when its reference max moved.  PV_{j-1}
      // has completed: S_j was committed after it.
      if (moved_before && dbg_warp(dbg_tmem(dbb, tO, D, warp, kChkOTmem))) {
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + c * 32, o);
          tmem_ld_wait();
          reg_fence(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
          tmem_st_32x32b_x32(tO + c * 32, o);
        }
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPFull + t));
    }

    // ---- epilogue: O / l → bf16 → smem (swizzled) → TMA store; lse
    if (nt > 0) {
      if (ok) {
        ok = wait_bounded(bar(L::kOFull + t), 0, ctl, kSiteSoftO | t);
        ok = __all_sync(0xffffffffu, ok);
      }
      if (ok) ok = dbg_warp(dbg_tmem(dbb, tO, D, warp, kChkOTmem));
      if (ok) {
        tc_fence_after_sync();
        const float inv_l = lq > 0.f ? 1.f / lq : 0.f;
        // Q_t's buffer is no longer read by any MMA: it stages this tile's output
        const uint32_t stage = sb + L::kQOff + t * L::kTileBytes;
#pragma unroll
        for (int c = 0; c < D / 32; ++c) {
          uint32_t o[32];
          tmem_ld_32x32b_x32(tO + c * 32, o);
          tmem_ld_wait();
          reg_fence(o);
#pragma unroll
          for (int q4 = 0; q4 < 4; ++q4) {
            const int unit = c * 4 + q4;  // 16-byte unit index along the row
            const int chunk = unit >> 3;
            const int u16 = unit & 7;
            const uint32_t addr = stage + chunk * L::kChunkBytes + row * 128 +
                                  ((u16 ^ (row & 7)) << 4);
            uint32_t w[4];
#pragma unroll
            for (int e = 0; e < 4; ++e)
              w[e] = pack_x2<F16>(__uint_as_float(o[q4 * 8 + 2 * e]) * inv_l,
                                 __uint_as_float(o[q4 * 8 + 2 * e + 1]) * inv_l);
            if (dbg_smem(dbb, addr, 16, 16, kChkStage)) st_shared_v4(addr, w[0], w[1], w[2], w[3]);
          }
        }
        fence_proxy_async_smem();
        __syncwarp();
        const int y0 = qt * kBlockM + wq * 32;  // stored if any of its 32 rows is inside
        if (lane == 0 && y0 < p.S) {
#pragma unroll
          for (int c = 0; c < L::kChunks; ++c) {
            const uint32_t src = stage + c * L::kChunkBytes + wq * 32 * 128;
            if (dbg_tma(dbb, src, 32 * 128, c * 64, y0, bh, true, kChkStore))
              tma_store_3d(&p.tm_o, src, c * 64, y0, bh);
          }
          tma_store_commit();
        }
        if (grow < p.S && dbg_row(dbb, bh, grow, 0, 0, kChkLse))
          p.lse[(int64_t)bh * p.S + grow] = (m + __log2f(l)) * kLn2;
        if (lane == 0) tma_store_wait_all();
      }
    }
    tc_fence_before_sync();
  } else {
    warpgroup_reg_release<kControlRegs>();
    if (warp == 9 && lane == 0) {
      // ======================= TMA producer =======================
      const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_o);
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if ((t == 0 ? n0 : n1) == 0) continue;
        mbar_arrive_expect_tx(bar(L::kQFull + t), L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          // a skipped copy leaves the stage's transaction count short: the
          // consumer's bounded wait then ends the kernel
          const uint32_t dst = sb + L::kQOff + t * L::kTileBytes + c * L::kChunkBytes;
          const int y = (t == 0 ? qt0 : qt1) * kBlockM;
          if (dbg_tma(dbb, dst, L::kChunkBytes, c * 64, y, bh, false, kChkLoadQ))
            tma_load_3d(dst, &p.tm_q, bar(L::kQFull + t), c * 64, y, bh, pol_q);
        }
      }
      int k_issued = 0, v_issued = 0;  // K / V tiles whose loads were issued
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        const int ks = j % L::kKStages;
        ok = wait_bounded(bar(L::kKEmpty + ks), ((j / L::kKStages) & 1) ^ 1, ctl, kSiteProducerK | j);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kKFull + ks), L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          const uint32_t dst = sb + L::kKOff + ks * L::kTileBytes + c * L::kChunkBytes;
          if (dbg_tma(dbb, dst, L::kChunkBytes, c * 64, j * kBlockN, bh, false, kChkLoadK))
            tma_load_3d(dst, &p.tm_k, bar(L::kKFull + ks), c * 64, j * kBlockN, bh, pol_kv);
        }
        k_issued = j + 1;
        const int vs = j % L::kVStages;
        ok = wait_bounded(bar(L::kVEmpty + vs), ((j / L::kVStages) & 1) ^ 1, ctl, kSiteProducerV | j);
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kVFull + vs), L::kTileBytes);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          const uint32_t dst = sb + L::kVOff + vs * L::kTileBytes + c * L::kChunkBytes;
          if (dbg_tma(dbb, dst, L::kChunkBytes, c * 64, j * kBlockN, bh, false, kChkLoadV))
            tma_load_3d(dst, &p.tm_v, bar(L::kVFull + vs), c * 64, j * kBlockN, bh, pol_kv);
        }
        v_issued = j + 1;
      }
      if (ok) {
        // Tail: wait until the tensor core has released every stage, so that
        // no commit-arrive on a ring barrier can land after this CTA is gone.
        for (int j = max(nkv - L::kKStages, 0); j < nkv && ok; ++j)
          ok = wait_bounded(bar(L::kKEmpty + j % L::kKStages), (j / L::kKStages) & 1, ctl,
                            kSiteProducerK | 0xff);
        for (int j = max(nkv - L::kVStages, 0); j < nkv && ok; ++j)
          ok = wait_bounded(bar(L::kVEmpty + j % L::kVStages), (j / L::kVStages) & 1, ctl,
                            kSiteProducerV | 0xff);
      }
      if (!ok) {
        // Abort: let every copy this thread started land before leaving.  The
        // last load into each stage completes its stage's latest full phase.
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if ((t == 0 ? n0 : n1) > 0) wait_drain(bar(L::kQFull + t), 0, kDrainLimitNs);
        for (int j = max(k_issued - L::kKStages, 0); j < k_issued; ++j)
          wait_drain(bar(L::kKFull + j % L::kKStages), (j / L::kKStages) & 1, kDrainLimitNs);
        for (int j = max(v_issued - L::kVStages, 0); j < v_issued; ++j)
          wait_drain(bar(L::kVFull + j % L::kVStages), (j / L::kVStages) & 1, kDrainLimitNs);
      }
    } else if (warp == 8) {
      // ======================= tcgen05 issuer =======================
      // The whole warp runs the schedule (so descriptors and loop state are
      // warp-uniform); one elected lane issues every tcgen05.mma and commit.
      const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};
      const bool leader = elect_one();
      constexpr uint32_t kIdescS = instr_desc_16bit(kBlockM, kBlockN, false, false, F16);
      constexpr uint32_t kIdescO = instr_desc_16bit(kBlockM, D, false, true, F16);
      // Descriptor bases; a K step or a stage only moves the start-address
      // field (16-byte units; no carry out of it: smem < 256 KB).
      const uint64_t dq = smem_desc_sw128(sb + L::kQOff, 16, 1024);
      const uint64_t dk = smem_desc_sw128(sb + L::kKOff, 16, 1024);
      const uint64_t dv = smem_desc_sw128(sb + L::kVOff, L::kChunkBytes, 1024);
      constexpr uint32_t kTileUnits = L::kTileBytes >> 4;

      // S_t = Q_t · K_stageᵀ: D/16 MMAs of K = 16 (32 bytes within a 128-byte
      // swizzle row; the next 64 columns are the next 16 KB block).
      auto issue_s = [&](int t, int ks) {
        if (!dbg_smem(dbb, sb + L::kQOff + t * L::kTileBytes, L::kTileBytes, 1024, kChkMmaQ) ||
            !dbg_smem(dbb, sb + L::kKOff + ks * L::kTileBytes, L::kTileBytes, 1024, kChkMmaK) ||
            !dbg_tmem_cols(dbb, tmem_base + t * 128, 128, kChkMmaTmem))
          return;  // S_t never completes: the softmax's bounded wait ends the kernel
        const uint64_t da = dq + t * kTileUnits;
        const uint64_t db = dk + ks * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = ((kk >> 2) * L::kChunkBytes + (kk & 3) * 32) >> 4;
          mma_ss(tmem_base + t * 128, da + off, db + off, kIdescS, kk > 0 ? 1u : 0u);
        }
      };
      // O_t += P_t · V_stage: 8 MMAs of K = 16 key rows (2 KB of V each).
      auto issue_pv = [&](int t, int vs, bool accumulate) {
        if (!dbg_smem(dbb, sb + L::kVOff + vs * L::kTileBytes, L::kTileBytes, 1024, kChkMmaV) ||
            !dbg_tmem_cols(dbb, tmem_base + 256 + t * D, D, kChkMmaTmem))
          return;
        const uint64_t db = dv + vs * kTileUnits;
#pragma unroll
        for (int kk = 0; kk < kBlockN / 16; ++kk)
          mma_ts(tmem_base + 256 + t * D, tmem_base + t * 128 + kk * 8, db + (kk * (2048 >> 4)),
                 kIdescO, (accumulate || kk > 0) ? 1u : 0u);
      };
      auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
        return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
      };

      bool ok = true;
      if (n0 > 0) ok = wait_warp(bar(L::kQFull + 0), 0, kSiteMmaQ);
      if (ok && n1 > 0) ok = wait_warp(bar(L::kQFull + 1), 0, kSiteMmaQ | 1);
      if (ok) ok = wait_warp(bar(L::kKFull + 0), 0, kSiteMmaK);
      if (ok) {
        tc_fence_after_sync();
        if (leader) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if ((t == 0 ? n0 : n1) == 0) continue;
            issue_s(t, 0);
            mma_commit(bar(L::kSFull + t));
          }
          mma_commit(bar(L::kKEmpty + 0));
        }
        __syncwarp();
        for (int j = 0; j < nkv && ok; ++j) {
          const int vs = j % L::kVStages;
          ok = wait_warp(bar(L::kVFull + vs), (j / L::kVStages) & 1, kSiteMmaV | j);
          if (!ok) break;
          const int kn = j + 1;
          const int ksn = kn % L::kKStages;
          bool k_next_ready = false;
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            const int ntt = t == 0 ? n0 : n1;
            if (!ok || j >= ntt) continue;
            ok = wait_warp(bar(L::kPFull + t), j & 1, kSiteMmaP | (t << 7) | j);
            if (!ok) break;
            tc_fence_after_sync();
            if (leader) issue_pv(t, vs, j > 0);
            if (kn < ntt) {
              if (!k_next_ready) {
                ok = wait_warp(bar(L::kKFull + ksn), (kn / L::kKStages) & 1, kSiteMmaK | kn);
                if (!ok) break;
                k_next_ready = true;
                tc_fence_after_sync();
              }
              if (leader) {
                issue_s(t, ksn);
                mma_commit(bar(L::kSFull + t));
              }
            } else if (leader) {
              mma_commit(bar(L::kOFull + t));
            }
            __syncwarp();
          }
          if (!ok) break;
          if (leader) {
            mma_commit(bar(L::kVEmpty + vs));
            if (k_next_ready) mma_commit(bar(L::kKEmpty + ksn));
          }
          __syncwarp();
        }
      }
      // Every MMA the leader issued has completed once `drain` arrives.
      if (leader) {
        mma_commit(bar(L::kDrain));
        wait_drain(bar(L::kDrain), 0, kDrainLimitNs);
      }
      __syncwarp();
    }
  }

  __syncthreads();
  if (warp == 8) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool F16>
cudaError_t launch_impl(const FwdParams& p, cudaStream_t stream) {
  using L = Layout<D>;
  auto kern = attn_fwd_kernel<D, CAUSAL, F16>;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  const long long grid = (long long)p.B * p.H * p.n_units;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
  cfg.blockDim = dim3(kThreads, 1, 1);
  cfg.dynamicSmemBytes = L::kAlloc;
  cfg.stream = stream;
  cfg.attrs = nullptr;
  cfg.numAttrs = 0;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

}  // namespace

size_t fwd_smem_bytes(int D) { return D == 64 ? Layout<64>::kAlloc : Layout<128>::kAlloc; }

template <bool F16>
static cudaError_t launch_typed(const FwdParams& p, int D, bool causal, cudaStream_t stream) {
  if (D == 64)
    return causal ? launch_impl<64, true, F16>(p, stream) : launch_impl<64, false, F16>(p, stream);
  return causal ? launch_impl<128, true, F16>(p, stream) : launch_impl<128, false, F16>(p, stream);
}

cudaError_t fwd_launch(const FwdParams& p, int D, bool causal, bool f16, cudaStream_t stream) {
  return f16 ? launch_typed<true>(p, D, causal, stream) : launch_typed<false>(p, D, causal, stream);
}

}  // namespace ea
