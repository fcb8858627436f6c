// attn_bwd256_sm103.cu — gradient of the attention forward for head
// dimensions above 128 (kernels 256 columns wide) on GB300 (sm_103a).
//
// The same computation as attn_bwd_sm103.cu: with P recomputed from the
// saved logsumexp, dP = dout·vᵀ and delta_i = rowsum(dout ⊙ out)_i,
//
//   dS = P ⊙ (dP − delta),   dq = scale·dS·k,   dk = scale·dSᵀ·q,   dv = Pᵀ·dout,
//
// the chain rule through the five steps of "Profiling in PyTorch (Part 3):
// Attention is all you profile", section "Naive attention"; no [S, S] matrix
// reaches HBM and tiles above the causal diagonal are skipped
// (FlashAttention-2 blog, "FlashAttention-2 Optimizations").  The
// FlashAttention issue "Pipelining GmemCopy on kHeadDim" speaks of kernels
// specialised on the head dimension; these are the 256-column ones.
//
// Why other layouts than at 128 columns: a 128-row fp32 accumulator of 256
// columns takes half of the 512 tensor-memory columns, so dK and dV together
// would fill it, and dQ beside Q and dO (the A operands of S and dP) would
// not fit either.  So:
//
//   attn_bwd_dq256_kernel   one CTA per (b·H + h, 128-row Q tile).  TMEM: S
//       [0, 64), dP [64, 128) of one 64-key step, Q [128, 256) (two 16-bit
//       values per column), dQ [256, 512).  dO stays in shared memory (64 KB),
//       so dP = dO·Vᵀ reads both operands from shared memory; K and V stream
//       in 64-key tiles (3 + 2 stages of 32 KB).
//   attn_bwd_dkdv_q64_kernel<256> one CTA per (b·H + h, 128-row K/V tile, half of the
//       head dimension): dK and dV of 128 columns each.  TMEM: Sᵀ [0, 64),
//       dPᵀ [64, 128) of one 64-query step, K [128, 256), dV [256, 384),
//       dK [384, 512).  V stays in shared memory (64 KB); Q and dO stream in
//       64-query tiles (2 stages of 64 KB).  Both halves form the same Sᵀ and
//       dPᵀ, a third more tensor work than one CTA per tile would do.
//
// In both kernels one S/dP step is in TMEM at a time; its 64 columns are
// split between the two elementwise warpgroups (warpgroup g takes columns
// [32g, 32g+32) and writes its 16-bit results over the first 16 of them,
// which is where the gradient products read them).  Roles as in the other
// backward kernels: warps 0-7 elementwise (one thread per TMEM lane), warp 8
// issues tcgen05.mma, warp 9 feeds the rings with TMA.  Every wait is bounded.
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "attn_bwd.h"
#include "bwd_common.cuh"
#include "ptx.cuh"
#include "umma.cuh"

namespace ea {
namespace {

constexpr float kLog2eW = 1.4426950408889634f;
constexpr uint64_t kDrainLimitNsW = 1000000000ull;
constexpr int kRowsW = 128;              // MMA M: rows of a Q tile (dq) or K/V tile (dk/dv)
constexpr int kStepW = 64;               // keys (dq) or queries (dk/dv) per step: MMA N of S, dP
constexpr int kBlk128 = kRowsW * 128;    // one 64-column block of a 128-row tile: 16 KB
constexpr int kBlk64 = kStepW * 128;     // one 64-column block of a 64-row tile: 8 KB
constexpr int kTile128 = 4 * kBlk128;    // 128 rows x 256 columns: 64 KB
constexpr int kTile64 = 4 * kBlk64;      // 64 rows x 256 columns: 32 KB

enum : int {
  kSiteW2Prod = 0x6100, kSiteW2MmaQ = 0x6200, kSiteW2MmaKV = 0x6300, kSiteW2MmaP = 0x6400,
  kSiteW2ElemS = 0x6500, kSiteW2ElemO = 0x6600,
  kSiteW3Prod = 0x6700, kSiteW3MmaKV = 0x6800, kSiteW3MmaQ = 0x6900, kSiteW3MmaP = 0x6a00,
  kSiteW3ElemS = 0x6b00, kSiteW3ElemO = 0x6c00
};
// debug-check sites (-DATTN_DEBUG)
enum : int { kChkWRowLoad = 0x5401, kChkWRowTmem, kChkWSTmem, kChkWStat, kChkWLoadA, kChkWLoadB,
             kChkWMmaA, kChkWMmaB };

// A offset (16-byte units) of K step kk (16 elements) in a K-major,
// 128-byte-swizzled tile whose 64-column blocks are `blk` bytes apart.
__device__ __forceinline__ uint32_t kstep_off(int kk, int blk) {
  return static_cast<uint32_t>(((kk >> 2) * blk + (kk & 3) * 32) >> 4);
}

// TMEM column of K step kk of a 16-bit operand that the two warpgroups wrote
// over the first 16 of their 32 columns: steps 0-1 from warpgroup 0, 2-3 from 1.
__device__ __forceinline__ uint32_t split_col(int kk) {
  return static_cast<uint32_t>(kk < 2 ? kk * 8 : 32 + (kk - 2) * 8);
}

// ============================================================== dq kernel

struct Dq256Layout {
  static constexpr int kKStages = 3, kVStages = 2;
  static constexpr int kDoOff = 0;
  static constexpr int kKOff = kDoOff + kTile128;
  static constexpr int kVOff = kKOff + kKStages * kTile64;
  static constexpr int kPartOff = kVOff + kVStages * kTile64;  // float [2][128] delta halves
  static constexpr int kBarOff = kPartOff + 2 * kRowsW * 4;
  static constexpr int kDoFull = 0, kQTmem = 1, kKFull = 2, kKEmpty = kKFull + kKStages,
                       kVFull = kKEmpty + kKStages, kVEmpty = kVFull + kVStages,
                       kSFull = kVEmpty + kVStages, kPFull = kSFull + 1, kOFull = kPFull + 1,
                       kDrain = kOFull + 1, kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  static_assert(kKStages * kTile64 >= 4 * kBlk128, "dQ staging must fit the K ring");
  static constexpr uint32_t kTmemCols = 512, kSCol = 0, kPCol = 64, kQCol = 128, kDqCol = 256;
};

template <bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dq256_kernel(const __grid_constant__ BwdParams p) {
  using L = Dq256Layout;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto bar = [sb](int idx) -> uint32_t { return sb + L::kBarOff + 8u * idx; };
  const uint32_t tmem_slot = sb + L::kMiscOff;
  const uint32_t abort_addr = sb + L::kMiscOff + 4;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const DbgBounds dbb{p.status, sb, smem_u32(smem_raw) + static_cast<uint32_t>(L::kAlloc), p.S,
                      p.d_cols, p.BH};
  int bh, i;
  schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh, &i);
  // 64-key steps: up to the Q tile's last row under the mask, and never one
  // that starts past the last key
  const int n_k64 = (p.S + kStepW - 1) / kStepW;
  const int nsteps = CAUSAL ? min(2 * (i + 1), n_k64) : n_k64;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kDoFull), 1);
    mbar_init(bar(L::kQTmem), 256);
    for (int s = 0; s < L::kKStages; ++s) {
      mbar_init(bar(L::kKFull + s), 1);
      mbar_init(bar(L::kKEmpty + s), 1);
    }
    for (int s = 0; s < L::kVStages; ++s) {
      mbar_init(bar(L::kVFull + s), 1);
      mbar_init(bar(L::kVEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kPFull), 256);
    mbar_init(bar(L::kOFull), 1);
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
  const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};

  if (warp < 8) {
    // ======================= elementwise: delta, dS, epilogue =======================
    const int g = warp >> 2;   // columns [32g, 32g+32) of every step; half g of every row
    const int wq = warp & 3;   // TMEM lane quarter
    const int row = wq * 32 + lane;
    const int grow = i * kRowsW + row;
    const bool valid = grow < p.S;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    // this row's half g of Q into TMEM (the A operand of every S product) and
    // that half of delta = rowsum(dout ⊙ out); columns past d_cols hold zero
    float part = 0.f;
    {
      uint32_t qw[64];
      const int64_t base = ((int64_t)bh * p.S + (valid ? grow : 0)) * p.d_cols + g * 128;
      const int lim = p.d_cols - g * 128;
      const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
      for (int u = 0; u < 16; ++u) {
        const bool in = valid && 8 * u < lim &&
                        dbg_row(dbb, bh, grow, g * 128 + 8 * u, 8, kChkWRowLoad);
        const uint4 qv = in ? __ldg(reinterpret_cast<const uint4*>(p.q + base) + u) : z;
        const uint4 dv = in ? __ldg(reinterpret_cast<const uint4*>(p.dout + base) + u) : z;
        const uint4 ov = in ? __ldg(reinterpret_cast<const uint4*>(p.out + base) + u) : z;
        part += dot8<F16>(ov, dv);
        qw[4 * u] = qv.x, qw[4 * u + 1] = qv.y, qw[4 * u + 2] = qv.z, qw[4 * u + 3] = qv.w;
      }
      const uint32_t tq = tmem_base + lane_bits + L::kQCol + 64 * g;
      if (dbg_warp(dbg_tmem(dbb, tq, 64, warp, kChkWRowTmem))) {
        tmem_st_32x32b_x32(tq, *reinterpret_cast<const uint32_t(*)[32]>(&qw[0]));
        tmem_st_32x32b_x32(tq + 32, *reinterpret_cast<const uint32_t(*)[32]>(&qw[32]));
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kQTmem));
    }
    st_shared_f32(sb + L::kPartOff + 4 * (g * kRowsW + row), part);
    named_bar_sync(1, 256);
    const float delta = ld_shared_f32(sb + L::kPartOff + 4 * row) +
                        ld_shared_f32(sb + L::kPartOff + 4 * (kRowsW + row));
    const bool row_ok = valid && dbg_row(dbb, bh, grow, 0, 0, kChkWRowLoad);
    if (g == 0 && row_ok) p.delta[(int64_t)bh * p.S + grow] = delta;
    const float lse2 = row_ok ? p.lse[(int64_t)bh * p.S + grow] * kLog2eW : 0.f;
    const float sl2 = p.scale_log2;
    const uint32_t tS = tmem_base + lane_bits + L::kSCol + 32 * g;
    const uint32_t tP = tmem_base + lane_bits + L::kPCol + 32 * g;

    bool ok = true;
    for (int s = 0; s < nsteps; ++s) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kSFull), s & 1, ctl,
                                                kSiteW2ElemS | (g << 7) | (s & 0x7f)));
      if (!ok) break;
      tc_fence_after_sync();
      if (!dbg_warp(dbg_tmem(dbb, tS, 32, warp, kChkWSTmem) && dbg_tmem(dbb, tP, 32, warp, kChkWSTmem))) {
        ok = false;
        break;
      }
      uint32_t sv[32], dpv[32];
      tmem_ld_32x32b_x32(tS, sv);
      tmem_ld_32x32b_x32(tP, dpv);
      tmem_ld_wait();
      reg_fence(sv);
      reg_fence(dpv);
      // allowed key columns of this warpgroup's 32: 0 .. lim (causal: key <= query; key < S)
      const int c0 = s * kStepW + 32 * g;
      int lim = p.S - 1 - c0;
      if (CAUSAL) lim = min(lim, grow - c0);
      if (!valid) lim = -1;
      const bool edge = lim < 31;
      uint32_t pk[16];
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2) {
        float p0 = ex2_approx(fmaf(__uint_as_float(sv[2 * e2]), sl2, -lse2));
        float p1 = ex2_approx(fmaf(__uint_as_float(sv[2 * e2 + 1]), sl2, -lse2));
        if (edge) {
          if (2 * e2 > lim) p0 = 0.f;
          if (2 * e2 + 1 > lim) p1 = 0.f;
        }
        pk[e2] = pack_x2<F16>(p0 * (__uint_as_float(dpv[2 * e2]) - delta),
                              p1 * (__uint_as_float(dpv[2 * e2 + 1]) - delta));
      }
      tmem_st_32x32b_x16(tS, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPFull));
    }

    // ---- epilogue: dQ · scale → 16-bit → swizzled staging (the K ring, idle
    // once every MMA has completed) → TMA store; warpgroup g stores blocks g, g+2
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kOFull), 0, ctl, kSiteW2ElemO));
    if (ok) {
      tc_fence_after_sync();
      for (int c = g; c < 4; c += 2)
        store_chunk<F16>(tmem_base + lane_bits + L::kDqCol + 64 * c, sb + L::kKOff + c * kBlk128, row,
                         p.scale, &p.tm_dq, c * 64, i * kRowsW, bh, wq, lane, dbb);
      if (lane == 0) {
        tma_store_commit();
        tma_store_wait_all();
      }
    }
    tc_fence_before_sync();
  } else if (warp == 9) {
    // ======================= TMA producer: dO once, K and V in 64-key tiles =======================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_k64);
      tma_prefetch_desc(&p.tm_v64);
      tma_prefetch_desc(&p.tm_dq);
      const uint64_t pol = l2_policy_evict_last();
      mbar_arrive_expect_tx(bar(L::kDoFull), kTile128);
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t dst = sb + L::kDoOff + c * kBlk128;
        if (dbg_tma(dbb, dst, kBlk128, c * 64, i * kRowsW, bh, false, kChkWLoadA))
          tma_load_3d(dst, &p.tm_do, bar(L::kDoFull), c * 64, i * kRowsW, bh, pol);
      }
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int s = 0; s < nsteps; ++s) {
        const int ks = s % L::kKStages;
        ok = wait_bounded(bar(L::kKEmpty + ks), ((s / L::kKStages) & 1) ^ 1, ctl,
                          kSiteW2Prod | (s & 0x7f));
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kKFull + ks), kTile64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t dst = sb + L::kKOff + ks * kTile64 + c * kBlk64;
          if (dbg_tma(dbb, dst, kBlk64, c * 64, s * kStepW, bh, false, kChkWLoadA))
            tma_load_3d(dst, &p.tm_k64, bar(L::kKFull + ks), c * 64, s * kStepW, bh, pol);
        }
        k_issued = s + 1;
        const int vs = s % L::kVStages;
        ok = wait_bounded(bar(L::kVEmpty + vs), ((s / L::kVStages) & 1) ^ 1, ctl,
                          kSiteW2Prod | 0x80 | (s & 0x7f));
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kVFull + vs), kTile64);
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          const uint32_t dst = sb + L::kVOff + vs * kTile64 + c * kBlk64;
          if (dbg_tma(dbb, dst, kBlk64, c * 64, s * kStepW, bh, false, kChkWLoadB))
            tma_load_3d(dst, &p.tm_v64, bar(L::kVFull + vs), c * 64, s * kStepW, bh, pol);
        }
        v_issued = s + 1;
      }
      if (ok) {
        for (int s = max(nsteps - L::kKStages, 0); s < nsteps && ok; ++s)
          ok = wait_bounded(bar(L::kKEmpty + s % L::kKStages), (s / L::kKStages) & 1, ctl,
                            kSiteW2Prod | 0x7f);
        for (int s = max(nsteps - L::kVStages, 0); s < nsteps && ok; ++s)
          ok = wait_bounded(bar(L::kVEmpty + s % L::kVStages), (s / L::kVStages) & 1, ctl,
                            kSiteW2Prod | 0xff);
      }
      if (!ok) {
        wait_drain(bar(L::kDoFull), 0, kDrainLimitNsW);
        for (int s = max(k_issued - L::kKStages, 0); s < k_issued; ++s)
          wait_drain(bar(L::kKFull + s % L::kKStages), (s / L::kKStages) & 1, kDrainLimitNsW);
        for (int s = max(v_issued - L::kVStages, 0); s < v_issued; ++s)
          wait_drain(bar(L::kVFull + s % L::kVStages), (s / L::kVStages) & 1, kDrainLimitNsW);
      }
    }
  } else {
    // ======================= tcgen05 issuer (warp 8) =======================
    // The whole warp runs the issue code; each product and commit is
    // predicated on the elected lane (mma_ts_p and co.), so that the warp
    // never branches around them: the waits stay warp-wide and converged,
    // which measured faster than a branch around each step's products.
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = instr_desc_16bit(kRowsW, kStepW, false, false, F16);
    constexpr uint32_t kIdescQ = instr_desc_16bit(kRowsW, 256, false, true, F16);
    constexpr uint32_t kTileUnits = kTile64 >> 4;
    const uint64_t d_do = smem_desc_sw128(sb + L::kDoOff, 16, 1024);
    const uint64_t d_k = smem_desc_sw128(sb + L::kKOff, 16, 1024);
    const uint64_t d_v = smem_desc_sw128(sb + L::kVOff, 16, 1024);
    const uint64_t d_kmn = smem_desc_sw128(sb + L::kKOff, kBlk64, 1024);
    auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
    };
    bool ok = wait_warp(bar(L::kDoFull), 0, kSiteW2MmaQ);
    if (ok) ok = wait_warp(bar(L::kQTmem), 0, kSiteW2MmaQ | 1);
    for (int s = 0; s < nsteps && ok; ++s) {
      const int ks = s % L::kKStages, vs = s % L::kVStages;
      ok = wait_warp(bar(L::kKFull + ks), (s / L::kKStages) & 1, kSiteW2MmaKV | (s & 0x7f));
      if (ok) ok = wait_warp(bar(L::kVFull + vs), (s / L::kVStages) & 1,
                             kSiteW2MmaKV | 0x80 | (s & 0x7f));
      if (!ok) break;
      tc_fence_after_sync();
      if (dbg_smem(dbb, sb + L::kKOff + ks * kTile64, kTile64, 1024, kChkWMmaA) &&
          dbg_smem(dbb, sb + L::kVOff + vs * kTile64, kTile64, 1024, kChkWMmaB)) {
        // S = Q · K_sᵀ (A = Q from TMEM) and dP = dO · V_sᵀ (both from shared memory)
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          mma_ts_p(leader, tmem_base + L::kSCol, tmem_base + L::kQCol + kk * 8,
                   d_k + ks * kTileUnits + kstep_off(kk, kBlk64), kIdescS, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < 16; ++kk)
          mma_ss_p(leader, tmem_base + L::kPCol, d_do + kstep_off(kk, kBlk128),
                   d_v + vs * kTileUnits + kstep_off(kk, kBlk64), kIdescS, kk > 0 ? 1u : 0u);
        mma_commit_p(leader, bar(L::kSFull));
        mma_commit_p(leader, bar(L::kVEmpty + vs));
      }
      ok = wait_warp(bar(L::kPFull), s & 1, kSiteW2MmaP | (s & 0x7f));
      if (!ok) break;
      tc_fence_after_sync();
      // dQ += dS · K_s (16 keys per step; K_s as an MN-major operand)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts_p(leader, tmem_base + L::kDqCol, tmem_base + L::kSCol + split_col(kk),
                 d_kmn + ks * kTileUnits + kk * (2048 >> 4), kIdescQ, (s > 0 || kk > 0) ? 1u : 0u);
      mma_commit_p(leader, bar(L::kKEmpty + ks));  // the next S overwrites dS: issued after these
    }
    if (leader) {
      if (ok) mma_commit(bar(L::kOFull));
      mma_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, kDrainLimitNsW);
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == 8) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

// ============================================================== dk/dv kernel
//
// 64-query steps, one Sᵀ/dPᵀ buffer.  D = 256 (the width the library runs
// on it): one CTA per half of the head dimension, V in shared memory (dPᵀ
// from two shared-memory operands).  The layout also holds D = 64 and 128
// (one CTA per K/V tile, K and V both in TMEM, at D = 128 filling the 512
// columns exactly); there the kernel of attn_bwd_sm103.cu, whose two
// warpgroups' elementwise work overlaps the tensor core's, is faster.

template <int D>
struct KvQ64Layout {
  static constexpr bool kSplit = D > 128;            // a CTA per half of the head dimension
  static constexpr int kCols = kSplit ? 128 : D;     // gradient columns per CTA
  static constexpr int kChunks = D / 64;             // 64-column blocks of a row
  static constexpr int kTileQ = kChunks * kBlk64;    // 64 queries x D
  static constexpr int kStages = kSplit ? 2 : (D == 128 ? 4 : 6);  // Q / dO ring
  static constexpr int kStatBytes = kStepW * 8;      // (lse·log2e, delta) per query
  static constexpr int kVOff = 0;                    // V tile (split only)
  static constexpr int kQOff = kVOff + (kSplit ? kChunks * kBlk128 : 0);
  static constexpr int kDoOff = kQOff + kStages * kTileQ;
  static constexpr int kStatOff = kDoOff + kStages * kTileQ;
  static constexpr int kBarOff = kStatOff + kStages * kStatBytes;
  static constexpr int kVFull = 0, kKTmem = 1, kFull = 2, kEmpty = kFull + kStages,
                       kSFull = kEmpty + kStages, kPFull = kSFull + 1, kOFull = kPFull + 1,
                       kDrain = kOFull + 1, kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  // the epilogue stages dV (warpgroup 0) and dK (warpgroup 1), 128 rows x kCols each
  static_assert(2 * kStages * kTileQ >= 2 * (kCols / 64) * kBlk128, "staging must fit the ring");
  static constexpr uint32_t kTmemCols = 512, kSCol = 0, kPCol = 64, kKCol = 128,
                            kVCol = 128 + D / 2, kDvCol = 256, kDkCol = 256 + kCols;
  static_assert(kSplit || kVCol + D / 2 <= kDvCol, "TMEM budget exceeded");
  static_assert(kDkCol + kCols <= kTmemCols, "TMEM budget exceeded");
};

// One thread's `n` 32-bit words (n = 16, 32 or 64) into TMEM at `taddr`.
template <int N>
__device__ __forceinline__ void tmem_st_row(uint32_t taddr, const uint32_t (&w)[N]) {
  if constexpr (N == 16) {
    tmem_st_32x32b_x16(taddr, w);
  } else {
#pragma unroll
    for (int c = 0; c < N / 32; ++c)
      tmem_st_32x32b_x32(taddr + 32 * c, *reinterpret_cast<const uint32_t(*)[32]>(&w[32 * c]));
  }
}

template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dkdv_q64_kernel(const __grid_constant__ BwdParams p) {
  using L = KvQ64Layout<D>;
  constexpr bool kSplit = L::kSplit;
  constexpr int kCols = L::kCols;
  constexpr int kTileQ = L::kTileQ;
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
  // with the head dimension split, the two halves of one K/V tile are neighbouring CTAs
  const int half = kSplit ? static_cast<int>(blockIdx.x & 1u) : 0;
  int bh, level;
  schedule_unit(p.sched, static_cast<int>(kSplit ? blockIdx.x >> 1 : blockIdx.x), &bh, &level);
  const int j = p.n_t - 1 - level;  // K/V tile
  const int n_q64 = (p.S + kStepW - 1) / kStepW;
  const int u0 = CAUSAL ? 2 * j : 0;  // first 64-query tile that sees this K/V tile
  const int n_sub = n_q64 - u0;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kVFull), 1);
    mbar_init(bar(L::kKTmem), 256);
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
    }
    mbar_init(bar(L::kSFull), 1);
    mbar_init(bar(L::kPFull), 256);
    mbar_init(bar(L::kOFull), 1);
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
  const WaitCtl ctl{abort_addr, p.status, p.timeout_ns};

  if (warp < 8) {
    // ======================= elementwise: K (and V) to TMEM, Pᵀ, dSᵀ, epilogue =======================
    const int g = warp >> 2;            // query columns [32g, 32g+32) of every step
    const int wq = warp & 3;
    const int r = wq * 32 + lane;       // key row within the tile (TMEM lane)
    const int gk = j * kRowsW + r;      // key row in the sequence
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const float sl2 = p.scale_log2;
    {
      // this row's half g of K (and of V unless it is in shared memory) into
      // TMEM; rows past the end and columns past d_cols hold zero
      constexpr int kU = D / 16;  // 16-byte groups in half a row
      uint32_t kw[4 * kU], vw[4 * kU];
      const bool in_row = gk < p.S;
      const int64_t base = ((int64_t)bh * p.S + (in_row ? gk : 0)) * p.d_cols + g * (D / 2);
      const int lim = p.d_cols - g * (D / 2);
#pragma unroll
      for (int u = 0; u < kU; ++u) {
        const bool in = in_row && 8 * u < lim &&
                        dbg_row(dbb, bh, gk, g * (D / 2) + 8 * u, 8, kChkWRowLoad);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
        const uint4 kv = in ? __ldg(reinterpret_cast<const uint4*>(p.k + base) + u) : z;
        kw[4 * u] = kv.x, kw[4 * u + 1] = kv.y, kw[4 * u + 2] = kv.z, kw[4 * u + 3] = kv.w;
        if constexpr (!kSplit) {
          const uint4 vv = in ? __ldg(reinterpret_cast<const uint4*>(p.v + base) + u) : z;
          vw[4 * u] = vv.x, vw[4 * u + 1] = vv.y, vw[4 * u + 2] = vv.z, vw[4 * u + 3] = vv.w;
        }
      }
      const uint32_t tk = tmem_base + lane_bits + L::kKCol + (D / 4) * g;
      const uint32_t tv = tmem_base + lane_bits + L::kVCol + (D / 4) * g;
      if (dbg_warp(dbg_tmem(dbb, tk, D / 4, warp, kChkWRowTmem) &&
                   (kSplit || dbg_tmem(dbb, tv, D / 4, warp, kChkWRowTmem)))) {
        tmem_st_row<4 * kU>(tk, kw);
        if constexpr (!kSplit) tmem_st_row<4 * kU>(tv, vw);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kKTmem));
    }
    const uint32_t tS = tmem_base + lane_bits + L::kSCol + 32 * g;
    const uint32_t tP = tmem_base + lane_bits + L::kPCol + 32 * g;
    bool ok = true;
    for (int t = 0; t < n_sub; ++t) {
      const int u = u0 + t;
      const int st = t % L::kStages;
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kSFull), t & 1, ctl,
                                                kSiteW3ElemS | (g << 7) | (t & 0x7f)));
      if (!ok) break;
      tc_fence_after_sync();
      if (!dbg_warp(dbg_tmem(dbb, tS, 32, warp, kChkWSTmem) && dbg_tmem(dbb, tP, 32, warp, kChkWSTmem))) {
        ok = false;
        break;
      }
      uint32_t sv[32], dpv[32];
      tmem_ld_32x32b_x32(tS, sv);
      tmem_ld_32x32b_x32(tP, dpv);
      tmem_ld_wait();
      reg_fence(sv);
      reg_fence(dpv);
      // allowed query columns of this warpgroup's 32: lo .. hi (causal: query >= key; query < S)
      const int c0 = u * kStepW + 32 * g;
      const int hi = p.S - 1 - c0;
      int lo = CAUSAL ? gk - c0 : 0;
      if (gk >= p.S) lo = 32;  // key row past the end: nothing
      const bool edge = lo > 0 || hi < 31;
      // (lse·log2e, delta) of these 32 query columns, two columns per load
      const float4* stat = reinterpret_cast<const float4*>(smem_gen + L::kStatOff +
                                                           st * L::kStatBytes + 8 * 32 * g);
      uint32_t ppk[16], dpk[16];
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2) {
        const int c = 2 * e2;
        const float4 sd = stat[e2];  // lse2[c], delta[c], lse2[c+1], delta[c+1]
        float p0 = ex2_approx(fmaf(__uint_as_float(sv[c]), sl2, -sd.x));
        float p1 = ex2_approx(fmaf(__uint_as_float(sv[c + 1]), sl2, -sd.z));
        if (edge) {
          if (c < lo || c > hi) p0 = 0.f;
          if (c + 1 < lo || c + 1 > hi) p1 = 0.f;
        }
        ppk[e2] = pack_x2<F16>(p0, p1);
        dpk[e2] = pack_x2<F16>(p0 * (__uint_as_float(dpv[c]) - sd.y),
                               p1 * (__uint_as_float(dpv[c + 1]) - sd.w));
      }
      tmem_st_32x32b_x16(tS, ppk);
      tmem_st_32x32b_x16(tP, dpk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPFull));
    }

    // ---- epilogue: warpgroup 0 stores dV, 1 stores dK · scale (this CTA's
    // columns), staged in the Q / dO ring (idle once every MMA has completed)
    if (ok) ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kOFull), 0, ctl, kSiteW3ElemO));
    if (ok) {
      tc_fence_after_sync();
      const uint32_t tAcc = tmem_base + lane_bits + (g == 0 ? L::kDvCol : L::kDkCol);
      const uint32_t stage = sb + L::kQOff + g * (kCols / 64) * kBlk128;
      const CUtensorMap* map = g == 0 ? &p.tm_dv : &p.tm_dk;
      const float mul = g == 0 ? 1.f : p.scale;
#pragma unroll
      for (int cc = 0; cc < kCols / 64; ++cc)
        store_chunk<F16>(tAcc + 64 * cc, stage + cc * kBlk128, r, mul, map, kCols * half + 64 * cc,
                         j * kRowsW, bh, wq, lane, dbb);
      if (lane == 0) {
        tma_store_commit();
        tma_store_wait_all();
      }
    }
    tc_fence_before_sync();
  } else if (warp == 9) {
    // ======================= producer: (V once;) Q, dO, stats per 64 queries =======================
    const uint64_t pol = l2_policy_evict_last();
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q64);
      tma_prefetch_desc(&p.tm_do64);
      tma_prefetch_desc(&p.tm_dk);
      tma_prefetch_desc(&p.tm_dv);
      if constexpr (kSplit) {
        tma_prefetch_desc(&p.tm_v);
        mbar_arrive_expect_tx(bar(L::kVFull), L::kChunks * kBlk128);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          const uint32_t dst = sb + L::kVOff + c * kBlk128;
          if (dbg_tma(dbb, dst, kBlk128, c * 64, j * kRowsW, bh, false, kChkWLoadB))
            tma_load_3d(dst, &p.tm_v, bar(L::kVFull), c * 64, j * kRowsW, bh, pol);
        }
      }
    }
    const int64_t row0 = (int64_t)bh * p.S;
    int issued = 0;
    bool ok = true;
    for (int t = 0; t < n_sub; ++t) {
      const int u = u0 + t;
      const int st = t % L::kStages;
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kEmpty + st), ((t / L::kStages) & 1) ^ 1,
                                                ctl, kSiteW3Prod | (t & 0xff)));
      if (!ok) break;
      // per-query statistics of these 64 queries; queries past the end read as 0
      const uint32_t stat = sb + L::kStatOff + st * L::kStatBytes;
#pragma unroll
      for (int h2 = 0; h2 < 2; ++h2) {
        const int c = lane + 32 * h2;
        const int q = u * kStepW + c;
        const bool in = q < p.S && dbg_row(dbb, bh, q, 0, 0, kChkWStat);
        st_shared_f32x2(stat + 8 * c, in ? p.lse[row0 + q] * kLog2eW : 0.f,
                        in ? p.delta[row0 + q] : 0.f);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(L::kFull + st), 2 * kTileQ);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          // a skipped copy leaves the stage's transaction count short: the
          // consumer's bounded wait then ends the kernel
          const uint32_t qd = sb + L::kQOff + st * kTileQ + c * kBlk64;
          const uint32_t dd = sb + L::kDoOff + st * kTileQ + c * kBlk64;
          if (dbg_tma(dbb, qd, kBlk64, c * 64, u * kStepW, bh, false, kChkWLoadA))
            tma_load_3d(qd, &p.tm_q64, bar(L::kFull + st), c * 64, u * kStepW, bh, pol);
          if (dbg_tma(dbb, dd, kBlk64, c * 64, u * kStepW, bh, false, kChkWLoadB))
            tma_load_3d(dd, &p.tm_do64, bar(L::kFull + st), c * 64, u * kStepW, bh, pol);
        }
      }
      issued = t + 1;
      __syncwarp();
    }
    if (lane == 0) {
      if (ok) {
        for (int t = max(n_sub - L::kStages, 0); t < n_sub && ok; ++t)
          ok = wait_bounded(bar(L::kEmpty + t % L::kStages), (t / L::kStages) & 1, ctl,
                            kSiteW3Prod | 0xff);
      }
      if (!ok) {
        if (kSplit) wait_drain(bar(L::kVFull), 0, kDrainLimitNsW);
        for (int t = max(issued - L::kStages, 0); t < issued; ++t)
          wait_drain(bar(L::kFull + t % L::kStages), (t / L::kStages) & 1, kDrainLimitNsW);
      }
    }
    __syncwarp();
  } else {
    // ======================= tcgen05 issuer (warp 8) =======================
    // The whole warp runs the issue code; each product and commit is
    // predicated on the elected lane (mma_ts_p and co.), so that the warp
    // never branches around them: the waits stay warp-wide and converged,
    // which measured faster than a branch around each step's products.
    const bool leader = elect_one();
    constexpr uint32_t kIdescS = instr_desc_16bit(kRowsW, kStepW, false, false, F16);
    constexpr uint32_t kIdescG = instr_desc_16bit(kRowsW, kCols, false, true, F16);
    constexpr uint32_t kTileUnits = kTileQ >> 4;
    const uint64_t d_v = smem_desc_sw128(sb + L::kVOff, 16, 1024);
    const uint64_t d_q = smem_desc_sw128(sb + L::kQOff, 16, 1024);
    const uint64_t d_do = smem_desc_sw128(sb + L::kDoOff, 16, 1024);
    // this CTA's gradient columns: blocks kCols/64 · half onwards
    const uint64_t d_q_mn =
        smem_desc_sw128(sb + L::kQOff + (kCols / 64) * half * kBlk64, kBlk64, 1024);
    const uint64_t d_do_mn =
        smem_desc_sw128(sb + L::kDoOff + (kCols / 64) * half * kBlk64, kBlk64, 1024);
    auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
    };
    bool ok = wait_warp(bar(L::kKTmem), 0, kSiteW3MmaKV);
    if (ok && kSplit) ok = wait_warp(bar(L::kVFull), 0, kSiteW3MmaKV | 1);
    for (int t = 0; t < n_sub && ok; ++t) {
      const int st = t % L::kStages;
      ok = wait_warp(bar(L::kFull + st), (t / L::kStages) & 1, kSiteW3MmaQ | (t & 0xff));
      if (!ok) break;
      tc_fence_after_sync();
      if (dbg_smem(dbb, sb + L::kQOff + st * kTileQ, kTileQ, 1024, kChkWMmaA) &&
          dbg_smem(dbb, sb + L::kDoOff + st * kTileQ, kTileQ, 1024, kChkWMmaB)) {
        // Sᵀ = K · Q_tᵀ (A = K from TMEM) and dPᵀ = V · dO_tᵀ (A = V from
        // TMEM, or from shared memory when the head dimension is split)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk)
          mma_ts_p(leader, tmem_base + L::kSCol, tmem_base + L::kKCol + kk * 8,
                   d_q + st * kTileUnits + kstep_off(kk, kBlk64), kIdescS, kk > 0 ? 1u : 0u);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint64_t db = d_do + st * kTileUnits + kstep_off(kk, kBlk64);
          if constexpr (kSplit)
            mma_ss_p(leader, tmem_base + L::kPCol, d_v + kstep_off(kk, kBlk128), db, kIdescS,
                     kk > 0 ? 1u : 0u);
          else
            mma_ts_p(leader, tmem_base + L::kPCol, tmem_base + L::kVCol + kk * 8, db, kIdescS,
                     kk > 0 ? 1u : 0u);
        }
        mma_commit_p(leader, bar(L::kSFull));
      }
      ok = wait_warp(bar(L::kPFull), t & 1, kSiteW3MmaP | (t & 0xff));
      if (!ok) break;
      tc_fence_after_sync();
      // dV += Pᵀ · dO_t and dK += dSᵀ · Q_t over this CTA's columns (16 queries per step)
#pragma unroll
      for (int kk = 0; kk < 4; ++kk) {
        const uint32_t acc = (t > 0 || kk > 0) ? 1u : 0u;
        const uint32_t bo = st * kTileUnits + kk * (2048 >> 4);
        mma_ts_p(leader, tmem_base + L::kDvCol, tmem_base + L::kSCol + split_col(kk), d_do_mn + bo,
                 kIdescG, acc);
        mma_ts_p(leader, tmem_base + L::kDkCol, tmem_base + L::kPCol + split_col(kk), d_q_mn + bo,
                 kIdescG, acc);
      }
      mma_commit_p(leader, bar(L::kEmpty + st));  // the next Sᵀ, dPᵀ overwrite Pᵀ, dSᵀ: issued after these
    }
    if (leader) {
      if (ok) mma_commit(bar(L::kOFull));
      mma_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, kDrainLimitNsW);
    }
    __syncwarp();
  }

  __syncthreads();
  if (warp == 8) {
    tc_fence_after_sync();
    tmem_dealloc(tmem_base, L::kTmemCols);
  }
}

template <int D, bool CAUSAL, bool F16>
cudaError_t dkdv_q64_launch(const BwdParams& p, cudaStream_t stream) {
  using L = KvQ64Layout<D>;
  auto kkv = attn_bwd_dkdv_q64_kernel<D, CAUSAL, F16>;
  cudaError_t e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, L::kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  // with the head dimension split, two CTAs (column halves) per K/V tile
  cfg.gridDim = dim3(static_cast<unsigned>((L::kSplit ? 2ll : 1ll) * p.BH * p.n_t), 1, 1);
  cfg.blockDim = dim3(kBwdThreads, 1, 1);
  cfg.stream = stream;
  cfg.dynamicSmemBytes = L::kAlloc;
  return cudaLaunchKernelEx(&cfg, kkv, p);
}

template <bool CAUSAL, bool F16>
cudaError_t launch_256(const BwdParams& p, cudaStream_t stream) {
  auto kdq = attn_bwd_dq256_kernel<CAUSAL, F16>;
  cudaError_t e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       Dq256Layout::kAlloc);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.BH * p.n_t), 1, 1);
  cfg.blockDim = dim3(kBwdThreads, 1, 1);
  cfg.stream = stream;
  cfg.dynamicSmemBytes = Dq256Layout::kAlloc;
  e = cudaLaunchKernelEx(&cfg, kdq, p);
  if (e != cudaSuccess) return e;
  return dkdv_q64_launch<256, CAUSAL, F16>(p, stream);
}

}  // namespace

cudaError_t bwd256_launch(const BwdParams& p, bool causal, bool f16, cudaStream_t stream) {
  if (f16) return causal ? launch_256<true, true>(p, stream) : launch_256<false, true>(p, stream);
  return causal ? launch_256<true, false>(p, stream) : launch_256<false, false>(p, stream);
}

}  // namespace ea
