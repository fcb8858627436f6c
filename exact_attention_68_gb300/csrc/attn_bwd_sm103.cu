// attn_bwd_sm103.cu — gradient of the fused attention forward on GB300 (sm_103a).
//
// The forward is out = softmax(scale·q·kᵀ + causal mask)·v, as defined step by
// step in "Profiling in PyTorch (Part 3): Attention is all you profile",
// section "Naive attention"; the same page's passage on in-place operations
// notes that the backward reuses what the forward saved.  Here the forward
// saved out and the row logsumexp lse, so the weights are recomputed tile by
// tile, P = exp(scale·q·kᵀ − lse), and the chain rule through the five steps
// gives, with dP = dout·vᵀ and delta_i = rowsum(dout ⊙ out)_i:
//
//   dS = P ⊙ (dP − delta),   dq = scale·dS·k,   dk = scale·dSᵀ·q,   dv = Pᵀ·dout.
//
// As in the forward (FlashAttention-2 blog, "FlashAttention-2 Optimizations")
// no [S, S] matrix reaches HBM and tiles above the causal diagonal are skipped.
// Two kernels, each owning the rows it writes, so no gradient is accumulated
// with atomics and the result does not depend on scheduling:
//
//   attn_bwd_dq_kernel    one CTA per (b·H + h, 128-row Q tile), walking the
//                         K/V tiles: S = Q·Kᵀ, dP = dO·Vᵀ, dS, dQ += dS·K.
//                         It also computes delta for its rows and stores it.
//   attn_bwd_dkdv_kernel  one CTA per (b·H + h, 128-row K/V tile), walking the
//                         Q tiles: Sᵀ = K·Qᵀ, dPᵀ = V·dOᵀ, Pᵀ and dSᵀ,
//                         dV += Pᵀ·dO, dK += dSᵀ·Q.
//
// GB300 mapping (per CTA): warps 0-7 do the elementwise work, one thread per
// TMEM lane (a tile row), in two warpgroups with a TMEM buffer each; warp 8
// issues tcgen05.mma (the whole warp runs the issue code, each product and
// commit predicated on its elected lane); warp 9 feeds the shared-memory
// rings with TMA.  While one warpgroup does its buffer's elementwise work,
// the tensor core runs the other buffer's products.
//
//   dq kernel     Q and dO rows are put into TMEM once (the A operand of every
//                 S and dP product); K/V tiles stream through shared memory.
//                 Each K/V tile is two 64-key halves, warpgroup g always
//                 taking half g; the MMA order per tile j is G(j,0),
//                 SP(j+1,0), G(j,1), SP(j+1,1) (SP: a half's S and dP
//                 products, G: its dQ product).  TMEM: half h's S [128h,
//                 128h+64) and dP [128h+64, 128h+128); dQ [256, 256+D);
//                 Q [384, 384+D/2), dO [384+D/2, 384+D).
//   dk/dv kernel  K and V rows are put into TMEM once (the A operand of every
//                 Sᵀ and dPᵀ product); Q and dO tiles stream through shared
//                 memory.  Each Q tile is four 32-query sub-steps, warpgroup b
//                 taking the sub-steps t ≡ b (mod 2); the MMA order is G(t),
//                 then SP(t+2) into the buffer G(t) has just read.  TMEM:
//                 buffer b's Sᵀ [64b, 64b+32) and dPᵀ [64b+32, 64b+64);
//                 K [128, 128+D/2), V [128+D/2, 128+D); dV [256, 256+D),
//                 dK [256+D, 256+2D).
//
// A warpgroup stores its 16-bit results (two per 32-bit column) over the
// first columns of the S and dP blocks it has just read: they are the A
// operand of the gradient products.  The elementwise arithmetic runs on
// packed f32x2 pairs (in the dk/dv kernel at D = 128 only), with the same
// roundings as the scalar form.
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

constexpr float kLog2e = 1.4426950408889634f;
constexpr uint64_t kDrainLimitNs = 1000000000ull;  // bound on waits while tearing down
constexpr int kTileRows = 128;
constexpr int kChunkBytes = kTileRows * 128;  // one 64-column, 128-row swizzled block

// Wait-site tags recorded in status[1] by the first wait that runs out.
enum : int {
  kSiteDqProducer = 0x1100, kSiteDqMmaQ = 0x1200, kSiteDqMmaKV = 0x1300, kSiteDqMmaP = 0x1400,
  kSiteDqElemS = 0x1500, kSiteDqElemO = 0x1600,
  kSiteKvProducer = 0x2100, kSiteKvMmaKV = 0x2200, kSiteKvMmaQ = 0x2300, kSiteKvMmaP = 0x2400,
  kSiteKvElemS = 0x2500, kSiteKvElemO = 0x2600
};
// debug-check sites (-DATTN_DEBUG); kChkAccTmem, kChkStage and kChkStore are in bwd_common.cuh
enum : int { kChkRowLoad = 0x5204, kChkRowTmem, kChkSTmem, kChkStat, kChkLoadA, kChkLoadB,
             kChkMmaA, kChkMmaB };

// ============================================================== dq kernel

template <int D>
struct DqLayout {
  static constexpr int kTile = kTileRows * D * 2;
  static constexpr int kChunks = D / 64;
  static constexpr int kKStages = (D == 128) ? 4 : 6;  // K ring depth
  static constexpr int kVStages = (D == 128) ? 3 : 5;  // V ring depth (V is released earlier)
  static constexpr int kKOff = 0;
  static constexpr int kVOff = kKOff + kKStages * kTile;
  static constexpr int kPartOff = kVOff + kVStages * kTile;  // float [2][128] delta halves
  static constexpr int kBarOff = kPartOff + 2 * kTileRows * 4;
  static constexpr int kQFull = 0;                   // Q and dO in TMEM (256 arrivals)
  static constexpr int kKFull = 1;                   // [kKStages]
  static constexpr int kKEmpty = kKFull + kKStages;  // [kKStages]
  static constexpr int kVFull = kKEmpty + kKStages;  // [kVStages]
  static constexpr int kVEmpty = kVFull + kVStages;  // [kVStages]
  static constexpr int kSFull = kVEmpty + kVStages;  // [2] S_h and dP_h computed
  static constexpr int kPFull = kSFull + 2;          // [2] dS_h stored (128 arrivals)
  static constexpr int kOFull = kPFull + 2;          // dQ final
  static constexpr int kDrain = kOFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;  // tmem base, abort flag
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  static constexpr uint32_t kTmemCols = 512;
  // TMEM columns of Q and dO as the A operand of S and dP (two 16-bit values
  // per column): after the two S/dP buffers and dQ
  static constexpr uint32_t kQCol = 384;
  static constexpr uint32_t kDoCol = 384 + D / 2;
  static_assert(kDoCol + D / 2 <= kTmemCols, "TMEM budget exceeded");
};

template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using L = DqLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  auto bar = [sb](int idx) -> uint32_t { return sb + L::kBarOff + 8u * idx; };
  const uint32_t tmem_slot = sb + L::kMiscOff;
  const uint32_t abort_addr = sb + L::kMiscOff + 4;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // Q tile i of slice bh, in the order of the grid schedule (schedule.h):
  // heavy tiles by L2-sized groups of heads, then the light ones over all heads
  const DbgBounds dbb{p.status, sb, smem_u32(smem_raw) + static_cast<uint32_t>(L::kAlloc), p.S,
                      p.d_cols, p.BH};
  int bh, i;
  schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh, &i);
  const int nkv = CAUSAL ? i + 1 : p.n_t;

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kQFull), 256);
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
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      mbar_init(bar(L::kSFull + h), 1);
      mbar_init(bar(L::kPFull + h), 128);
    }
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
    const int g = warp >> 2;   // half of every K/V tile this warpgroup takes
    const int wq = warp & 3;   // TMEM lane quarter
    const int row = wq * 32 + lane;
    const int grow = i * kTileRows + row;
    const bool valid = grow < p.S;
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_bits + 128 * g;
    const uint32_t tP = tS + 64;
    const uint32_t tQ = tmem_base + lane_bits + 256;

    // Each warpgroup takes half of its row's D columns: it puts that half of
    // the Q and dO rows into TMEM (the A operand of S and dP for the whole
    // loop, so shared memory only feeds the K/V side) and sums that half of
    // delta = rowsum(dout ⊙ out).
    float part = 0.f;
    {
      constexpr int kU = D / 16;  // 16-byte groups in half a row
      uint32_t qw[4 * kU], dw[4 * kU];
      if (valid) {
        // columns past d_cols hold zero
        const int64_t base = ((int64_t)bh * p.S + grow) * p.d_cols + g * (D / 2);
        const int lim = p.d_cols - g * (D / 2);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const bool in = 8 * u < lim && dbg_row(dbb, bh, grow, g * (D / 2) + 8 * u, 8, kChkRowLoad);
          const uint4 qv = in ? __ldg(reinterpret_cast<const uint4*>(p.q + base) + u) : z;
          const uint4 dv = in ? __ldg(reinterpret_cast<const uint4*>(p.dout + base) + u) : z;
          const uint4 ov = in ? __ldg(reinterpret_cast<const uint4*>(p.out + base) + u) : z;
          part += dot8<F16>(ov, dv);
          qw[4 * u] = qv.x, qw[4 * u + 1] = qv.y, qw[4 * u + 2] = qv.z, qw[4 * u + 3] = qv.w;
          dw[4 * u] = dv.x, dw[4 * u + 1] = dv.y, dw[4 * u + 2] = dv.z, dw[4 * u + 3] = dv.w;
        }
      } else {
#pragma unroll
        for (int w = 0; w < 4 * kU; ++w) qw[w] = dw[w] = 0u;
      }
      if (dbg_warp(dbg_tmem(dbb, tmem_base + lane_bits + L::kQCol + g * (D / 4), D / 4, warp,
                            kChkRowTmem) &&
                   dbg_tmem(dbb, tmem_base + lane_bits + L::kDoCol + g * (D / 4), D / 4, warp,
                            kChkRowTmem))) {
        tmem_st_words(tmem_base + lane_bits + L::kQCol + g * (D / 4), qw);
        tmem_st_words(tmem_base + lane_bits + L::kDoCol + g * (D / 4), dw);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kQFull));
    }
    st_shared_f32(sb + L::kPartOff + 4 * (g * kTileRows + row), part);
    named_bar_sync(1, 256);
    const float delta = ld_shared_f32(sb + L::kPartOff + 4 * row) +
                        ld_shared_f32(sb + L::kPartOff + 4 * (kTileRows + row));
    const bool row_ok = valid && dbg_row(dbb, bh, grow, 0, 0, kChkRowLoad);
    if (g == 0 && row_ok) p.delta[(int64_t)bh * p.S + grow] = delta;
    const float lse2 = row_ok ? p.lse[(int64_t)bh * p.S + grow] * kLog2e : 0.f;
    const float sl2 = p.scale_log2;

    bool ok = true;
    for (int j = 0; j < nkv; ++j) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kSFull + g), j & 1, ctl,
                                                kSiteDqElemS | (g << 7) | (j & 0x7f)));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t s[2][32], dp[2][32];
      if (!dbg_warp(dbg_tmem(dbb, tS, 64, warp, kChkSTmem) && dbg_tmem(dbb, tP, 64, warp, kChkSTmem))) {
        ok = false;
        break;
      }
      tmem_ld_32x32b_x32(tS, s[0]);
      tmem_ld_32x32b_x32(tS + 32, s[1]);
      tmem_ld_32x32b_x32(tP, dp[0]);
      tmem_ld_32x32b_x32(tP + 32, dp[1]);
      tmem_ld_wait();
      reg_fence(s[0]);
      reg_fence(s[1]);
      reg_fence(dp[0]);
      reg_fence(dp[1]);
      // allowed key columns of this half: 0 .. lim (causal: key <= query; key < S)
      const int c0 = j * kTileRows + 64 * g;
      int lim = p.S - 1 - c0;
      if (CAUSAL) lim = min(lim, grow - c0);
      if (!valid) lim = -1;
      const bool edge = lim < 63;
      uint32_t pk[32];
#pragma unroll
      for (int e2 = 0; e2 < 32; ++e2) {
        const int h = e2 >> 4;
        const int e = (2 * e2) & 31;
        // key pairs in packed f32x2 arithmetic (the same roundings as the
        // scalar form, half the FP32 instructions)
        const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[h][e]), __uint_as_float(s[h][e + 1])),
                                    make_float2(sl2, sl2), make_float2(-lse2, -lse2));
        float p0 = ex2_approx(x.x);
        float p1 = ex2_approx(x.y);
        if (edge) {
          if (2 * e2 > lim) p0 = 0.f;
          if (2 * e2 + 1 > lim) p1 = 0.f;
        }
        const float2 dd = __fadd2_rn(make_float2(__uint_as_float(dp[h][e]), __uint_as_float(dp[h][e + 1])),
                                     make_float2(-delta, -delta));
        const float2 ds = __fmul2_rn(make_float2(p0, p1), dd);
        pk[e2] = pack_x2<F16>(ds.x, ds.y);
      }
      tmem_st_32x32b_x32(tS, pk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPFull + g));
    }

    // ---- epilogue: dQ · scale → 16-bit → swizzled staging (K stage 0, idle
    // once every MMA has completed) → TMA store
    if (ok) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kOFull), 0, ctl, kSiteDqElemO));
    }
    if (ok) {
      tc_fence_after_sync();
      for (int c = g; c < L::kChunks; c += 2)
        store_chunk<F16>(tQ + c * 64, sb + L::kKOff + c * kChunkBytes, row, p.scale, &p.tm_dq, c * 64,
                         i * kTileRows, bh, wq, lane, dbb);
      if (lane == 0) {
        tma_store_commit();
        tma_store_wait_all();
      }
    }
    tc_fence_before_sync();
  } else if (warp == 9) {
    // ======================= TMA producer =======================
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_k);
      tma_prefetch_desc(&p.tm_v);
      tma_prefetch_desc(&p.tm_dq);
      const uint64_t pol_kv = l2_policy_evict_last();
      int k_issued = 0, v_issued = 0;
      bool ok = true;
      for (int j = 0; j < nkv; ++j) {
        const int ks = j % L::kKStages;
        ok = wait_bounded(bar(L::kKEmpty + ks), ((j / L::kKStages) & 1) ^ 1, ctl,
                          kSiteDqProducer | (j & 0x7f));
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kKFull + ks), L::kTile);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          // a skipped copy leaves the stage's transaction count short: the
          // consumer's bounded wait then ends the kernel
          const uint32_t dst = sb + L::kKOff + ks * L::kTile + c * kChunkBytes;
          if (dbg_tma(dbb, dst, kChunkBytes, c * 64, j * kTileRows, bh, false, kChkLoadA))
            tma_load_3d(dst, &p.tm_k, bar(L::kKFull + ks), c * 64, j * kTileRows, bh, pol_kv);
        }
        k_issued = j + 1;
        const int vs = j % L::kVStages;
        ok = wait_bounded(bar(L::kVEmpty + vs), ((j / L::kVStages) & 1) ^ 1, ctl,
                          kSiteDqProducer | 0x80 | (j & 0x7f));
        if (!ok) break;
        mbar_arrive_expect_tx(bar(L::kVFull + vs), L::kTile);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          const uint32_t dst = sb + L::kVOff + vs * L::kTile + c * kChunkBytes;
          if (dbg_tma(dbb, dst, kChunkBytes, c * 64, j * kTileRows, bh, false, kChkLoadB))
            tma_load_3d(dst, &p.tm_v, bar(L::kVFull + vs), c * 64, j * kTileRows, bh, pol_kv);
        }
        v_issued = j + 1;
      }
      if (ok) {
        // every stage released by the tensor core before this CTA may exit
        for (int j = max(nkv - L::kKStages, 0); j < nkv && ok; ++j)
          ok = wait_bounded(bar(L::kKEmpty + j % L::kKStages), (j / L::kKStages) & 1, ctl,
                            kSiteDqProducer | 0x7f);
        for (int j = max(nkv - L::kVStages, 0); j < nkv && ok; ++j)
          ok = wait_bounded(bar(L::kVEmpty + j % L::kVStages), (j / L::kVStages) & 1, ctl,
                            kSiteDqProducer | 0xff);
      }
      if (!ok) {
        for (int j = max(k_issued - L::kKStages, 0); j < k_issued; ++j)
          wait_drain(bar(L::kKFull + j % L::kKStages), (j / L::kKStages) & 1, kDrainLimitNs);
        for (int j = max(v_issued - L::kVStages, 0); j < v_issued; ++j)
          wait_drain(bar(L::kVFull + j % L::kVStages), (j / L::kVStages) & 1, kDrainLimitNs);
      }
    }
  } else {
    // ======================= tcgen05 issuer (warp 8) =======================
    // The whole warp runs the issue code; each product and commit is
    // predicated on the elected lane (mma_ts_p and co.), so that the warp
    // never branches around them: the waits stay warp-wide and converged,
    // which measured faster than a branch around each step's products.
    const bool leader = elect_one();
    constexpr uint32_t kIdescSP = instr_desc_16bit(kTileRows, 64, false, false, F16);  // 64 keys
    constexpr uint32_t kIdescQ = instr_desc_16bit(kTileRows, D, false, true, F16);
    constexpr uint32_t kTileUnits = L::kTile >> 4;
    constexpr uint32_t kHalfUnits = (64 * 128) >> 4;  // 64 rows of a 128-byte-row block
    const uint64_t dk = smem_desc_sw128(sb + L::kKOff, 16, 1024);
    const uint64_t dv = smem_desc_sw128(sb + L::kVOff, 16, 1024);
    const uint64_t dk_mn = smem_desc_sw128(sb + L::kKOff, kChunkBytes, 1024);
    auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
    };
    // SP(j, h): S_h = Q · K_j[64h, 64h+64)ᵀ and dP_h = dO · V_j[64h, 64h+64)ᵀ,
    // A (Q, dO) from TMEM, 8 columns per K step of 16
    auto issue_sp = [&](int ks, int vs, int h) {
      if (!dbg_smem(dbb, sb + L::kKOff + ks * L::kTile, L::kTile, 1024, kChkMmaA) ||
          !dbg_smem(dbb, sb + L::kVOff + vs * L::kTile, L::kTile, 1024, kChkMmaB))
        return;  // S_h never completes: the elementwise warps' bounded wait ends the kernel
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ts_p(leader, tmem_base + 128 * h, tmem_base + L::kQCol + kk * 8,
               dk + ks * kTileUnits + h * kHalfUnits + off, kIdescSP, kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ts_p(leader, tmem_base + 128 * h + 64, tmem_base + L::kDoCol + kk * 8,
               dv + vs * kTileUnits + h * kHalfUnits + off, kIdescSP, kk > 0 ? 1u : 0u);
      }
      mma_commit_p(leader, bar(L::kSFull + h));
    };
    // G(j, h): dQ += dS_h · K_j[64h, 64h+64) (16 key rows per step)
    auto issue_g = [&](int ks, int h, bool first) {
#pragma unroll
      for (int kk = 0; kk < 4; ++kk)
        mma_ts_p(leader, tmem_base + 256, tmem_base + 128 * h + kk * 8,
               dk_mn + ks * kTileUnits + (4 * h + kk) * (2048 >> 4), kIdescQ,
               (first && kk == 0) ? 0u : 1u);
    };
    auto wait_kv = [&](int j) {
      bool r = wait_warp(bar(L::kKFull + j % L::kKStages), (j / L::kKStages) & 1,
                         kSiteDqMmaKV | (j & 0x7f));
      if (r) r = wait_warp(bar(L::kVFull + j % L::kVStages), (j / L::kVStages) & 1,
                           kSiteDqMmaKV | 0x80 | (j & 0x7f));
      return r;
    };

    bool ok = wait_warp(bar(L::kQFull), 0, kSiteDqMmaQ);
    if (ok) ok = wait_kv(0);
    if (ok) {
      tc_fence_after_sync();
      issue_sp(0, 0, 0);
      issue_sp(0, 0, 1);
      mma_commit_p(leader, bar(L::kVEmpty + 0));
    }
    for (int j = 0; j < nkv && ok; ++j) {
      const int ks = j % L::kKStages;
      const bool more = j + 1 < nkv;
      const int ksn = (j + 1) % L::kKStages;
      const int vsn = (j + 1) % L::kVStages;
      // At D = 64 the next K/V tile is waited for before dS_0 (it has normally
      // landed long before), which keeps that wait off the path from dS_0 to
      // S/dP of the next tile; at D = 128 that order measured slower.
      constexpr bool kKvFirst = D == 64;
      if (kKvFirst && more) ok = wait_kv(j + 1);
      if (ok) ok = wait_warp(bar(L::kPFull + 0), j & 1, kSiteDqMmaP | (j & 0x7f));
      if (!ok) break;
      tc_fence_after_sync();
      issue_g(ks, 0, j == 0);
      if (more) {
        if (!kKvFirst) {
          ok = wait_kv(j + 1);
          if (!ok) break;
          tc_fence_after_sync();
        }
        issue_sp(ksn, vsn, 0);
      }
      ok = wait_warp(bar(L::kPFull + 1), j & 1, kSiteDqMmaP | 0x80 | (j & 0x7f));
      if (!ok) break;
      tc_fence_after_sync();
      issue_g(ks, 1, false);
      mma_commit_p(leader, bar(L::kKEmpty + ks));  // K_j: last read by G(j, 1)
      if (more) {
        issue_sp(ksn, vsn, 1);
        mma_commit_p(leader, bar(L::kVEmpty + vsn));  // V_{j+1}: last read by SP(j+1, 1)
      }
    }
    if (leader) {
      if (ok) mma_commit(bar(L::kOFull));
      mma_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, kDrainLimitNs);
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
// K_j and V_j are the A operand of every Sᵀ / dPᵀ product of the CTA, so they
// are put into TMEM once; shared memory then only feeds Q and dO.  Each Q tile
// is taken as four 32-column quarters ("sub-steps" t = 4·it + q) in two TMEM
// buffers; warpgroup b takes the sub-steps with t ≡ b (mod 2), i.e. quarters
// b and b+2 of every tile.  TMEM columns (D = 128):
//   buffer b: Sᵀ [64b, 64b+32), dPᵀ [64b+32, 64b+64)
//   K [128, 128+D/2), V [128+D/2, 128+D)   (two 16-bit values per column)
//   dV [256, 256+D), dK [256+D, 256+2D)

template <int D>
struct KvLayout {
  static constexpr int kTile = kTileRows * D * 2;
  static constexpr int kChunks = D / 64;
  static constexpr int kStages = (D == 128) ? 3 : 4;  // Q/dO ring depth
  static constexpr int kStatBytes = 2 * kTileRows * 4;  // (−lse·log2e, −delta) per query row
  static constexpr int kQOff = 0;
  static constexpr int kDoOff = kQOff + kStages * kTile;
  static constexpr int kStatOff = kDoOff + kStages * kTile;
  static constexpr int kBarOff = kStatOff + kStages * kStatBytes;
  static constexpr int kKVTmem = 0;                 // K_j, V_j in TMEM (256 arrivals)
  static constexpr int kFull = 1;                   // [kStages] Q_i, dO_i, stats landed
  static constexpr int kEmpty = kFull + kStages;    // [kStages]
  static constexpr int kSFull = kEmpty + kStages;   // [2] Sᵀ and dPᵀ of buffer b computed
  static constexpr int kPFull = kSFull + 2;         // [2] Pᵀ and dSᵀ of buffer b stored (128)
  static constexpr int kOFull = kPFull + 2;         // dK, dV final
  static constexpr int kDrain = kOFull + 1;
  static constexpr int kNumBars = kDrain + 1;
  static constexpr int kMiscOff = kBarOff + kNumBars * 8;
  static constexpr int kAlloc = kMiscOff + 16 + 1024;
  static_assert(kAlloc <= 232448, "shared memory budget exceeded");
  static constexpr uint32_t kTmemCols = 512;
  static constexpr uint32_t kKCol = 128;
  static constexpr uint32_t kVCol = 128 + D / 2;
  static constexpr uint32_t kDvCol = 256;
  static constexpr uint32_t kDkCol = 256 + D;
  static_assert(kDkCol + D <= kTmemCols, "TMEM budget exceeded");
  static_assert(2 * kTile <= kStages * kTile, "dK/dV staging must fit the Q ring");
};

template <int D, bool CAUSAL, bool F16>
__global__ void __launch_bounds__(kBwdThreads, 1) attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using L = KvLayout<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t sb = (smem_u32(smem_raw) + 1023u) & ~1023u;
  const uint8_t* smem_gen = smem_raw + (sb - smem_u32(smem_raw));  // same window, generic
  auto bar = [sb](int idx) -> uint32_t { return sb + L::kBarOff + 8u * idx; };
  const uint32_t tmem_slot = sb + L::kMiscOff;
  const uint32_t abort_addr = sb + L::kMiscOff + 4;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;

  // K/V tile j of slice bh; under the mask tile j meets Q tiles j .. n_t-1,
  // so its schedule level is n_t - 1 - j (grid order as in the dq kernel)
  const DbgBounds dbb{p.status, sb, smem_u32(smem_raw) + static_cast<uint32_t>(L::kAlloc), p.S,
                      p.d_cols, p.BH};
  int bh, level;
  schedule_unit(p.sched, static_cast<int>(blockIdx.x), &bh, &level);
  const int j = p.n_t - 1 - level;
  const int i0 = CAUSAL ? j : 0;
  const int nq = p.n_t - i0;
  const int n_sub = 4 * nq;  // quarter sub-steps

  if (threadIdx.x == 0) {
    mbar_init(bar(L::kKVTmem), 256);
#pragma unroll
    for (int s = 0; s < L::kStages; ++s) {
      mbar_init(bar(L::kFull + s), 1);
      mbar_init(bar(L::kEmpty + s), 1);
    }
#pragma unroll
    for (int b = 0; b < 2; ++b) {
      mbar_init(bar(L::kSFull + b), 1);
      mbar_init(bar(L::kPFull + b), 128);
    }
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
    // ======================= elementwise: K/V to TMEM, Pᵀ, dSᵀ, epilogue =======================
    const int g = warp >> 2;            // TMEM buffer (quarters g and g+2) of this warpgroup
    const int wq = warp & 3;
    const int r = wq * 32 + lane;       // key row within the tile (TMEM lane)
    const int gk = j * kTileRows + r;   // key row in the sequence
    const uint32_t lane_bits = static_cast<uint32_t>(wq * 32) << 16;
    const uint32_t tS = tmem_base + lane_bits + 64 * g;
    const uint32_t tP = tS + 32;
    const float sl2 = p.scale_log2;
    {
      // this row's K and V, half of D per warpgroup, into TMEM (rows past the end: 0)
      constexpr int kU = D / 16;  // 16-byte groups in half a row
      uint32_t kw[4 * kU], vw[4 * kU];
      if (gk < p.S) {
        // columns past d_cols hold zero
        const int64_t base = ((int64_t)bh * p.S + gk) * p.d_cols + g * (D / 2);
        const int lim = p.d_cols - g * (D / 2);
        const uint4 z = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
        for (int u = 0; u < kU; ++u) {
          const bool in = 8 * u < lim && dbg_row(dbb, bh, gk, g * (D / 2) + 8 * u, 8, kChkRowLoad);
          const uint4 kv = in ? __ldg(reinterpret_cast<const uint4*>(p.k + base) + u) : z;
          const uint4 vv = in ? __ldg(reinterpret_cast<const uint4*>(p.v + base) + u) : z;
          kw[4 * u] = kv.x, kw[4 * u + 1] = kv.y, kw[4 * u + 2] = kv.z, kw[4 * u + 3] = kv.w;
          vw[4 * u] = vv.x, vw[4 * u + 1] = vv.y, vw[4 * u + 2] = vv.z, vw[4 * u + 3] = vv.w;
        }
      } else {
#pragma unroll
        for (int w = 0; w < 4 * kU; ++w) kw[w] = vw[w] = 0u;
      }
      if (dbg_warp(dbg_tmem(dbb, tmem_base + lane_bits + L::kKCol + g * (D / 4), D / 4, warp,
                            kChkRowTmem) &&
                   dbg_tmem(dbb, tmem_base + lane_bits + L::kVCol + g * (D / 4), D / 4, warp,
                            kChkRowTmem))) {
        tmem_st_words(tmem_base + lane_bits + L::kKCol + g * (D / 4), kw);
        tmem_st_words(tmem_base + lane_bits + L::kVCol + g * (D / 4), vw);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kKVTmem));
    }
    bool ok = true;
    for (int t = g; t < n_sub; t += 2) {
      const int it = t >> 2;
      const int q = t & 3;
      const int i = i0 + it;
      const int st = it % L::kStages;
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kSFull + g), (t >> 1) & 1, ctl,
                                                kSiteKvElemS | (g << 7) | (t & 0x7f)));
      if (!ok) break;
      tc_fence_after_sync();
      uint32_t s[32], dp[32];
      if (!dbg_warp(dbg_tmem(dbb, tS, 32, warp, kChkSTmem) && dbg_tmem(dbb, tP, 32, warp, kChkSTmem))) {
        ok = false;
        break;
      }
      tmem_ld_32x32b_x32(tS, s);
      tmem_ld_32x32b_x32(tP, dp);
      tmem_ld_wait();
      reg_fence(s);
      reg_fence(dp);
      // allowed query columns of this quarter: lo .. hi (causal: query >= key; query < S)
      const int c0 = i * kTileRows + 32 * q;
      const int hi = p.S - 1 - c0;
      int lo = CAUSAL ? gk - c0 : 0;
      if (gk >= p.S) lo = 32;  // key row past the end: nothing
      const bool edge = lo > 0 || hi < 31;
      // (−lse·log2e, −delta) of this quarter's 32 query columns, two columns per load
      const float4* stat = reinterpret_cast<const float4*>(
          smem_gen + L::kStatOff + st * L::kStatBytes + 8 * 32 * q);
      uint32_t ppk[16], dpk[16];
#pragma unroll
      for (int e2 = 0; e2 < 16; ++e2) {
        const int c = 2 * e2;
        const float4 sd = stat[e2];  // -lse2[c], -delta[c], -lse2[c+1], -delta[c+1]
        // column pairs in packed f32x2 arithmetic at D = 128 (the same roundings
        // as the scalar form; measured faster there, slower at D = 64)
        constexpr bool kPacked = D == 128;
        float p0, p1;
        if constexpr (kPacked) {
          const float2 x = __ffma2_rn(make_float2(__uint_as_float(s[c]), __uint_as_float(s[c + 1])),
                                      make_float2(sl2, sl2), make_float2(sd.x, sd.z));
          p0 = ex2_approx(x.x);
          p1 = ex2_approx(x.y);
        } else {
          p0 = ex2_approx(fmaf(__uint_as_float(s[c]), sl2, sd.x));
          p1 = ex2_approx(fmaf(__uint_as_float(s[c + 1]), sl2, sd.z));
        }
        if (edge) {
          if (c < lo || c > hi) p0 = 0.f;
          if (c + 1 < lo || c + 1 > hi) p1 = 0.f;
        }
        float ds0, ds1;
        if constexpr (kPacked) {
          const float2 dd = __fadd2_rn(make_float2(__uint_as_float(dp[c]), __uint_as_float(dp[c + 1])),
                                       make_float2(sd.y, sd.w));
          const float2 ds = __fmul2_rn(make_float2(p0, p1), dd);
          ds0 = ds.x, ds1 = ds.y;
        } else {
          ds0 = p0 * (__uint_as_float(dp[c]) + sd.y);
          ds1 = p1 * (__uint_as_float(dp[c + 1]) + sd.w);
        }
        ppk[e2] = pack_x2<F16>(p0, p1);
        dpk[e2] = pack_x2<F16>(ds0, ds1);
      }
      tmem_st_32x32b_x16(tS, ppk);
      tmem_st_32x32b_x16(tP, dpk);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(bar(L::kPFull + g));
    }

    // ---- epilogue: warpgroup 0 stores dV, 1 stores dK · scale, staged in the
    // (idle once every MMA has completed) Q ring
    if (ok) {
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kOFull), 0, ctl, kSiteKvElemO));
    }
    if (ok) {
      tc_fence_after_sync();
      const uint32_t tAcc = tmem_base + lane_bits + (g == 0 ? L::kDvCol : L::kDkCol);
      const uint32_t stage = sb + L::kQOff + g * L::kTile;
      const CUtensorMap* map = g == 0 ? &p.tm_dv : &p.tm_dk;
      const float mul = g == 0 ? 1.f : p.scale;
#pragma unroll
      for (int c = 0; c < L::kChunks; ++c)
        store_chunk<F16>(tAcc + c * 64, stage + c * kChunkBytes, r, mul, map, c * 64, j * kTileRows,
                         bh, wq, lane, dbb);
      if (lane == 0) {
        tma_store_commit();
        tma_store_wait_all();
      }
    }
    tc_fence_before_sync();
  } else if (warp == 9) {
    // ======================= producer: Q_i, dO_i, stats per Q tile =======================
    const uint64_t pol_q = l2_policy_evict_last();
    if (lane == 0) {
      tma_prefetch_desc(&p.tm_q);
      tma_prefetch_desc(&p.tm_do);
      tma_prefetch_desc(&p.tm_dk);
      tma_prefetch_desc(&p.tm_dv);
    }
    const int64_t row0 = (int64_t)bh * p.S;
    int issued = 0;
    bool ok = true;
    for (int it = 0; it < nq; ++it) {
      const int i = i0 + it;
      const int st = it % L::kStages;
      ok = __all_sync(0xffffffffu, wait_bounded(bar(L::kEmpty + st), ((it / L::kStages) & 1) ^ 1,
                                                ctl, kSiteKvProducer | (it & 0xff)));
      if (!ok) break;
      // per-query-row statistics of Q tile i; rows past the end read as 0
      const uint32_t stat = sb + L::kStatOff + st * L::kStatBytes;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int c = lane + 32 * t;
        const int q = i * kTileRows + c;
        const bool in = q < p.S && dbg_row(dbb, bh, q, 0, 0, kChkStat);
        st_shared_f32x2(stat + 8 * c, in ? -(p.lse[row0 + q] * kLog2e) : 0.f,
                        in ? -p.delta[row0 + q] : 0.f);
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(bar(L::kFull + st), 2 * L::kTile);
#pragma unroll
        for (int c = 0; c < L::kChunks; ++c) {
          // a skipped copy leaves the stage's transaction count short: the
          // consumer's bounded wait then ends the kernel
          const uint32_t dq_dst = sb + L::kQOff + st * L::kTile + c * kChunkBytes;
          const uint32_t do_dst = sb + L::kDoOff + st * L::kTile + c * kChunkBytes;
          if (dbg_tma(dbb, dq_dst, kChunkBytes, c * 64, i * kTileRows, bh, false, kChkLoadA))
            tma_load_3d(dq_dst, &p.tm_q, bar(L::kFull + st), c * 64, i * kTileRows, bh, pol_q);
          if (dbg_tma(dbb, do_dst, kChunkBytes, c * 64, i * kTileRows, bh, false, kChkLoadB))
            tma_load_3d(do_dst, &p.tm_do, bar(L::kFull + st), c * 64, i * kTileRows, bh, pol_q);
        }
      }
      issued = it + 1;
      __syncwarp();
    }
    if (lane == 0) {
      if (ok) {
        for (int it = max(nq - L::kStages, 0); it < nq && ok; ++it)
          ok = wait_bounded(bar(L::kEmpty + it % L::kStages), (it / L::kStages) & 1, ctl,
                            kSiteKvProducer | 0xff);
      }
      if (!ok) {
        for (int it = max(issued - L::kStages, 0); it < issued; ++it)
          wait_drain(bar(L::kFull + it % L::kStages), (it / L::kStages) & 1, kDrainLimitNs);
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
    constexpr uint32_t kIdescSP = instr_desc_16bit(kTileRows, 32, false, false, F16);  // 32 queries
    constexpr uint32_t kIdescG = instr_desc_16bit(kTileRows, D, false, true, F16);
    constexpr uint32_t kTileUnits = L::kTile >> 4;
    constexpr uint32_t kQuarterUnits = (32 * 128) >> 4;  // 32 rows of a 128-byte-row block
    const uint64_t dq = smem_desc_sw128(sb + L::kQOff, 16, 1024);
    const uint64_t ddo = smem_desc_sw128(sb + L::kDoOff, 16, 1024);
    const uint64_t dq_mn = smem_desc_sw128(sb + L::kQOff, kChunkBytes, 1024);
    const uint64_t ddo_mn = smem_desc_sw128(sb + L::kDoOff, kChunkBytes, 1024);
    auto wait_warp = [&](uint32_t b, uint32_t parity, int site) {
      return __all_sync(0xffffffffu, wait_bounded(b, parity, ctl, site));
    };
    // SP(t): Sᵀ = K_j · Q_i[32q, 32q+32)ᵀ and dPᵀ = V_j · dO_i[32q, 32q+32)ᵀ into
    // buffer t & 1; A (K, V) from TMEM, 8 columns per K step of 16
    auto issue_sp = [&](int t) {
      const int b = t & 1, q = t & 3, st = (t >> 2) % L::kStages;
      if (!dbg_smem(dbb, sb + L::kQOff + st * L::kTile, L::kTile, 1024, kChkMmaA) ||
          !dbg_smem(dbb, sb + L::kDoOff + st * L::kTile, L::kTile, 1024, kChkMmaB))
        return;  // S never completes: the elementwise warps' bounded wait ends the kernel
      const uint32_t bq = st * kTileUnits + q * kQuarterUnits;
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ts_p(leader, tmem_base + 64 * b, tmem_base + L::kKCol + kk * 8, dq + bq + off, kIdescSP,
               kk > 0 ? 1u : 0u);
      }
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = ((kk >> 2) * kChunkBytes + (kk & 3) * 32) >> 4;
        mma_ts_p(leader, tmem_base + 64 * b + 32, tmem_base + L::kVCol + kk * 8, ddo + bq + off, kIdescSP,
               kk > 0 ? 1u : 0u);
      }
      mma_commit_p(leader, bar(L::kSFull + b));
    };
    // G(t): dV += Pᵀ · dO_i[32q, 32q+32), dK += dSᵀ · Q_i[32q, 32q+32)
    auto issue_g = [&](int t) {
      const int b = t & 1, q = t & 3, st = (t >> 2) % L::kStages;
#pragma unroll
      for (int kk = 0; kk < 2; ++kk) {
        const uint32_t a = 64 * b + kk * 8;
        const uint32_t bo = st * kTileUnits + (2 * q + kk) * (2048 >> 4);
        const uint32_t acc = (t == 0 && kk == 0) ? 0u : 1u;
        mma_ts_p(leader, tmem_base + L::kDvCol, tmem_base + a, ddo_mn + bo, kIdescG, acc);
        mma_ts_p(leader, tmem_base + L::kDkCol, tmem_base + a + 32, dq_mn + bo, kIdescG, acc);
      }
    };

    bool ok = wait_warp(bar(L::kKVTmem), 0, kSiteKvMmaKV);
    if (ok) ok = wait_warp(bar(L::kFull + 0), 0, kSiteKvMmaQ);
    if (ok) {
      tc_fence_after_sync();
      issue_sp(0);
      issue_sp(1);
    }
    for (int t = 0; t < n_sub && ok; ++t) {
      const int b = t & 1;
      const int t2 = t + 2;
      if ((t2 & 3) == 0 && t2 < n_sub) {
        // the sub-step issued after this one opens Q tile t2 / 4: its stage
        // must have landed (normally long before this P, so waited for first)
        const int it2 = t2 >> 2;
        ok = wait_warp(bar(L::kFull + it2 % L::kStages), (it2 / L::kStages) & 1,
                       kSiteKvMmaQ | (it2 & 0xff));
      }
      if (ok) ok = wait_warp(bar(L::kPFull + b), (t >> 1) & 1, kSiteKvMmaP | (b << 7) | (t & 0x7f));
      if (!ok) break;
      tc_fence_after_sync();
      issue_g(t);
      if ((t & 3) == 3) mma_commit_p(leader, bar(L::kEmpty + (t >> 2) % L::kStages));  // Q_i, dO_i done
      if (t2 < n_sub) issue_sp(t2);
    }
    if (leader) {
      if (ok) mma_commit(bar(L::kOFull));
      mma_commit(bar(L::kDrain));
      wait_drain(bar(L::kDrain), 0, kDrainLimitNs);
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
cudaError_t launch_impl(const BwdParams& p, cudaStream_t stream) {
  auto kdq = attn_bwd_dq_kernel<D, CAUSAL, F16>;
  auto kkv = attn_bwd_dkdv_kernel<D, CAUSAL, F16>;
  cudaError_t e = cudaFuncSetAttribute(kdq, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       DqLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  e = cudaFuncSetAttribute(kkv, cudaFuncAttributeMaxDynamicSharedMemorySize, KvLayout<D>::kAlloc);
  if (e != cudaSuccess) return e;
  // cudaLaunchKernelEx reports this launch's own status (no reliance on the
  // thread's last-error state, which other code on the thread may have set)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>((long long)p.BH * p.n_t), 1, 1);
  cfg.blockDim = dim3(kBwdThreads, 1, 1);
  cfg.stream = stream;
  cfg.dynamicSmemBytes = DqLayout<D>::kAlloc;
  e = cudaLaunchKernelEx(&cfg, kdq, p);
  if (e != cudaSuccess) return e;
  cfg.dynamicSmemBytes = KvLayout<D>::kAlloc;
  return cudaLaunchKernelEx(&cfg, kkv, p);
}

template <bool F16>
cudaError_t launch_typed(const BwdParams& p, int D, bool causal, cudaStream_t stream) {
  if (D == 64)
    return causal ? launch_impl<64, true, F16>(p, stream) : launch_impl<64, false, F16>(p, stream);
  return causal ? launch_impl<128, true, F16>(p, stream) : launch_impl<128, false, F16>(p, stream);
}

}  // namespace

cudaError_t bwd_launch(const BwdParams& p, int D, bool causal, bool f16, cudaStream_t stream) {
  return f16 ? launch_typed<true>(p, D, causal, stream) : launch_typed<false>(p, D, causal, stream);
}

}  // namespace ea
