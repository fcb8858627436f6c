// umma_unit.cu — test-only unit kernel pinning the tcgen05 operand conventions
// the attention kernel relies on, with small-integer inputs whose products are
// exact in fp32:
//   S = A · Bᵀ   A, B: 128 x D bf16, K-major, TMA-loaded with 128-byte swizzle
//                (the Q·Kᵀ step)
//   O = P · V    P: 128 x 128 bf16 written to tensor memory with tcgen05.st
//                (two per 32-bit column), V: 128 x D bf16 MN-major from smem
//                (the P·V step)
// S and O are read back with tcgen05.ld and written to global memory.
// With `predicated` set, the whole MMA warp runs the issue path and every
// product and commit goes through the predicated wrappers (mma_ss_p,
// mma_ts_p, mma_commit_p) with lane 0 as the issuing lane, the form the
// backward kernels use; the results must be the same.
#include <cstdint>
#include <cstring>

#include <cuda.h>
#include <cuda_runtime.h>

#include "ptx.cuh"
#include "tmap.h"
#include "umma.cuh"

namespace {

using namespace ea;

struct UnitParams {
  CUtensorMap tm_a, tm_b, tm_v;
  const uint32_t* p_packed;  // [128][64] bf16x2
  float* s_out;              // [128][128]
  float* o_out;              // [128][D]
  int* status;
  int D;
  int predicated;
};

constexpr int kSmem = 3 * 32768 + 1024 + 256 + 1024;

__global__ void __launch_bounds__(160, 1) umma_unit_kernel(const __grid_constant__ UnitParams p) {
  extern __shared__ uint8_t raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(raw) + 1023) & ~uintptr_t(1023));
  const int tile = 128 * p.D * 2;
  uint8_t* sA = smem;
  uint8_t* sB = smem + 32768;
  uint8_t* sV = smem + 65536;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + 3 * 32768);
  uint64_t* b_load = bars;
  uint64_t* b_s = bars + 1;
  uint64_t* b_p = bars + 2;
  uint64_t* b_o = bars + 3;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(bars + 4);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(bars + 5);
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;

  if (threadIdx.x == 0) {
    mbar_init(b_load, 1);
    mbar_init(b_s, 1);
    mbar_init(b_p, 128);
    mbar_init(b_o, 1);
    mbar_init(bars + 6, 1);  // drain
    *abort_flag = 0;
    fence_barrier_init();
  }
  if (warp == 4) {
    tmem_alloc(tmem_slot, 512);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *tmem_slot;
  WaitCtl ctl{smem_u32(const_cast<int*>(abort_flag)), p.status, 1000000000ull};

  if (warp == 4) {
    // predicated: every lane of the warp runs this and lane 0 issues; else
    // lane 0 alone runs it
    const bool pred = p.predicated != 0;
    if (pred || lane == 0) {
      const bool issue = lane == 0;
      auto all = [&](bool ok) { return pred ? __all_sync(0xffffffffu, ok) : ok; };
      if (issue) {
        const uint64_t pol = l2_policy_evict_first();
        mbar_arrive_expect_tx(b_load, 3 * tile);
        for (int c = 0; c < p.D / 64; ++c) {
          tma_load_3d(sA + c * 16384, &p.tm_a, b_load, c * 64, 0, 0, pol);
          tma_load_3d(sB + c * 16384, &p.tm_b, b_load, c * 64, 0, 0, pol);
          tma_load_3d(sV + c * 16384, &p.tm_v, b_load, c * 64, 0, 0, pol);
        }
      }
      bool ok = all(wait_bounded(b_load, 0, ctl, 1));
      if (ok) {
        const uint32_t idesc_s = instr_desc_bf16(128, 128, false, false);
        for (int kk = 0; kk < p.D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * 16384 + (kk & 3) * 32;
          const uint64_t da = smem_desc_sw128(smem_u32(sA) + off, 16, 1024);
          const uint64_t db = smem_desc_sw128(smem_u32(sB) + off, 16, 1024);
          if (pred)
            mma_ss_p(issue, tmem + 0, da, db, idesc_s, kk > 0);
          else
            mma_ss(tmem + 0, da, db, idesc_s, kk > 0);
        }
        if (pred)
          mma_commit_p(issue, smem_u32(b_s));
        else
          mma_commit(b_s);
        ok = all(wait_bounded(b_p, 0, ctl, 2));
      }
      if (ok) {
        tc_fence_after_sync();
        const uint32_t idesc_o = instr_desc_bf16(128, p.D, false, true);
        for (int kk = 0; kk < 8; ++kk) {
          const uint64_t dv = smem_desc_sw128(smem_u32(sV) + kk * 2048, 16384, 1024);
          if (pred)
            mma_ts_p(issue, tmem + 256, tmem + 128 + kk * 8, dv, idesc_o, kk > 0);
          else
            mma_ts(tmem + 256, tmem + 128 + kk * 8, dv, idesc_o, kk > 0);
        }
        if (pred)
          mma_commit_p(issue, smem_u32(b_o));
        else
          mma_commit(b_o);
      }
      if (pred)
        mma_commit_p(issue, smem_u32(bars + 6));
      else
        mma_commit(bars + 6);
    }
    __syncwarp();
  } else {
    const int row = warp * 32 + lane;
    const uint32_t lane_bits = static_cast<uint32_t>(warp * 32) << 16;
    bool ok = __all_sync(0xffffffffu, wait_bounded(b_s, 0, ctl, 3));
    if (ok) {
      tc_fence_after_sync();
      for (int c = 0; c < 4; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + lane_bits + c * 32, r);
        tmem_ld_wait();
        reg_fence(r);
        for (int i = 0; i < 32; ++i) p.s_out[row * 128 + c * 32 + i] = __uint_as_float(r[i]);
      }
      for (int h = 0; h < 2; ++h) {
        uint32_t r[32];
        for (int i = 0; i < 32; ++i) r[i] = p.p_packed[row * 64 + h * 32 + i];
        tmem_st_32x32b_x32(tmem + lane_bits + 128 + h * 32, r);
      }
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(b_p);
      ok = __all_sync(0xffffffffu, wait_bounded(b_o, 0, ctl, 4));
    }
    if (ok) {
      tc_fence_after_sync();
      for (int c = 0; c < p.D / 32; ++c) {
        uint32_t r[32];
        tmem_ld_32x32b_x32(tmem + lane_bits + 256 + c * 32, r);
        tmem_ld_wait();
        reg_fence(r);
        for (int i = 0; i < 32; ++i) p.o_out[row * p.D + c * 32 + i] = __uint_as_float(r[i]);
      }
    }
    tc_fence_before_sync();
  }
  __syncthreads();
  if (warp == 4) {
    if (lane == 0) wait_drain(bars + 6, 0, 1000000000ull);
    __syncwarp();
    tc_fence_after_sync();
    tmem_dealloc(tmem, 512);
  }
}

}  // namespace

// Runs the unit kernel once and synchronises.  a, b, v: device bf16 [128][D];
// p_packed: device u32 [128][64]; s_out: device f32 [128][128]; o_out: device
// f32 [128][D]; status: device int[2]; predicated: 0 or 1 (see above).
// Returns a cudaError_t value (0 = ok), or -1 for bad arguments / tensor-map
// failure.
extern "C" __attribute__((visibility("default"))) int umma_unit_run(
    const void* a, const void* b, const void* v, const uint32_t* p_packed, float* s_out,
    float* o_out, int* status, int D, int predicated) {
  if ((D != 64 && D != 128) || (predicated != 0 && predicated != 1)) return -1;
  UnitParams prm;
  std::memset(&prm, 0, sizeof(prm));
  if (!encode_bhsd_bf16(&prm.tm_a, a, 1, 128, D, 128) || !encode_bhsd_bf16(&prm.tm_b, b, 1, 128, D, 128) ||
      !encode_bhsd_bf16(&prm.tm_v, v, 1, 128, D, 128))
    return -1;
  prm.p_packed = p_packed;
  prm.s_out = s_out;
  prm.o_out = o_out;
  prm.status = status;
  prm.D = D;
  prm.predicated = predicated;
  cudaError_t e = cudaFuncSetAttribute(umma_unit_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmem);
  if (e != cudaSuccess) return static_cast<int>(e);
  umma_unit_kernel<<<1, 160, kSmem>>>(prm);
  e = cudaGetLastError();
  if (e != cudaSuccess) return static_cast<int>(e);
  return static_cast<int>(cudaDeviceSynchronize());
}
