// bwd_common.cuh — device helpers shared by the backward kernels (head
// dimensions up to 128 in attn_bwd_sm103.cu, up to 256 in attn_bwd256_sm103.cu).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_fp16.h>

#include "ptx.cuh"

namespace ea {
namespace {

// debug-check sites (-DATTN_DEBUG) of the output store below
enum : int { kChkAccTmem = 0x5201, kChkStage = 0x5202, kChkStore = 0x5203 };

__device__ __forceinline__ float bf16_lo(uint32_t x) { return __uint_as_float(x << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t x) { return __uint_as_float(x & 0xffff0000u); }

__device__ __forceinline__ float2 f16x2_to_f32(uint32_t x) {
  return __half22float2(*reinterpret_cast<const __half2*>(&x));
}

// Σ a_e·b_e over 8 packed 16-bit values (fp16 if F16, else bf16), in fp32.
template <bool F16>
__device__ __forceinline__ float dot8(uint4 a, uint4 b) {
  const uint32_t av[4] = {a.x, a.y, a.z, a.w};
  const uint32_t bv[4] = {b.x, b.y, b.z, b.w};
  float s = 0.f;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    if constexpr (F16) {
      const float2 x = f16x2_to_f32(av[t]), y = f16x2_to_f32(bv[t]);
      s = fmaf(x.x, y.x, s);
      s = fmaf(x.y, y.y, s);
    } else {
      s = fmaf(bf16_lo(av[t]), bf16_lo(bv[t]), s);
      s = fmaf(bf16_hi(av[t]), bf16_hi(bv[t]), s);
    }
  }
  return s;
}

__device__ __forceinline__ void st_shared_f32x2(uint32_t addr, float a, float b) {
  asm volatile("st.shared.v2.f32 [%0], {%1, %2};" ::"r"(addr), "f"(a), "f"(b) : "memory");
}

// One warp's 32 rows × 64 columns of an fp32 TMEM accumulator, times `mul`,
// to bf16 in the 128-byte-swizzled staging block `chunk_base` (row = TMEM
// lane), then one TMA store of the warp's rows.  Only lane 0 issues the store.
// A chunk that starts at or past the tensor's last column (dbb.cols) is not
// stored: a store box never starts outside the tensor.  Call with the full warp.
template <bool F16>
__device__ __forceinline__ void store_chunk(uint32_t tmem_col, uint32_t chunk_base, int row,
                                            float mul, const CUtensorMap* map, int x, int y0,
                                            int z, int wq, int lane, const DbgBounds& dbb) {
  if (x >= dbb.cols) return;
  if (!dbg_warp(dbg_tmem(dbb, tmem_col, 64, wq, kChkAccTmem))) return;
#pragma unroll
  for (int half = 0; half < 2; ++half) {
    uint32_t o[32];
    tmem_ld_32x32b_x32(tmem_col + half * 32, o);
    tmem_ld_wait();
    reg_fence(o);
#pragma unroll
    for (int q4 = 0; q4 < 4; ++q4) {
      const int u16 = half * 4 + q4;  // 16-byte unit along the 128-byte row
      const uint32_t addr = chunk_base + row * 128 + ((u16 ^ (row & 7)) << 4);
      uint32_t w[4];
#pragma unroll
      for (int e = 0; e < 4; ++e)
        w[e] = pack_x2<F16>(__uint_as_float(o[q4 * 8 + 2 * e]) * mul,
                           __uint_as_float(o[q4 * 8 + 2 * e + 1]) * mul);
      if (dbg_smem(dbb, addr, 16, 16, kChkStage)) st_shared_v4(addr, w[0], w[1], w[2], w[3]);
    }
  }
  fence_proxy_async_smem();
  __syncwarp();
  // the warp's 32 rows, if any of them is inside the tensor
  const int y = y0 + wq * 32;
  const uint32_t src = chunk_base + wq * 32 * 128;
  if (lane == 0 && y < dbb.rows && dbg_tma(dbb, src, 32 * 128, x, y, z, true, kChkStore))
    tma_store_3d(map, src, x, y, z);
}

}  // namespace
}  // namespace ea
