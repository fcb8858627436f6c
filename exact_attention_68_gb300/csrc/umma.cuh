// umma.cuh — descriptors of the tcgen05 (5th-generation tensor core) MMA.
//
// Shared-memory matrix descriptor (64 bit) and instruction descriptor
// (32 bit, kind::f16) as laid out for sm_100-family tensor cores.  Field
// positions:
//   smem descriptor: [0,14) start address >> 4; [16,30) leading-dimension byte
//     offset >> 4; [32,46) stride-dimension byte offset >> 4; [46,48) version
//     (1 on this tensor-core generation); [49,52) base offset; [52] LBO mode;
//     [61,64) swizzle (2 = 128-byte swizzle).
//   instruction descriptor: [4,6) D format (1 = f32); [7,10) A format
//     (1 = bf16); [10,13) B format; [15] A major (0 = K-major); [16] B major
//     (1 = MN-major); [17,23) N >> 3; [24,29) M >> 4.
//
// Operand layouts used (all 128-byte swizzled, as TMA writes them):
//   K-major tile of R rows x 64 bf16 (128 B per row): 8-row groups of 1024 B,
//     SBO = 1024 (next 8 rows), LBO unused; a K step of 16 elements is +32 B on
//     the start address, and the next 64-element column block is a separate
//     R x 128 B region.
//   MN-major tile (V as the B operand of P·V, N = head dim contiguous):
//     LBO = byte distance between 64-element N blocks, SBO = 1024 (next 8 K
//     rows); a K step of 16 rows is +2048 B.
#pragma once

#include <cstdint>

namespace ea {

__host__ __device__ constexpr uint64_t smem_desc_sw128(uint32_t saddr, uint32_t lbo_bytes,
                                                       uint32_t sbo_bytes) {
  return (uint64_t)((saddr >> 4) & 0x3FFFu) | ((uint64_t)((lbo_bytes >> 4) & 0x3FFFu) << 16) |
         ((uint64_t)((sbo_bytes >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (2ull << 61);
}

// A, B both fp16 (f16 = true, format 0) or both bf16 (format 1) -> f32, dense.
__host__ __device__ constexpr uint32_t instr_desc_16bit(int M, int N, bool a_mn_major,
                                                        bool b_mn_major, bool f16) {
  return (1u << 4) | ((f16 ? 0u : 1u) << 7) | ((f16 ? 0u : 1u) << 10) |
         ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// bf16 x bf16 -> f32, dense.
__host__ __device__ constexpr uint32_t instr_desc_bf16(int M, int N, bool a_mn_major,
                                                       bool b_mn_major) {
  return instr_desc_16bit(M, N, a_mn_major, b_mn_major, false);
}

}  // namespace ea
