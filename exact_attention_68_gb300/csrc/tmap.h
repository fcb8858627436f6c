// tmap.h — host-side TMA tensor-map encoding for [B·H, S, D] bf16 tensors.
//
// cuTensorMapEncodeTiled is a driver entry point; it is resolved through the
// runtime (cudaGetDriverEntryPointByVersion) so that the library links no
// driver library and loads on machines without a GPU.
#pragma once

#include <cstdint>
#include <mutex>
#include <cuda.h>
#include <cuda_runtime_api.h>
#include <cudaTypedefs.h>

namespace ea {

inline PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault,
                                         &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
  });
  return fn;
}

// 3-D map (D, S, BH) of a contiguous 16-bit (fp16 if f16, else bf16)
// [BH, S, D] tensor with a box of
// 64 columns x box_rows rows x 1, 128-byte swizzle.  Rows past S read as zero
// and are not written by stores, so tiles never cross into the next head.
inline bool encode_bhsd_16bit(CUtensorMap* map, const void* base, int64_t BH, int64_t S, int64_t D,
                              uint32_t box_rows, bool f16) {
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return false;
  cuuint64_t dims[3] = {(cuuint64_t)D, (cuuint64_t)S, (cuuint64_t)BH};
  cuuint64_t strides[2] = {(cuuint64_t)(D * 2), (cuuint64_t)(S * D * 2)};
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = enc(map, f16 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT16 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3,
                   const_cast<void*>(base), dims, strides,
                   box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                   CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

inline bool encode_bhsd_bf16(CUtensorMap* map, const void* base, int64_t BH, int64_t S, int64_t D,
                             uint32_t box_rows) {
  return encode_bhsd_16bit(map, base, BH, S, D, box_rows, false);
}

}  // namespace ea
