// attn_host.h — host helpers shared by the C-ABI translation units: argument
// validation and the tensor-map + launch step with a caller-chosen status
// word pair.
#pragma once

#include <cstdint>
#include <cuda_runtime_api.h>

#include "attn.h"

namespace ea {

// Argument checks of attn_fwd; touches no CUDA API.
attn_status_t validate_args(const void* q, const void* k, const void* v, const void* out,
                            const void* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                            float scale, int causal);

// Encodes the tensor maps and launches the forward with `status` (device
// int[2]: error bits, first wait site that ran out) as its status words.
// f16: the 16-bit tensors are fp16 (else bf16).
attn_status_t launch_with_status(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                 float scale, int causal, bool f16, uint64_t timeout_ns,
                                 int* status, cudaStream_t stream);

// What the last ATTN_ERR_CUDA on this thread came from: a cudaError_t, or
// kErrTensorMap when a TMA tensor map could not be encoded (0: none).
constexpr int kErrTensorMap = -1;
inline thread_local int g_last_cuda_error = 0;
inline attn_status_t cuda_failure(int code) {
  g_last_cuda_error = code;
  return ATTN_ERR_CUDA;
}

// The calling thread's current device, with its primary context made current
// on this thread: the TMA tensor maps are encoded by a driver call, which
// needs a current context, and a thread that has only ever called
// cudaGetDevice has none yet.
inline cudaError_t current_device_bound(int* dev) {
  cudaError_t e = cudaGetDevice(dev);
  if (e == cudaSuccess) e = cudaSetDevice(*dev);
  return e;
}

// Columns of the kernel that runs a head dimension D (a multiple of 8, at
// most 256): the smallest of 64, 128, 256 that holds D.
inline int kernel_head_dim(int64_t D) { return D <= 64 ? 64 : D <= 128 ? 128 : 256; }
// The forward also has a kernel 192 columns wide, so that head dimensions
// 136-192 do not pay for 256.
inline int forward_head_dim(int64_t D) { return D <= 128 ? kernel_head_dim(D) : D <= 192 ? 192 : 256; }

// The status a non-zero device status word reports: its bits are 1 (a wait
// ran out) and 2 (an index check of a debug build failed).
inline attn_status_t status_of_words(int bits) {
  return (bits & 2) ? ATTN_ERR_DEVICE_CHECK : ATTN_ERR_TIMEOUT;
}

// True if the byte ranges [a, a+na) and [b, b+nb) intersect.
inline bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// The current device's status word pair (allocated on first use), after the
// architecture check.
attn_status_t current_status_words(int** status);

}  // namespace ea
