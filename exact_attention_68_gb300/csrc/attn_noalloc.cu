// attn_noalloc.cu — attn_fwd_noalloc: the attention forward for callers that
// may not allocate device memory.
//
// Who needs it: a program whose device memory is owned by its own allocator
// (a serving process or framework that reserves the HBM it will use up front
// and hands out slices of it), code that must stay within a fixed, audited
// device-memory budget, and latency-critical paths that may not pay for
// cudaMalloc, which can synchronise the whole device.  The other entry points
// cudaMalloc one small status buffer on their first call on each device; this
// one calls no cudaMalloc, no cudaFree and no other allocating routine.
//
// Its scratch — the kernel's two status words (error bits, and the first
// in-kernel wait that ran out) — lives instead in g_noalloc_scratch below, a
// file-scope __device__ array of ATTN_NOALLOC_SCRATCH_BYTES.  Every GPU that
// loads this library holds that array until the process exits.  In host code
// the array's name is only a host-side stand-in, not a device address, so the
// address passed to the kernel comes from cudaGetSymbolAddress, taken once
// per device with that device current, on the first call on that device.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"
#include "attn_host.h"

namespace {

constexpr int kMaxDevices = 64;
constexpr uint64_t kWaitTimeoutNs = ATTN_DEFAULT_WAIT_TIMEOUT_NS;  // the bound attn_fwd uses
// Scratch the forward kernel needs: its two status words.  The need does not
// grow with B, H, S or D.
constexpr size_t kScratchNeedBytes = 2 * sizeof(int);
static_assert(kScratchNeedBytes <= ATTN_NOALLOC_SCRATCH_BYTES,
              "the kernel's scratch must fit the static array (a build-time limit)");

static __device__ __align__(256) int g_noalloc_scratch[ATTN_NOALLOC_SCRATCH_BYTES / sizeof(int)];

struct NoAllocDevice {
  bool ready = false;
  bool supported = false;
  int* scratch = nullptr;  // device address of g_noalloc_scratch on this device
};

std::mutex g_mu;
NoAllocDevice g_dev[kMaxDevices];

// One-time set-up of the current device: architecture check and the device
// address of the scratch array.  Nothing is allocated.
attn_status_t noalloc_setup(int** scratch) {
  int dev = -1;
  // binds the device's primary context to this thread (the tensor maps are
  // encoded by a driver call); allocates nothing
  const cudaError_t e = ea::current_device_bound(&dev);
  if (e != cudaSuccess) return ea::cuda_failure(static_cast<int>(e));
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  NoAllocDevice& d = g_dev[dev];
  if (!d.ready) {
    int major = 0, minor = 0;
    cudaError_t ae = cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev);
    if (ae == cudaSuccess) ae = cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev);
    if (ae != cudaSuccess) return ea::cuda_failure(static_cast<int>(ae));
    d.supported = (major == 10 && minor == 3);
    if (d.supported) {
      void* ptr = nullptr;
      const cudaError_t se = cudaGetSymbolAddress(&ptr, g_noalloc_scratch);
      // not marked ready on failure: the next call tries again
      if (se != cudaSuccess) return ea::cuda_failure(static_cast<int>(se));
      if (ptr == nullptr) return ea::cuda_failure(static_cast<int>(cudaErrorInvalidSymbol));
      d.scratch = static_cast<int*>(ptr);
    }
    d.ready = true;
  }
  if (!d.supported) return ATTN_ERR_UNSUPPORTED;
  *scratch = d.scratch;
  return ATTN_OK;
}

}  // namespace

extern "C" attn_status_t attn_fwd_noalloc(const void* q, const void* k, const void* v, void* out,
                                          float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                          float scale, int causal, int check_status,
                                          cudaStream_t stream) {
  attn_status_t s = ea::validate_args(q, k, v, out, lse, B, H, S, D, scale, causal);
  if (s != ATTN_OK) return s;
  if (check_status != 0 && check_status != 1) return ATTN_ERR_INVALID_ARG;
  int* scratch = nullptr;
  s = noalloc_setup(&scratch);
  if (s != ATTN_OK) return s;
  if (check_status) {
    // check_status synchronises the stream, which a stream being captured
    // into a graph does not allow: refuse before anything is enqueued
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    const cudaError_t ce = cudaStreamIsCapturing(stream, &cap);
    if (ce != cudaSuccess) return ea::cuda_failure(static_cast<int>(ce));
    if (cap != cudaStreamCaptureStatusNone) return ATTN_ERR_INVALID_ARG;
  }
  // The array keeps the previous call's words: clear them for this call.
  cudaError_t e = cudaMemsetAsync(scratch, 0, kScratchNeedBytes, stream);
  if (e != cudaSuccess) return ea::cuda_failure(static_cast<int>(e));
  s = ea::launch_with_status(q, k, v, out, lse, B, H, S, D, scale, causal, /*f16=*/false,
                             kWaitTimeoutNs, scratch, stream);
  if (s != ATTN_OK || !check_status) return s;
  int words[2] = {0, 0};
  e = cudaMemcpyAsync(words, scratch, sizeof(words), cudaMemcpyDeviceToHost, stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(stream);
  if (e != cudaSuccess) return ea::cuda_failure(static_cast<int>(e));
  return words[0] != 0 ? ea::status_of_words(words[0]) : ATTN_OK;
}
