// attn_api.cu — the C ABI declared in include/attn.h: argument validation,
// per-device state, TMA tensor maps, launch.  No torch types, no allocation
// per call; the only memory the library owns is one status word pair per
// device, allocated on first use.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include <cuda_runtime.h>

#include "attn.h"
#include "attn_fwd.h"
#include "attn_host.h"
#include "tmap.h"

namespace {

constexpr uint64_t kDefaultWaitTimeoutNs = ATTN_DEFAULT_WAIT_TIMEOUT_NS;
constexpr int kMaxDevices = 64;
// attn_fwd_staged: inputs per chunk, and the most chunks one call uses.
constexpr int64_t kStagedChunkBytes = 48ll << 20;
constexpr int kMaxStagedChunks = 8;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int* status = nullptr;  // [0] error bits, [1] first wait site that ran out
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

// Streams and events of attn_fwd_staged on one device: uploads, kernels and
// downloads of consecutive chunks run on three streams and overlap.  Created
// on the first staged call on the device, kept until process exit; `mu`
// serialises the enqueueing of staged calls, which share the events.
struct StagedState {
  std::mutex mu;
  bool ready = false;
  cudaStream_t up = nullptr, run = nullptr, down = nullptr;
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t uploaded[kMaxStagedChunks] = {};
  cudaEvent_t computed[kMaxStagedChunks] = {};
};
StagedState g_staged[kMaxDevices];

bool staged_setup(StagedState& r) {
  if (r.ready) return true;
  const unsigned sf = cudaStreamNonBlocking;
  const unsigned ef = cudaEventDisableTiming;
  if (cudaStreamCreateWithFlags(&r.up, sf) != cudaSuccess ||
      cudaStreamCreateWithFlags(&r.run, sf) != cudaSuccess ||
      cudaStreamCreateWithFlags(&r.down, sf) != cudaSuccess ||
      cudaEventCreateWithFlags(&r.start, ef) != cudaSuccess ||
      cudaEventCreateWithFlags(&r.done, ef) != cudaSuccess)
    return false;
  for (int c = 0; c < kMaxStagedChunks; ++c)
    if (cudaEventCreateWithFlags(&r.uploaded[c], ef) != cudaSuccess ||
        cudaEventCreateWithFlags(&r.computed[c], ef) != cudaSuccess)
      return false;
  r.ready = true;
  return true;
}

using ea::overlaps;

// Validation common to every entry point; touches no CUDA API.
attn_status_t validate(const void* q, const void* k, const void* v, const void* out,
                       const void* lse, int64_t B, int64_t H, int64_t S, int64_t D, float scale,
                       int causal) {
  if (!q || !k || !v || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D > 256 || D % 8 != 0) return ATTN_ERR_UNSUPPORTED;  // 16-byte rows for TMA
  // sizes: B·H and the grid fit int32, every byte count fits int64 (2^62)
  if (B > INT32_MAX || H > INT32_MAX || S > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = B * H;  // < 2^62, no overflow
  if (BH > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  const int64_t n_qt = (S + ea::kBlockM - 1) / ea::kBlockM;
  if (BH * n_qt > INT32_MAX) return ATTN_ERR_INVALID_ARG;  // one grid CTA per Q tile
  if (BH > (int64_t(1) << 62) / (S * D * 2)) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(k) |
       reinterpret_cast<uintptr_t>(v) | reinterpret_cast<uintptr_t>(out)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return ATTN_ERR_MISALIGNED;
  const uint64_t nt = static_cast<uint64_t>(BH * S * D * 2);
  const uint64_t nl = static_cast<uint64_t>(BH * S * 4);
  if (overlaps(out, nt, q, nt) || overlaps(out, nt, k, nt) || overlaps(out, nt, v, nt) ||
      overlaps(lse, nl, q, nt) || overlaps(lse, nl, k, nt) || overlaps(lse, nl, v, nt) ||
      overlaps(lse, nl, out, nt))
    return ATTN_ERR_INVALID_ARG;
  return ATTN_OK;
}

// Per-device set-up on first use: architecture check and the status words.
attn_status_t device_state(int* dev_out, DeviceState** st_out) {
  int dev = -1;
  const cudaError_t e = ea::current_device_bound(&dev);
  if (e != cudaSuccess) return ea::cuda_failure(static_cast<int>(e));
  if (dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceState& st = g_dev[dev];
  if (!st.ready) {
    int major = 0, minor = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
      return ATTN_ERR_CUDA;
    st.supported = (major == 10 && minor == 3);
    if (st.supported) {
      void* p = nullptr;
      if (cudaMalloc(&p, 2 * sizeof(int)) != cudaSuccess) return ATTN_ERR_CUDA;
      if (cudaMemset(p, 0, 2 * sizeof(int)) != cudaSuccess) {
        cudaFree(p);
        return ATTN_ERR_CUDA;
      }
      st.status = static_cast<int*>(p);
    }
    st.ready = true;
  }
  if (!st.supported) return ATTN_ERR_UNSUPPORTED;
  *dev_out = dev;
  *st_out = &st;
  return ATTN_OK;
}

attn_status_t launch(const void* q, const void* k, const void* v, void* out, float* lse, int64_t B,
                     int64_t H, int64_t S, int64_t D, float scale, int causal, bool f16,
                     uint64_t timeout_ns, cudaStream_t stream) {
  int dev = -1;
  DeviceState* st = nullptr;
  attn_status_t s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  return ea::launch_with_status(q, k, v, out, lse, B, H, S, D, scale, causal, f16, timeout_ns,
                                st->status, stream);
}

}  // namespace

namespace ea {

attn_status_t validate_args(const void* q, const void* k, const void* v, const void* out,
                            const void* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                            float scale, int causal) {
  return validate(q, k, v, out, lse, B, H, S, D, scale, causal);
}

attn_status_t current_status_words(int** status) {
  int dev = -1;
  DeviceState* st = nullptr;
  attn_status_t s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  *status = st->status;
  return ATTN_OK;
}

attn_status_t launch_with_status(const void* q, const void* k, const void* v, void* out,
                                 float* lse, int64_t B, int64_t H, int64_t S, int64_t D,
                                 float scale, int causal, bool f16, uint64_t timeout_ns,
                                 int* status, cudaStream_t stream) {
  const int64_t BH = B * H;
  // The kernels exist for 64, 128, 192 and 256 columns; another head
  // dimension runs on the next one up.  The tensor maps carry the real column count,
  // so TMA loads read zeros past it and stores leave those columns out; the
  // zero columns add nothing to q·kᵀ and give zero output columns.
  const int dk = forward_head_dim(D);
  // 64 and 128 columns: the persistent kernel (one CTA per SM walking Q
  // tiles); 192 and 256 columns: one Q tile per CTA with 64-row K/V tiles
  // (their output tile does not fit the persistent kernel's staging buffer).
  const bool persistent = dk <= 128;
  const int bn = dk > 128 ? 64 : 128;  // rows of one K/V tile
  Fwd1QParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_bhsd_16bit(&p.tm_k, k, BH, S, D, bn, f16) ||
      !encode_bhsd_16bit(&p.tm_v, v, BH, S, D, bn, f16) ||
      !encode_bhsd_16bit(&p.tm_o, out, BH, S, D, 32, f16) ||
      !encode_bhsd_16bit(&p.tm_q, q, BH, S, D, 128, f16))
    return cuda_failure(kErrTensorMap);
  p.q = static_cast<const uint16_t*>(q);
  p.lse = lse;
  p.status = status;
  p.BH = static_cast<int>(BH);
  p.S = static_cast<int>(S);
  p.d_cols = static_cast<int>(D);
  p.n_qt = static_cast<int>((S + kBlockM - 1) / kBlockM);
  p.n_kt = static_cast<int>((S + bn - 1) / bn);
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return cuda_failure(static_cast<int>(e));
  p.sched = plan_schedule(BH, p.n_qt, S, D, causal != 0, kL2GroupBytes, sms);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.timeout_ns = timeout_ns;
  e = persistent ? fwd1qp_launch(p, dk, causal != 0, f16, stream)
                 : fwd1q_launch(p, dk, causal != 0, f16, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return cuda_failure(static_cast<int>(e));
  }
  return ATTN_OK;
}

}  // namespace ea

extern "C" {

attn_status_t attn_fwd_bounded(const void* q, const void* k, const void* v, void* out, float* lse,
                               int64_t B, int64_t H, int64_t S, int64_t D, float scale, int causal,
                               uint64_t wait_timeout_ns, cudaStream_t stream) {
  attn_status_t s = validate(q, k, v, out, lse, B, H, S, D, scale, causal);
  if (s != ATTN_OK) return s;
  return launch(q, k, v, out, lse, B, H, S, D, scale, causal, false, wait_timeout_ns, stream);
}

attn_status_t attn_fwd_ex(const void* q, const void* k, const void* v, void* out, float* lse,
                          int64_t B, int64_t H, int64_t S, int64_t D, float scale, int causal,
                          attn_dtype_t dtype, uint64_t wait_timeout_ns, cudaStream_t stream) {
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_INVALID_ARG;
  attn_status_t s = validate(q, k, v, out, lse, B, H, S, D, scale, causal);
  if (s != ATTN_OK) return s;
  return launch(q, k, v, out, lse, B, H, S, D, scale, causal, dtype == ATTN_F16, wait_timeout_ns,
                stream);
}

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* out, float* lse,
                       int64_t B, int64_t H, int64_t S, int64_t D, float scale, int causal,
                       cudaStream_t stream) {
  return attn_fwd_bounded(q, k, v, out, lse, B, H, S, D, scale, causal, kDefaultWaitTimeoutNs,
                          stream);
}

attn_status_t attn_fwd_staged(const void* q_h, const void* k_h, const void* v_h, void* out_h,
                              float* lse_h, void* q_d, void* k_d, void* v_d, void* out_d,
                              float* lse_d, int64_t B, int64_t H, int64_t S, int64_t D,
                              float scale, int causal, cudaStream_t stream) {
  if (!q_h || !k_h || !v_h || !out_h || !lse_h) return ATTN_ERR_INVALID_ARG;
  attn_status_t s = validate(q_d, k_d, v_d, out_d, lse_d, B, H, S, D, scale, causal);
  if (s != ATTN_OK) return s;
  if (q_d == k_d || q_d == v_d || k_d == v_d) return ATTN_ERR_INVALID_ARG;
  int dev = -1;
  DeviceState* st = nullptr;
  s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  StagedState& r = g_staged[dev];
  std::lock_guard<std::mutex> lock(r.mu);
  if (!staged_setup(r)) return ATTN_ERR_CUDA;

  // Chunks of (b, h) slices: chunk c's kernel overlaps chunk c+1's upload
  // and chunk c-1's download.  Every stream starts after the work already on
  // `stream`, and `stream` continues once the last download is done.
  const int64_t BH = B * H;
  const int64_t slice = S * D * 2;  // bytes of one slice of q, k, v or out
  const int n = ea::staged_chunk_count(BH, 3 * slice, kStagedChunkBytes, kMaxStagedChunks);
  auto ok = [](cudaError_t e) { return e == cudaSuccess; };
  if (!ok(cudaEventRecord(r.start, stream)) || !ok(cudaStreamWaitEvent(r.up, r.start, 0)) ||
      !ok(cudaStreamWaitEvent(r.run, r.start, 0)) || !ok(cudaStreamWaitEvent(r.down, r.start, 0)))
    return ATTN_ERR_CUDA;
  const auto H2D = cudaMemcpyHostToDevice;
  const auto D2H = cudaMemcpyDeviceToHost;
  for (int c = 0; c < n; ++c) {
    int64_t first = 0, count = 0;
    ea::staged_chunk_range(BH, n, c, &first, &count);
    const size_t off = static_cast<size_t>(first * slice), len = static_cast<size_t>(count * slice);
    const size_t loff = static_cast<size_t>(first * S), llen = static_cast<size_t>(count * S * 4);
    auto dptr = [off](void* p) { return static_cast<char*>(p) + off; };
    auto hptr = [off](const void* p) { return static_cast<const char*>(p) + off; };
    if (!ok(cudaMemcpyAsync(dptr(q_d), hptr(q_h), len, H2D, r.up)) ||
        !ok(cudaMemcpyAsync(dptr(k_d), hptr(k_h), len, H2D, r.up)) ||
        !ok(cudaMemcpyAsync(dptr(v_d), hptr(v_h), len, H2D, r.up)) ||
        !ok(cudaEventRecord(r.uploaded[c], r.up)) ||
        !ok(cudaStreamWaitEvent(r.run, r.uploaded[c], 0)))
      return ATTN_ERR_CUDA;
    s = ea::launch_with_status(dptr(q_d), dptr(k_d), dptr(v_d), dptr(out_d), lse_d + loff, 1,
                               count, S, D, scale, causal, false, kDefaultWaitTimeoutNs,
                               st->status, r.run);
    if (s != ATTN_OK) return s;
    if (!ok(cudaEventRecord(r.computed[c], r.run)) ||
        !ok(cudaStreamWaitEvent(r.down, r.computed[c], 0)) ||
        !ok(cudaMemcpyAsync(static_cast<char*>(out_h) + off, dptr(out_d), len, D2H, r.down)) ||
        !ok(cudaMemcpyAsync(lse_h + loff, lse_d + loff, llen, D2H, r.down)))
      return ATTN_ERR_CUDA;
  }
  if (!ok(cudaEventRecord(r.done, r.down)) || !ok(cudaStreamWaitEvent(stream, r.done, 0)))
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_device_status(cudaStream_t stream) {
  int dev = -1;
  DeviceState* st = nullptr;
  attn_status_t s = device_state(&dev, &st);
  if (s != ATTN_OK) return s;
  if (cudaStreamSynchronize(stream) != cudaSuccess) return ATTN_ERR_CUDA;
  int h[2] = {0, 0};
  if (cudaMemcpy(h, st->status, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess)
    return ATTN_ERR_CUDA;
  if (h[0] == 0) return ATTN_OK;
  if (cudaMemset(st->status, 0, sizeof(h)) != cudaSuccess) return ATTN_ERR_CUDA;
  return ea::status_of_words(h[0]);
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED:
      return "unsupported (head_dim must be a multiple of 8, at most 256 (128 for the backward); "
             "device must be sm_103)";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer (q/k/v/out need 16 bytes, lse 4 bytes)";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "an in-kernel wait ran out of time";
    case ATTN_ERR_DEVICE_CHECK:
      return "an in-kernel index check failed (debug build); the access was skipped";
  }
  return "unknown status";
}

attn_status_t attn_shard_range(int64_t units, int world, int rank, int64_t* first,
                               int64_t* count) {
  if (units < 0 || world < 1 || rank < 0 || rank >= world || !first || !count)
    return ATTN_ERR_INVALID_ARG;
  const int64_t base = units / world, extra = units % world;
  *count = base + (rank < extra ? 1 : 0);
  *first = rank * base + (rank < extra ? rank : extra);
  return ATTN_OK;
}

int attn_abi_version(void) { return 1; }

int attn_last_cuda_error(void) { return ea::g_last_cuda_error; }

}  // extern "C"
