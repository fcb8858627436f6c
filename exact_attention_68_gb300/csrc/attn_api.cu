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

constexpr uint64_t kDefaultWaitTimeoutNs = 2000000000ull;  // 2 s per in-kernel wait
// K/V bytes of the (b, h) slices one scheduling group spans: well under the
// 129 MB L2, so that the CTAs running at one time re-read K/V tiles from L2.
constexpr int64_t kL2GroupBytes = 48ll << 20;
constexpr int kMaxDevices = 64;

struct DeviceState {
  bool ready = false;
  bool supported = false;
  int* status = nullptr;  // [0] error bits, [1] first wait site that ran out
};

std::mutex g_mu;
DeviceState g_dev[kMaxDevices];

bool overlaps(const void* a, uint64_t na, const void* b, uint64_t nb) {
  const uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
  return x < y + nb && y < x + na;
}

// Validation common to every entry point; touches no CUDA API.
attn_status_t validate(const void* q, const void* k, const void* v, const void* out,
                       const void* lse, int64_t B, int64_t H, int64_t S, int64_t D, float scale,
                       int causal) {
  if (!q || !k || !v || !out || !lse) return ATTN_ERR_INVALID_ARG;
  if (B < 1 || H < 1 || S < 1 || D < 1) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || !(scale > 0.f)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // sizes: B·H and the grid fit int32, every byte count fits int64 (2^62)
  if (B > INT32_MAX || H > INT32_MAX || S > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  const int64_t BH = B * H;  // < 2^62, no overflow
  if (BH > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  const int64_t n_qt = (S + ea::kBlockM - 1) / ea::kBlockM;
  const int64_t n_units = (n_qt + ea::kQTilesPerUnit - 1) / ea::kQTilesPerUnit;
  if (BH * n_units > INT32_MAX) return ATTN_ERR_INVALID_ARG;
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
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return ATTN_ERR_CUDA;
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
  FwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int64_t BH = B * H;
  if (!encode_bhsd_16bit(&p.tm_q, q, BH, S, D, kBlockM, f16) ||
      !encode_bhsd_16bit(&p.tm_k, k, BH, S, D, kBlockN, f16) ||
      !encode_bhsd_16bit(&p.tm_v, v, BH, S, D, kBlockN, f16) ||
      !encode_bhsd_16bit(&p.tm_o, out, BH, S, D, 32, f16))
    return ATTN_ERR_CUDA;
  p.lse = lse;
  p.status = status;
  p.B = static_cast<int>(B);
  p.H = static_cast<int>(H);
  p.S = static_cast<int>(S);
  p.n_qt = static_cast<int>((S + kBlockM - 1) / kBlockM);
  p.n_units = (p.n_qt + kQTilesPerUnit - 1) / kQTilesPerUnit;
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
    return ATTN_ERR_CUDA;
  p.sched = plan_schedule(BH, p.n_units, S, D, causal != 0, kL2GroupBytes, sms);
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.timeout_ns = timeout_ns;
  if (fwd_launch(p, static_cast<int>(D), causal != 0, f16, stream) != cudaSuccess) {
    (void)cudaGetLastError();
    return ATTN_ERR_CUDA;
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
  const size_t nt = static_cast<size_t>(B * H * S * D * 2);
  const size_t nl = static_cast<size_t>(B * H * S * 4);
  if (cudaMemcpyAsync(q_d, q_h, nt, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(k_d, k_h, nt, cudaMemcpyHostToDevice, stream) != cudaSuccess ||
      cudaMemcpyAsync(v_d, v_h, nt, cudaMemcpyHostToDevice, stream) != cudaSuccess)
    return ATTN_ERR_CUDA;
  s = launch(q_d, k_d, v_d, out_d, lse_d, B, H, S, D, scale, causal, false, kDefaultWaitTimeoutNs,
             stream);
  if (s != ATTN_OK) return s;
  if (cudaMemcpyAsync(out_h, out_d, nt, cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
      cudaMemcpyAsync(lse_h, lse_d, nl, cudaMemcpyDeviceToHost, stream) != cudaSuccess)
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
  return ATTN_ERR_TIMEOUT;
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported (head_dim must be 64 or 128; device must be sm_103)";
    case ATTN_ERR_MISALIGNED: return "misaligned pointer (q/k/v/out need 16 bytes, lse 4 bytes)";
    case ATTN_ERR_CUDA: return "CUDA call failed";
    case ATTN_ERR_TIMEOUT: return "an in-kernel wait ran out of time";
  }
  return "unknown status";
}

int attn_abi_version(void) { return 1; }

}  // extern "C"
