// attn_bwd_api.cu — the backward entry points of the C ABI declared in
// include/attn.h: argument validation, tensor maps, launch of the two kernels.
#include <cmath>
#include <cstdint>
#include <cstring>

#include <cuda_runtime.h>

#include "attn.h"
#include "attn_bwd.h"
#include "attn_host.h"
#include "tmap.h"

namespace {

constexpr uint64_t kDefaultWaitTimeoutNs = ATTN_DEFAULT_WAIT_TIMEOUT_NS;
using ea::overlaps;

// Checks of attn_bwd; touches no CUDA API.
attn_status_t validate_bwd(const void* q, const void* k, const void* v, const void* out,
                           const float* lse, const void* dout, const void* dq, const void* dk,
                           const void* dv, const float* delta, int64_t B, int64_t H, int64_t S,
                           int64_t D, float scale, int causal) {
  // shapes, scale, mask flag, q/k/v/out/lse pointers and alignment
  attn_status_t s = ea::validate_args(q, k, v, out, lse, B, H, S, D, scale, causal);
  if (s != ATTN_OK) return s;
  if (!dout || !dq || !dk || !dv || !delta) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(dout) | reinterpret_cast<uintptr_t>(dq) |
       reinterpret_cast<uintptr_t>(dk) | reinterpret_cast<uintptr_t>(dv)) & 15u)
    return ATTN_ERR_MISALIGNED;
  if (reinterpret_cast<uintptr_t>(delta) & 3u) return ATTN_ERR_MISALIGNED;
  const uint64_t nt = static_cast<uint64_t>(B * H * S * D * 2);
  const uint64_t nl = static_cast<uint64_t>(B * H * S * 4);
  const void* ins[6] = {q, k, v, out, lse, dout};
  const uint64_t in_bytes[6] = {nt, nt, nt, nt, nl, nt};
  const void* outs[4] = {dq, dk, dv, delta};
  const uint64_t out_bytes[4] = {nt, nt, nt, nl};
  for (int a = 0; a < 4; ++a) {
    for (int b = 0; b < 6; ++b)
      if (overlaps(outs[a], out_bytes[a], ins[b], in_bytes[b])) return ATTN_ERR_INVALID_ARG;
    for (int b = a + 1; b < 4; ++b)
      if (overlaps(outs[a], out_bytes[a], outs[b], out_bytes[b])) return ATTN_ERR_INVALID_ARG;
  }
  return ATTN_OK;
}

}  // namespace

extern "C" {

attn_status_t attn_bwd_ex(const void* q, const void* k, const void* v, const void* out,
                          const float* lse, const void* dout, void* dq, void* dk, void* dv,
                          float* delta, int64_t B, int64_t H, int64_t S, int64_t D, float scale,
                          int causal, attn_dtype_t dtype, uint64_t wait_timeout_ns,
                          cudaStream_t stream) {
  if (dtype != ATTN_BF16 && dtype != ATTN_F16) return ATTN_ERR_INVALID_ARG;
  const bool f16 = dtype == ATTN_F16;
  attn_status_t s = validate_bwd(q, k, v, out, lse, dout, dq, dk, dv, delta, B, H, S, D, scale,
                                 causal);
  if (s != ATTN_OK) return s;
  int* status = nullptr;
  s = ea::current_status_words(&status);
  if (s != ATTN_OK) return s;
  ea::BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int64_t BH = B * H;
  if (!ea::encode_bhsd_16bit(&p.tm_q, q, BH, S, D, 128, f16) ||
      !ea::encode_bhsd_16bit(&p.tm_k, k, BH, S, D, 128, f16) ||
      !ea::encode_bhsd_16bit(&p.tm_v, v, BH, S, D, 128, f16) ||
      !ea::encode_bhsd_16bit(&p.tm_do, dout, BH, S, D, 128, f16) ||
      !ea::encode_bhsd_16bit(&p.tm_dq, dq, BH, S, D, 32, f16) ||
      !ea::encode_bhsd_16bit(&p.tm_dk, dk, BH, S, D, 32, f16) ||
      !ea::encode_bhsd_16bit(&p.tm_dv, dv, BH, S, D, 32, f16))
    return ea::cuda_failure(ea::kErrTensorMap);
  const int width = ea::kernel_head_dim(D);
  if (width == 256 && (!ea::encode_bhsd_16bit(&p.tm_q64, q, BH, S, D, 64, f16) ||
                       !ea::encode_bhsd_16bit(&p.tm_k64, k, BH, S, D, 64, f16) ||
                       !ea::encode_bhsd_16bit(&p.tm_v64, v, BH, S, D, 64, f16) ||
                       !ea::encode_bhsd_16bit(&p.tm_do64, dout, BH, S, D, 64, f16)))
    return ea::cuda_failure(ea::kErrTensorMap);
  p.q = static_cast<const uint16_t*>(q);
  p.k = static_cast<const uint16_t*>(k);
  p.v = static_cast<const uint16_t*>(v);
  p.out = static_cast<const uint16_t*>(out);
  p.dout = static_cast<const uint16_t*>(dout);
  p.lse = lse;
  p.delta = delta;
  p.status = status;
  p.BH = static_cast<int>(BH);
  p.S = static_cast<int>(S);
  p.d_cols = static_cast<int>(D);
  p.n_t = static_cast<int>((S + 127) / 128);
  if (static_cast<int64_t>(p.BH) * p.n_t > INT32_MAX) return ATTN_ERR_INVALID_ARG;
  int dev = 0, sms = 0;
  cudaError_t de = cudaGetDevice(&dev);
  if (de == cudaSuccess) de = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (de != cudaSuccess) return ea::cuda_failure(static_cast<int>(de));
  // one grid order for both kernels: each streams one slice's tiles of two
  // tensors (K, V or Q, dout), as many bytes as the forward's K, V
  p.sched = ea::plan_schedule(BH, p.n_t, S, D, causal != 0, ea::kL2GroupBytes, sms);
  p.scale = scale;
  p.scale_log2 = static_cast<float>(static_cast<double>(scale) * 1.4426950408889634);
  p.timeout_ns = wait_timeout_ns;
  // kernels of 64, 128 or 256 columns; the tensor maps carry the real column
  // count (zeros read past it, those columns never stored)
  const cudaError_t e = width == 256 ? ea::bwd256_launch(p, causal != 0, f16, stream)
                                     : ea::bwd_launch(p, width, causal != 0, f16, stream);
  if (e != cudaSuccess) {
    (void)cudaGetLastError();
    return ea::cuda_failure(static_cast<int>(e));
  }
  return ATTN_OK;
}

attn_status_t attn_bwd_bounded(const void* q, const void* k, const void* v, const void* out,
                               const float* lse, const void* dout, void* dq, void* dk, void* dv,
                               float* delta, int64_t B, int64_t H, int64_t S, int64_t D,
                               float scale, int causal, uint64_t wait_timeout_ns,
                               cudaStream_t stream) {
  return attn_bwd_ex(q, k, v, out, lse, dout, dq, dk, dv, delta, B, H, S, D, scale, causal,
                     ATTN_BF16, wait_timeout_ns, stream);
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* out,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       float* delta, int64_t B, int64_t H, int64_t S, int64_t D, float scale,
                       int causal, cudaStream_t stream) {
  return attn_bwd_bounded(q, k, v, out, lse, dout, dq, dk, dv, delta, B, H, S, D, scale, causal,
                          kDefaultWaitTimeoutNs, stream);
}

}  // extern "C"
