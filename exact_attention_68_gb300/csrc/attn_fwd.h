// attn_fwd.h — kernel parameters and launch entry shared by the host API and
// the kernel translation unit (host-compilable, no device code).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "schedule.h"

namespace ea {

// Rows of one Q tile (the tcgen05 M).
constexpr int kBlockM = 128;

// The running max that serves as the exponent reference of a row is only
// moved when a tile's max exceeds it by more than this many log2 units.  The
// result is exact for any threshold (O and both sums share the reference);
// the threshold bounds every p = 2^(t - m) by 2^threshold.  P must hold that
// value: bf16 reaches 2^127, fp16 only 65504 < 2^16.  The fp32 sums then
// stay finite while n_keys·2^threshold·max|v| < 2^128, i.e. for |v| < 2^65
// at threshold 32 and any key count below 2^31.  Rounding is relative, so
// the reference's distance from the true max costs no precision; and the
// reference never exceeds the true max, so no p underflows earlier than with
// the exact max.  A high threshold makes moves (a redo of the tile's
// exponentials and a rescale of O in TMEM) rare even for peaked softmaxes.
template <bool F16>
constexpr float kRescaleThreshold = F16 ? 8.0f : 32.0f;

// Parameters of the forward kernels: one 128-row Q tile at a time, Q in TMEM,
// BN-row K/V tiles (BN = 64 at D = 256, else 128).
struct Fwd1QParams {
  CUtensorMap tm_k;    // k as (D, S, B·H), box 64 x BN rows, 128-byte swizzle
  CUtensorMap tm_v;    // v, same box
  CUtensorMap tm_o;    // out, box 64 x 32 rows
  CUtensorMap tm_q;    // q, box 64 x 128 rows: L2 prefetch of a Q tile (persistent kernel)
  const uint16_t* q;   // 16-bit [B·H, S, d_cols]: rows read into TMEM
  float* lse;          // [B·H, S]
  int* status;
  int BH, S;
  int d_cols;          // the tensors' head dimension (<= D, a multiple of 8); the
                       // kernel's columns past it are zero and never stored
  int n_qt;            // ceil(S / 128)
  int n_kt;            // ceil(S / BN)
  UnitSchedule sched;  // CTA index -> (b·H + h, Q tile): a unit is one Q tile here
  float scale_log2;
  uint64_t timeout_ns;
};

// One Q tile per CTA, Q in TMEM: D = 256 (64-row K/V tiles) and D = 128
// (128-row K/V tiles).  The library runs D = 256 on it.
cudaError_t fwd1q_launch(const Fwd1QParams& p, int D, bool causal, bool f16, cudaStream_t stream);

// The same computation with one CTA per SM walking Q tiles (D = 64 or 128):
// a running CTA takes over the Q tile of the next CTA of the grid that has not
// been launched yet, so the next tile's start overlaps this tile's end.
cudaError_t fwd1qp_launch(const Fwd1QParams& p, int D, bool causal, bool f16, cudaStream_t stream);

}  // namespace ea
