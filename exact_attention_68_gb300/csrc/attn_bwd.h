// attn_bwd.h — parameters and launch entry of the attention backward kernels,
// shared by the host API and the kernel translation unit (no device code).
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda.h>
#include <cuda_runtime_api.h>

#include "schedule.h"

namespace ea {

// Both backward kernels: warps 0-7 elementwise (two groups of four warps, one
// per half of a tile's 128 columns), warp 8 tcgen05 issuer, warp 9 producer.
constexpr int kBwdThreads = 320;

struct BwdParams {
  CUtensorMap tm_q;   // q as (D, S, B·H), box 64 x 128 rows, 128-byte swizzle
  CUtensorMap tm_k;   // k, same box
  CUtensorMap tm_v;   // v, same box
  CUtensorMap tm_do;  // dout, same box
  CUtensorMap tm_dq;  // dq, box 64 x 32 rows (one warp's rows)
  CUtensorMap tm_dk;  // dk, same
  CUtensorMap tm_dv;  // dv, same
  // 256-column kernels only (head dimension above 128): boxes of 64 columns x
  // 64 rows, for the 64-key (K, V) and 64-query (Q, dout) steps
  CUtensorMap tm_q64;
  CUtensorMap tm_k64;
  CUtensorMap tm_v64;
  CUtensorMap tm_do64;
  const uint16_t* q;     // 16-bit [B·H, S, d_cols]: rows read into TMEM by the dq kernel
  const uint16_t* k;     // 16-bit [B·H, S, d_cols]: rows read into TMEM by the dk/dv kernel
  const uint16_t* v;     // 16-bit [B·H, S, d_cols]: rows read into TMEM by the dk/dv kernel
  const uint16_t* out;   // 16-bit [B·H, S, d_cols]: forward output (rows read for delta)
  const uint16_t* dout;  // 16-bit [B·H, S, d_cols]
  const float* lse;      // [B·H, S]: natural-log logsumexp saved by the forward
  float* delta;          // [B·H, S]: rowsum(dout ⊙ out), written by the dq kernel
  int* status;           // device status word pair (error bits, first wait site)
  int BH, S;
  int d_cols;            // the tensors' head dimension (<= the kernel's D, a multiple
                         // of 8); the kernel's columns past it are zero
  int n_t;               // ceil(S / 128): tiles along the sequence
  UnitSchedule sched;    // CTA index -> (b·H + h, unit level): the level of a Q tile i
                         // is i, of a K/V tile j is n_t - 1 - j (both cost level + 1
                         // tile-steps under the causal mask)
  float scale;           // softmax scale
  float scale_log2;      // scale · log2(e)
  uint64_t timeout_ns;
};

// Launches the dq kernel (which also writes delta) and then the dk/dv kernel
// on `stream`.  f16: the 16-bit tensors are fp16 (else bf16).
cudaError_t bwd_launch(const BwdParams& p, int D, bool causal, bool f16, cudaStream_t stream);

// The same for head dimensions above 128 (kernels 256 columns wide): the dq
// kernel, then the dk/dv kernel with one CTA per K/V tile and half of the
// head dimension.
cudaError_t bwd256_launch(const BwdParams& p, bool causal, bool f16, cudaStream_t stream);

}  // namespace ea
