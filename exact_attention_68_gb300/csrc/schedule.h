// schedule.h — which work unit each CTA of the forward kernel's 1-D grid takes.
//
// A work unit is one (b·H + h) slice and one 128-row Q tile: unit level u is
// Q tile u.  Under the causal mask level u does u+1 K/V tile-steps (of 128
// keys), so the levels differ in cost and the order of the grid decides both
// the load balance and how often K/V tiles come back from DRAM:
//
//   phase 1  levels n_units-1 .. tail_levels, one group of heads_per_group
//            slices at a time; within a group the levels go heaviest first and
//            the slices of a level sit side by side.  One group's K/V is sized
//            to stay in L2, so the CTAs in flight re-read tiles from L2.
//   phase 2  levels tail_levels-1 .. 0 over all slices, heaviest first: the
//            light units that even out the finish times of the SMs.
//
// Host and device share this mapping; it is a bijection from
// [0, BH·n_units) onto (slice, level) pairs.
#pragma once

#include <cstdint>

#ifdef __CUDACC__
#define EA_HOST_DEVICE __host__ __device__ __forceinline__
#else
#define EA_HOST_DEVICE inline
#endif

namespace ea {

struct UnitSchedule {
  int BH;               // B·H slices
  int n_units;          // unit levels per slice
  int heads_per_group;  // slices per group in phase 1 (>= 1)
  int tail_levels;      // levels run in phase 2, 0 .. n_units
};

// CTA index x in [0, BH·n_units) -> slice *bh and unit level *u.
EA_HOST_DEVICE void schedule_unit(const UnitSchedule& s, int x, int* bh, int* u) {
  const int grouped_levels = s.n_units - s.tail_levels;
  const int phase1 = s.BH * grouped_levels;
  if (x < phase1) {
    const int per_group = s.heads_per_group * grouped_levels;
    const int group = x / per_group;
    const int g0 = group * s.heads_per_group;
    const int rest = s.BH - g0;
    const int g_size = s.heads_per_group < rest ? s.heads_per_group : rest;
    const int r = x - group * per_group;
    const int level_rev = r / g_size;
    *bh = g0 + (r - level_rev * g_size);
    *u = s.n_units - 1 - level_rev;
  } else {
    const int y = x - phase1;
    const int level_rev = y / s.BH;
    *bh = y - level_rev * s.BH;
    *u = s.tail_levels - 1 - level_rev;
  }
}

// K/V bytes of the (b, h) slices one phase-1 group spans: well under the
// 129 MB L2, so that the CTAs running at one time re-read K/V tiles from L2.
constexpr int64_t kL2GroupBytes = 48ll << 20;

// Host choice of the schedule.  kv_group_bytes: K/V bytes one group may span;
// sms: the device's SM count.  Phase 2 gets about sqrt(n_units·sms/(2·BH))
// levels, about a quarter of the heaviest unit's cost per SM: enough light
// units to even out the finish times phase 1 leaves.  Phase 2 walks the first
// tail_levels K/V tiles of every slice again after phase 1 evicted them, so a
// shorter tail reads less from DRAM (c5: twice this tail read 584 MB per
// launch, this one 442 MB, at the same speed).  Without the causal mask every
// unit costs the same and phase 2 is empty.
inline UnitSchedule plan_schedule(int64_t BH, int64_t n_units, int64_t S, int64_t D, bool causal,
                                  int64_t kv_group_bytes, int sms) {
  UnitSchedule s;
  s.BH = static_cast<int>(BH);
  s.n_units = static_cast<int>(n_units);
  const int64_t kv_bytes = S * D * 2 * 2;  // K and V of one slice, bf16
  int64_t g = kv_group_bytes / kv_bytes;
  if (g < 1) g = 1;
  if (g > BH) g = BH;
  s.heads_per_group = static_cast<int>(g);
  int64_t tail = 0;
  if (causal) {
    const int64_t want = n_units * (sms > 0 ? sms : 1) / 2;
    while (tail < n_units && tail * tail * BH < want) ++tail;
  }
  s.tail_levels = static_cast<int>(tail);
  return s;
}

// Host: how the staged (host-buffer) entry point splits the B·H slices into
// chunks whose host↔device copies and kernels overlap.  About `target_bytes`
// of inputs per chunk, at least one slice per chunk, at most `max_chunks`.
inline int staged_chunk_count(int64_t BH, int64_t in_bytes_per_slice, int64_t target_bytes,
                              int max_chunks) {
  int64_t n = (BH * in_bytes_per_slice + target_bytes - 1) / target_bytes;
  if (n > max_chunks) n = max_chunks;
  if (n > BH) n = BH;
  if (n < 1) n = 1;
  return static_cast<int>(n);
}

// Slices [*first, *first + *count) of chunk c of n (n <= BH).  The last
// chunk takes half an even share (at least one slice): its kernel and its
// download are the part of the call that no upload hides.  The other chunks
// share the rest evenly, the first ones taking one more.
inline void staged_chunk_range(int64_t BH, int n, int c, int64_t* first, int64_t* count) {
  if (n <= 1) {
    *first = 0;
    *count = BH;
    return;
  }
  int64_t last = BH / n / 2;
  if (last < 1) last = 1;
  const int64_t rest = BH - last;  // >= n - 1
  if (c == n - 1) {
    *first = rest;
    *count = last;
    return;
  }
  const int64_t base = rest / (n - 1), rem = rest % (n - 1);
  *count = base + (c < rem ? 1 : 0);
  *first = c * base + (c < rem ? c : rem);
}

}  // namespace ea
