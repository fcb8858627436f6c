// sched_check.cpp — test-only host shim over the forward kernel's grid
// schedule (schedule.h), so that CPU tests can check the CTA -> work-unit map.
#include <cstdint>

#include "schedule.h"

extern "C" {

// Fills bh[x], u[x] for every CTA index x of a BH x n_units grid.
__attribute__((visibility("default"))) void sched_map(int BH, int n_units, int heads_per_group,
                                                      int tail_levels, int* bh, int* u) {
  const ea::UnitSchedule s{BH, n_units, heads_per_group, tail_levels};
  for (int x = 0; x < BH * n_units; ++x) ea::schedule_unit(s, x, bh + x, u + x);
}

// The host's choice; out = {heads_per_group, tail_levels}.
__attribute__((visibility("default"))) void sched_plan(int64_t BH, int64_t n_units, int64_t S,
                                                       int64_t D, int causal,
                                                       int64_t kv_group_bytes, int sms,
                                                       int* out) {
  const ea::UnitSchedule s = ea::plan_schedule(BH, n_units, S, D, causal != 0, kv_group_bytes, sms);
  out[0] = s.heads_per_group;
  out[1] = s.tail_levels;
}

// The staged entry point's chunk plan: out[c] = {first, count} for c < n;
// returns n.
__attribute__((visibility("default"))) int staged_plan(int64_t BH, int64_t in_bytes_per_slice,
                                                       int64_t target_bytes, int max_chunks,
                                                       int64_t* out) {
  const int n = ea::staged_chunk_count(BH, in_bytes_per_slice, target_bytes, max_chunks);
  for (int c = 0; c < n; ++c) ea::staged_chunk_range(BH, n, c, out + 2 * c, out + 2 * c + 1);
  return n;
}
}
