// Host-side consistency check of one layer call's plan, for debug runs
// (enabled per handle by MOE_CHECK_PLANS=1 in the environment at init).
// Plain C++ over plain arrays, with no CUDA dependency, so that it can be
// built and exercised without a GPU.
//
// What a plan must satisfy (the slot table of "llama.cpp + MoE expert cache",
// "The idea: cache the hot experts on the GPU", step 2: slot = -1 when not
// cached; per-layer slots under a fixed budget, "Longhaul MoE loading"):
//   1  every routed id in [0, E), distinct within a token;
//   2  every pair's slot in [0, S), or -1 for a miss computed without taking a
//      slot (the score policy's bypass);
//   3  every pair's stage in [0, n_stages);
//   4  every miss record: expert in [0, E), slot in [-1, S), evicted in
//      [-1, E), stage in [0, n_stages); at most min(E, T k) records;
//   5  the layer state after the call: slot_expert[s] in [-1, E), no expert in
//      two slots, expert_slot the inverse of slot_expert;
//   6  a pair of the last stage whose slot is not -1 finds its expert there;
//   7  a pair of an earlier stage names the slot its expert occupied in that
//      stage: the miss record of the expert with that stage, or, in stage 0,
//      a hit (the expert is still in that slot, or its record says so).
// Returns 0 when all hold, else the number of the first rule found broken.
#pragma once

#include <stdint.h>

#include <vector>

namespace moe {

inline int plan_check(int T, int k, int E, int S, int n_stages, int n_miss, const int32_t *ids,
                      const int32_t *gpu_slot, const int32_t *stage,
                      const int32_t *miss,  // n_miss records of 4 int32: expert, slot, evicted, stage
                      const int32_t *slot_expert, const int32_t *expert_slot) {
  const int P = T * k;
  if (n_stages < 1) return 3;
  for (int t = 0; t < T; ++t)
    for (int q = 0; q < k; ++q) {
      const int e = ids[t * k + q];
      if (e < 0 || e >= E) return 1;
      for (int q2 = 0; q2 < q; ++q2)
        if (ids[t * k + q2] == e) return 1;
    }
  for (int p = 0; p < P; ++p) {
    if (gpu_slot[p] < -1 || gpu_slot[p] >= S) return 2;
    if (stage[p] < 0 || stage[p] >= n_stages) return 3;
  }
  const int max_miss = E < P ? E : P;
  if (n_miss < 0 || n_miss > max_miss) return 4;
  for (int i = 0; i < n_miss; ++i) {
    const int32_t *m = miss + 4 * i;
    if (m[0] < 0 || m[0] >= E || m[1] < -1 || m[1] >= S || m[2] < -1 || m[2] >= E || m[3] < 0 ||
        m[3] >= n_stages)
      return 4;
  }
  std::vector<int> seen(E, -1);
  for (int s = 0; s < S; ++s) {
    const int e = slot_expert[s];
    if (e < -1 || e >= E) return 5;
    if (e >= 0) {
      if (seen[e] >= 0 || expert_slot[e] != s) return 5;
      seen[e] = s;
    }
  }
  for (int e = 0; e < E; ++e)
    if (expert_slot[e] != seen[e]) return 5;
  const int last = n_stages - 1;
  for (int p = 0; p < P; ++p) {
    const int e = ids[p], s = gpu_slot[p], st = stage[p];
    if (s < 0) continue;
    if (st == last) {
      if (slot_expert[s] != e) return 6;
      continue;
    }
    bool ok = false;
    for (int i = 0; i < n_miss && !ok; ++i) {
      const int32_t *m = miss + 4 * i;
      ok = m[0] == e && m[3] == st && m[1] == s;
    }
    if (!ok && st == 0) {
      // a hit of stage 0: no miss record of this expert in stage 0
      bool missed0 = false;
      for (int i = 0; i < n_miss; ++i) missed0 = missed0 || (miss[4 * i] == e && miss[4 * i + 3] == 0);
      ok = !missed0;
    }
    if (!ok) return 7;
  }
  return 0;
}

}  // namespace moe
