// Router top-k + per-layer LRU slot map + work lists, in one CTA per call.
//
// Router ("llama.cpp + MoE expert cache", "The idea: cache the hot experts on
// the GPU", step 1): one warp per token; top-k of the raw logits (descending,
// ties to the lower expert id) by k warp arg-max rounds; weights are softmax
// probabilities over all E (mode 0) or renormalised over the chosen k (mode 1).
//
// Slot map ("Longhaul MoE loading": per-layer LRU under a fixed budget; the
// batch's experts are protected from eviction; duplicates load once; more
// experts than slots -> stages): the state lives in device memory and is
// updated here; the plan (gpu_slot, stage, miss list, work items/units) goes to
// per-call scratch and, when the host must issue copies, to a mapped mailbox.
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {


// Exclusive scan over the 1024 threads of the block; returns the prefix and
// writes the total to *total.  `ws` is shared scratch of 33 ints.
__device__ int block_exclusive_scan(int v, int *ws, int *total) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  int incl = v;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    int n = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += n;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (warp == 0) {
    int wv = ws[lane];
    int wi = wv;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      int n = __shfl_up_sync(0xffffffffu, wi, o);
      if (lane >= o) wi += n;
    }
    ws[lane] = wi - wv;  // exclusive per warp
    if (lane == 31) ws[32] = wi;
  }
  __syncthreads();
  int r = ws[warp] + incl - v;
  *total = ws[32];
  __syncthreads();
  return r;
}

// Router for one token, VPL logits per lane (value e = i*32 + lane).
template <int VPL>
__device__ void route_token(const float *row, int E, int k, int weight_mode, int32_t *ids,
                            float *w, int *bad_flag) {
  const int lane = threadIdx.x & 31;
  float v[VPL];
  bool bad = false;
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    int e = i * 32 + lane;
    v[i] = -INFINITY;
    if (e < E) {
      float x = row[e];
      if (!isfinite(x)) bad = true;
      v[i] = x;
      m = fmaxf(m, x);
    }
  }
  if (__any_sync(0xffffffffu, bad)) {
    if (lane == 0) atomicExch(bad_flag, 1);
    return;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  float z = 0.f;
#pragma unroll
  for (int i = 0; i < VPL; ++i)
    if (i * 32 + lane < E) z += expf(v[i] - m);
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) z += __shfl_xor_sync(0xffffffffu, z, o);

  uint32_t taken = 0;
  float psum = 0.f;
  for (int q = 0; q < k; ++q) {
    float bv = -INFINITY;
    int bi = 0x7fffffff;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
      int e = i * 32 + lane;
      if (e < E && !((taken >> i) & 1u)) {
        if (v[i] > bv || (v[i] == bv && e < bi)) { bv = v[i]; bi = e; }
      }
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) {
      float ov = __shfl_xor_sync(0xffffffffu, bv, o);
      int oi = __shfl_xor_sync(0xffffffffu, bi, o);
      if (ov > bv || (ov == bv && oi < bi)) { bv = ov; bi = oi; }
    }
    if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
    if (lane == 0) {
      float p = expf(bv - m) / z;
      ids[q] = bi;
      w[q] = p;
      psum += p;
    }
  }
  if (weight_mode == 1 && lane == 0)
    for (int q = 0; q < k; ++q) w[q] = w[q] / psum;
}

template <int VPL>
__device__ void route_all(const PlanArgs &a, int *bad_flag) {
  const int warp = threadIdx.x >> 5;
  for (int t = warp; t < a.T; t += kPlanThreads / 32)
    route_token<VPL>(a.logits + (size_t)t * a.E, a.E, a.k, a.weight_mode, a.ids + (size_t)t * a.k,
                     a.w + (size_t)t * a.k, bad_flag);
}

struct SmemPlan {
  int *cnt, *hit_rank, *miss_rank, *e_slot, *e_stage, *M, *new_es, *item_pairs, *item_units;
  int *se0, *cand, *victim, *occ0, *fin, *touched;
  unsigned long long *stamp0;
  int *wcnt;  // [32][E]
  int *ws;    // scan scratch [33]
  int *scal;  // scalars
};

__global__ void __launch_bounds__(kPlanThreads, 1) plan_kernel(PlanArgs a) {
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int E = a.E, S = a.S, k = a.k, T = a.T;
  const int P = T * k;
  const int tid = threadIdx.x;
  const int lane = tid & 31, warp = tid >> 5;

  SmemPlan s;
  {
    unsigned char *p = smem_raw;
    auto take_u64 = [&](int n) { unsigned long long *r = (unsigned long long *)p; p += 8 * (size_t)n; return r; };
    auto take = [&](int n) { int *r = (int *)p; p += 4 * (size_t)((n + 3) / 4 * 4); return r; };
    s.stamp0 = take_u64(S);
    s.cnt = take(E); s.hit_rank = take(E); s.miss_rank = take(E); s.e_slot = take(E);
    s.e_stage = take(E); s.M = take(E); s.new_es = take(E); s.item_pairs = take(E + 1);
    s.item_units = take(E + 1);
    s.se0 = take(S); s.cand = take(S); s.victim = take(S); s.occ0 = take(S); s.fin = take(S);
    s.touched = take(S);
    s.wcnt = take(32 * E);
    s.ws = take(36);
    s.scal = take(16);
  }
  int *bad = &s.scal[0];
  if (tid == 0) bad[0] = 0;
  __syncthreads();

  // ---- 1. router
  const int vpl = (E + 31) / 32;
  if (vpl <= 1) route_all<1>(a, bad);
  else if (vpl <= 2) route_all<2>(a, bad);
  else if (vpl <= 4) route_all<4>(a, bad);
  else if (vpl <= 8) route_all<8>(a, bad);
  else if (vpl <= 16) route_all<16>(a, bad);
  else route_all<32>(a, bad);
  __syncthreads();
  if (bad[0]) {
    if (tid == 0) {
      PlanHdr h = {};
      h.error = 1;
      *a.hdr = h;
      atomicExch(a.err_flag, 1);
      __threadfence_system();
      if (a.mailbox) {
        a.mailbox->hdr = h;
        __threadfence_system();
        a.mailbox->seq = a.seq;
        __threadfence_system();
      }
    }
    return;
  }

  // ---- 2. distinct experts, hits and misses (ascending expert order)
  for (int e = tid; e < E; e += kPlanThreads) s.cnt[e] = 0;
  for (int i = tid; i < S; i += kPlanThreads) {
    s.se0[i] = a.slot_expert[i];
    s.stamp0[i] = a.slot_stamp[i];
    s.touched[i] = 0;
  }
  __syncthreads();
  for (int p = tid; p < P; p += kPlanThreads) atomicAdd(&s.cnt[a.ids[p]], 1);
  __syncthreads();

  int is_hit = 0, is_miss = 0, e_old_slot = -1;
  if (tid < E) {
    e_old_slot = a.expert_slot[tid];
    const bool used = s.cnt[tid] > 0;
    is_hit = used && e_old_slot >= 0;
    is_miss = used && e_old_slot < 0;
  }
  int nH, nM;
  int hr = block_exclusive_scan(is_hit, s.ws, &nH);
  int mr = block_exclusive_scan(is_miss, s.ws, &nM);
  const int nU = nH + nM;
  int ph = block_exclusive_scan(is_hit ? s.cnt[tid] : 0, s.ws, &s.scal[1]);
  (void)ph;
  const int pick_hits = s.scal[1];
  if (tid < E) {
    s.hit_rank[tid] = is_hit ? hr : -1;
    s.miss_rank[tid] = is_miss ? mr : -1;
    s.e_slot[tid] = -1;
    s.e_stage[tid] = -1;
    if (is_miss) s.M[mr] = tid;
    if (is_hit) { s.e_slot[tid] = e_old_slot; s.e_stage[tid] = 0; s.touched[e_old_slot] = 1; }
  }

  // ---- 3. stage-0 victims: empty slots (by index), then slots whose expert the
  // call does not pick, by (stamp, index)
  for (int i = tid; i < S; i += kPlanThreads) {
    int e = s.se0[i];
    s.cand[i] = (e < 0) || (s.cnt[e] == 0);
  }
  __syncthreads();
  for (int i = tid; i < S; i += kPlanThreads) {
    if (!s.cand[i]) continue;
    const int ci = s.se0[i] < 0 ? 0 : 1;
    const unsigned long long ti = ci ? s.stamp0[i] : 0ull;
    int rank = 0;
    for (int j = 0; j < S; ++j) {
      if (!s.cand[j] || j == i) continue;
      const int cj = s.se0[j] < 0 ? 0 : 1;
      const unsigned long long tj = cj ? s.stamp0[j] : 0ull;
      const bool before = (cj < ci) || (cj == ci && (tj < ti || (tj == ti && j < i)));
      rank += before;
    }
    s.victim[rank] = i;
  }
  const int n0 = (nU <= S) ? nM : (S - nH);
  for (int i = tid; i < S; i += kPlanThreads) s.occ0[i] = s.se0[i];
  __syncthreads();
  for (int i = tid; i < n0; i += kPlanThreads) {
    s.occ0[s.victim[i]] = s.M[i];
    s.touched[s.victim[i]] = 1;
  }
  __syncthreads();

  // ---- 4. miss assignment (stage 0 closed over victims; later stages reuse
  // slots in ascending index, all slots then carrying this call's stamp)
  int *n_evict = &s.scal[2];
  if (tid == 0) *n_evict = 0;
  __syncthreads();
  for (int i = tid; i < nM; i += kPlanThreads) {
    const int e = s.M[i];
    int slot, stg, ev;
    if (i < n0) {
      slot = s.victim[i];
      stg = 0;
      ev = s.se0[slot];
    } else {
      const int r = i - n0;
      stg = 1 + r / S;
      slot = r % S;
      ev = (stg == 1) ? s.occ0[slot] : s.M[i - S];
    }
    s.e_slot[e] = slot;
    s.e_stage[e] = stg;
    if (ev >= 0) atomicAdd(n_evict, 1);
    a.miss[i] = MissItem{e, slot, ev, stg};
  }
  const int n_later = nM - n0;
  const int n_stages = n_later > 0 ? 1 + (n_later + S - 1) / S : 1;
  __syncthreads();

  // ---- 5. new state
  const unsigned long long now = *a.clock + 1ull;
  for (int i = tid; i < S; i += kPlanThreads) {
    int f = s.occ0[i];
    if (n_later > i) {
      const int last = n0 + i + S * ((n_later - 1 - i) / S);
      f = s.M[last];
    }
    s.fin[i] = f;
    const bool t = s.touched[i] || n_later > 0;
    a.slot_expert[i] = f;
    if (t) a.slot_stamp[i] = now;
  }
  for (int e = tid; e < E; e += kPlanThreads) s.new_es[e] = -1;
  __syncthreads();
  for (int i = tid; i < S; i += kPlanThreads)
    if (s.fin[i] >= 0) s.new_es[s.fin[i]] = i;
  __syncthreads();
  for (int e = tid; e < E; e += kPlanThreads) a.expert_slot[e] = s.new_es[e];

  // ---- 6. per-pair slot and stage
  for (int p = tid; p < P; p += kPlanThreads) {
    const int e = a.ids[p];
    a.gpu_slot[p] = s.e_slot[e];
    a.stage[p] = s.e_stage[e];
  }

  // ---- 7. work items (hits ascending, then misses ascending) and units
  int item = -1;
  if (tid < E) {
    if (is_hit) item = hr;
    else if (is_miss) item = nH + mr;
  }
  int n_pairs_tot, n_units_tot;
  const int my_pairs = item >= 0 ? s.cnt[tid] : 0;
  const int my_units = item >= 0 ? (my_pairs + kTokPerUnit - 1) / kTokPerUnit : 0;
  // prefix over item order: scatter counts by item index, then scan by item
  if (tid < E && item >= 0) { s.item_pairs[item] = my_pairs; s.item_units[item] = my_units; }
  __syncthreads();
  const int vp = tid < nU ? s.item_pairs[tid] : 0;
  const int vu = tid < nU ? s.item_units[tid] : 0;
  const int pb = block_exclusive_scan(vp, s.ws, &n_pairs_tot);
  const int ub = block_exclusive_scan(vu, s.ws, &n_units_tot);
  if (tid < nU) { s.item_pairs[tid] = pb; s.item_units[tid] = ub; }
  if (tid == 0) { s.item_pairs[nU] = n_pairs_tot; s.item_units[nU] = n_units_tot; }
  __syncthreads();
  if (tid < E && item >= 0) {
    WorkItem it;
    it.expert = tid;
    it.slot = s.e_slot[tid];
    it.stage = s.e_stage[tid];
    it.is_miss = is_miss;
    it.pair_begin = s.item_pairs[item];
    it.pair_count = my_pairs;
    a.items[item] = it;
    const int u0 = s.item_units[item];
    for (int j = 0; j < my_units; ++j) {
      WorkUnit u;
      u.item = item;
      u.pair_begin = it.pair_begin + j * kTokPerUnit;
      u.pair_count = min(kTokPerUnit, my_pairs - j * kTokPerUnit);
      u.stage = it.stage;
      a.units[u0 + j] = u;
    }
  }
  // stage unit ranges: stage 0 = items [0, nH + n0); stage j>=1 = next S misses
  int hit_units = s.item_units[nH];
  for (int j = tid; j <= n_stages; j += kPlanThreads) {
    const int first_item = (j == 0) ? 0 : min(nU, nH + n0 + (j - 1) * S);
    a.unit_begin[j] = s.item_units[first_item];
  }

  // ---- 8. perm: pairs grouped by item, ascending pair index inside an item
  // (stable counting sort; warp w owns a contiguous chunk of pairs)
  const int chunk = (P + 31) / 32;
  const int c0 = warp * chunk, c1 = min(P, c0 + chunk);
  for (int i = tid; i < 32 * E; i += kPlanThreads) s.wcnt[i] = 0;
  __syncthreads();
  for (int base = c0; base < c1; base += 32) {
    const int p = base + lane;
    const bool act = p < c1;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int e = a.ids[p];
      const unsigned m = __match_any_sync(am, e);
      if ((__ffs(m) - 1) == lane) s.wcnt[warp * E + e] += __popc(m);
    }
    __syncwarp();
  }
  __syncthreads();
  for (int e = tid; e < E; e += kPlanThreads) {
    if (s.cnt[e] == 0) continue;
    const int it = s.hit_rank[e] >= 0 ? s.hit_rank[e] : nH + s.miss_rank[e];
    int run = s.item_pairs[it];
    for (int w2 = 0; w2 < 32; ++w2) {
      const int c = s.wcnt[w2 * E + e];
      s.wcnt[w2 * E + e] = run;
      run += c;
    }
  }
  __syncthreads();
  for (int base = c0; base < c1; base += 32) {
    const int p = base + lane;
    const bool act = p < c1;
    const unsigned am = __ballot_sync(0xffffffffu, act);
    if (act) {
      const int e = a.ids[p];
      const unsigned m = __match_any_sync(am, e);
      const int rank = __popc(m & ((1u << lane) - 1u));
      a.perm[s.wcnt[warp * E + e] + rank] = p;
      __syncwarp(m);
      if ((__ffs(m) - 1) == lane) s.wcnt[warp * E + e] += __popc(m);
    }
    __syncwarp();
  }
  __syncthreads();

  // ---- 9. header, stats, clock, mailbox
  if (tid == 0) {
    PlanHdr h = {};
    h.error = 0;
    h.n_unique = nU;
    h.n_hits = nH;
    h.n_miss = nM;
    h.n_stage0_miss = n0;
    h.n_stages = n_stages;
    h.n_units = n_units_tot;
    h.n_evict = *n_evict;
    h.pick_hits = pick_hits;
    h.pick_misses = P - pick_hits;
    h.hit_units = hit_units;
    *a.hdr = h;
    *a.clock = now;
    uint64_t *st = a.stats;
    st[0] += 1;
    st[1] += (uint64_t)pick_hits;
    st[2] += (uint64_t)(P - pick_hits);
    st[3] += (uint64_t)nH;
    st[4] += (uint64_t)nM;
    st[5] += (uint64_t)*n_evict;
    st[6] += (uint64_t)nM * a.expert_bytes;
    st[7] += (uint64_t)n_stages;
    st[8] += n_stages > 1 ? 1ull : 0ull;
    if (a.mailbox) a.mailbox->hdr = h;
  }
  if (a.mailbox) {
    int32_t *mub = reinterpret_cast<int32_t *>(a.mailbox + 1);
    MissItem *mm = reinterpret_cast<MissItem *>(mub + a.mailbox_stage_cap);
    for (int j = tid; j <= n_stages; j += kPlanThreads) {
      const int first_item = (j == 0) ? 0 : min(nU, nH + n0 + (j - 1) * S);
      mub[j] = s.item_units[first_item];
    }
    for (int i = tid; i < nM; i += kPlanThreads) mm[i] = a.miss[i];
    __threadfence_system();
    __syncthreads();
    if (tid == 0) {
      __threadfence_system();
      a.mailbox->seq = a.seq;
      __threadfence_system();
    }
  }
}

}  // namespace

size_t plan_smem_bytes(int E, int S) {
  auto r4 = [](size_t n) { return 4 * ((n + 3) / 4 * 4); };
  size_t b = 8 * (size_t)S;
  b += 7 * r4(E) + 2 * r4(E + 1);
  b += 6 * r4(S);
  b += r4(32 * (size_t)E) + r4(36) + r4(16);
  return b + 64;
}

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t st) {
  const size_t smem = plan_smem_bytes(a.E, a.S);
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(plan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  plan_kernel<<<1, kPlanThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
