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
//
// Stage-0 victims are ranked by (empty first, stamp, slot index); later stages
// reuse all slots in ascending index (after stage 0 every slot holds an expert
// of the call, all carrying the call's stamp).  Two other replacement policies:
// the decayed usage score with admission ("llama.cpp + MoE expert cache",
// "Keeping the cache fresh"; single-stage calls, plan_small_kernel<1>), and
// adopt ("llama.cpp: fork with multi gpu acceleration ...", "Prefill preheat";
// plan_kernel): a staged call takes its misses lowest rank first and streams
// its later stages through the C slots that do not hold its highest-ranked
// stage-0 experts, so that it ends holding its most-used experts.
#include <math.h>

#include "common.cuh"

namespace moe {
namespace {

__device__ __forceinline__ uint32_t smem_addr(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

constexpr int NT = kPlanThreads;
constexpr int NW = NT / 32;

// In-place exclusive scan of a[0..n) held in shared memory; returns the total.
// ws: shared scratch of NW + 1 elements.  Every thread of the block calls it.
template <typename V>
__device__ V block_scan_array(V *a, int n, V *ws) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int per = (n + NT - 1) / NT;
  const int i0 = min(n, tid * per), i1 = min(n, i0 + per);
  V local = 0;
  for (int i = i0; i < i1; ++i) local += a[i];
  V incl = local;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const V v = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += v;
  }
  if (lane == 31) ws[warp] = incl;
  __syncthreads();
  if (tid == 0) {
    V run = 0;
    for (int w = 0; w < NW; ++w) { const V t = ws[w]; ws[w] = run; run += t; }
    ws[NW] = run;
  }
  __syncthreads();
  V run = ws[warp] + incl - local;
  for (int i = i0; i < i1; ++i) { const V t = a[i]; a[i] = run; run += t; }
  const V total = ws[NW];
  __syncthreads();
  return total;
}

// One token's logits, VPL per lane (value e = i*32 + lane; -inf past E).
template <int VPL>
__device__ __forceinline__ void load_logits(const float *row, int E, float v[VPL]) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int i = 0; i < VPL; ++i) v[i] = (i * 32 + lane < E) ? row[i * 32 + lane] : -INFINITY;
}

// Router for one token from its loaded logits (s_ids: an optional copy of the
// ids in shared memory).
template <int VPL>
__device__ void route_values(const float v[VPL], int E, int k, int weight_mode, int32_t *ids, float *w,
                             int *bad_flag, int32_t *s_ids = nullptr) {
  const int lane = threadIdx.x & 31;
  bool bad = false;
  float m = -INFINITY;
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    if (i * 32 + lane < E) {
      if (!isfinite(v[i])) bad = true;
      m = fmaxf(m, v[i]);
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

  // k rounds: the largest remaining value, ties to the lower id.  A value's
  // key orders like the float (-0 taken as +0); one warp max over keys, then
  // one warp min over the ids holding that key.
  uint32_t key[VPL];
#pragma unroll
  for (int i = 0; i < VPL; ++i) {
    const uint32_t b = __float_as_uint(v[i] == 0.f ? 0.f : v[i]);
    key[i] = (i * 32 + lane < E) ? ((b & 0x80000000u) ? ~b : (b | 0x80000000u)) : 0u;
  }
  uint32_t taken = 0, my_key = 0;
  int my_id = -1;
  for (int q = 0; q < k; ++q) {
    uint32_t bk = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (i * 32 + lane < E && !((taken >> i) & 1u) && key[i] > bk) bk = key[i];
    const uint32_t mk = __reduce_max_sync(0xffffffffu, bk);
    uint32_t bi = 0xffffffffu;
#pragma unroll
    for (int i = 0; i < VPL; ++i)
      if (i * 32 + lane < E && !((taken >> i) & 1u) && key[i] == mk && (uint32_t)(i * 32 + lane) < bi)
        bi = (uint32_t)(i * 32 + lane);
    const int id = (int)__reduce_min_sync(0xffffffffu, bi);
    if ((id & 31) == lane) taken |= 1u << (id >> 5);
    if (lane == q) { my_key = mk; my_id = id; }
  }
  // pick q's probability on lane q, all k at once: its value is its key
  // mapped back (-0 came out as +0, which has the same exponential)
  float my_p = 0.f;
  if (lane < k) {
    const uint32_t kb = (my_key & 0x80000000u) ? (my_key & 0x7fffffffu) : ~my_key;
    my_p = expf(__uint_as_float(kb) - m) / z;
  }
  float sum = lane < k ? my_p : 0.f;
  if (weight_mode == 1)  // the sum over the picks renormalises (mode 1 only)
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) sum += __shfl_xor_sync(0xffffffffu, sum, o);
  if (lane < k) {
    ids[lane] = my_id;
    if (s_ids) s_ids[lane] = my_id;
    w[lane] = weight_mode == 1 ? my_p / sum : my_p;
  }
}

// Router for one token, VPL logits per lane.
template <int VPL>
__device__ void route_token(const float *row, int E, int k, int weight_mode, int32_t *ids,
                            float *w, int *bad_flag, int32_t *s_ids = nullptr) {
  float v[VPL];
  load_logits<VPL>(row, E, v);
  route_values<VPL>(v, E, k, weight_mode, ids, w, bad_flag, s_ids);
}

// Routing of a large call as its own grid: one warp per token; a non-finite
// logit sets *bad (read and cleared by plan_kernel).
template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float *logits, int T, int E, int k, int weight_mode,
                                                  int32_t *ids, float *w, int *bad) {
  const int t = blockIdx.x * 8 + (threadIdx.x >> 5);
  if (t >= T) return;
  route_token<VPL>(logits + (size_t)t * E, E, k, weight_mode, ids + (size_t)t * k, w + (size_t)t * k, bad);
}

template <int VPL>
__device__ void route_all(const PlanArgs &a, int *bad_flag) {
  const int warp = threadIdx.x >> 5;
  for (int t = warp; t < a.T; t += NW)
    route_token<VPL>(a.logits + (size_t)t * a.E, a.E, a.k, a.weight_mode, a.ids + (size_t)t * a.k,
                     a.w + (size_t)t * a.k, bad_flag);
}

__device__ void write_error(const PlanArgs &a) {
  if (threadIdx.x != 0) return;
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

// Miss i of the call: stage 0 into its victim; after that C misses per stage,
// the r-th later miss into later-stage slot qslot[r % C].
__device__ __forceinline__ MissItem miss_record(int i, int n0, int C, const int *M,
                                                const int *victim, const int *qslot,
                                                const int *se0, const int *occ0) {
  MissItem m;
  m.expert = M[i];
  if (i < n0) {
    m.slot = victim[i];
    m.stage = 0;
    m.evicted = se0[m.slot];
  } else {
    const int r = i - n0;
    m.stage = 1 + r / C;
    m.slot = qslot[r % C];
    m.evicted = (m.stage == 1) ? occ0[m.slot] : M[i - C];
  }
  return m;
}

__global__ void __launch_bounds__(NT, 1) plan_kernel(PlanArgs a) {
  // launched in stream order (the caller's inputs are complete): a dependent
  // launched programmatically may start its plan-independent prologue now
  asm volatile("griddepcontrol.launch_dependents;");
  extern __shared__ __align__(16) unsigned char smem_raw[];
  const int E = a.E, S = a.S, k = a.k, T = a.T;
  const int P = T * k;
  const int tid = threadIdx.x, lane = tid & 31;

  // ---- shared memory carve-up (sizes mirrored in plan_smem_bytes)
  unsigned char *sp = smem_raw;
  auto take64 = [&](int n) { long long *r = (long long *)sp; sp += 8 * (size_t)((n + 1) / 2 * 2); return r; };
  auto take = [&](int n) { int *r = (int *)sp; sp += 4 * (size_t)((n + 3) / 4 * 4); return r; };
  unsigned long long *stamp0 = (unsigned long long *)take64(S);
  long long *itm = take64(E + 1);  // per item: pairs | units << 32, then its exclusive scan
  long long *ws64 = take64(NW + 2);
  int *cnt = take(E), *es0 = take(E), *code = take(E), *e_slot = take(E), *e_stage = take(E);
  int *M = take(E), *new_es = take(E), *item_of = take(E), *gitm = take(E + 1);
  int *se0 = take(S), *vpos = take(S), *occ0 = take(S), *touched = take(S), *victim = take(S);
  int *qpos = take(S), *qslot = take(S);  // later-stage slots: position of a slot, slot of a position
  int *vclass = take(S);  // stage-0 victim class of a slot: -1 not a victim, 0 empty, 1 evictable
  int *ws = take(NW + 2);
  int *scal = take(8);  // 0 bad, 1 pick hits, 2 evictions

  // ---- A. prefetch state, reset counters, route
  for (int i = tid; i < S; i += NT) {
    se0[i] = a.slot_expert[i];
    stamp0[i] = a.slot_stamp[i];
    touched[i] = 0;
  }
  for (int e = tid; e < E; e += NT) {
    es0[e] = a.expert_slot[e];
    cnt[e] = 0;
    new_es[e] = -1;
    e_slot[e] = -1;
    e_stage[e] = -1;
  }
  for (int i = tid; i < a.sync_n; i += NT) a.sync[i] = 0;
  if (tid < 8) scal[tid] = 0;
  const unsigned long long now = *a.clock + 1ull;
  const uint32_t epoch = *a.epoch + 1u;
  __syncthreads();
  if (a.routed) {
    // ids and weights come from route_kernel (earlier on the stream)
    if (tid == 0) {
      scal[0] = *a.route_bad;
      *a.route_bad = 0;
    }
  } else {
    int *bad = &scal[0];
    if (E <= 128) route_all<4>(a, bad);
    else if (E <= 256) route_all<8>(a, bad);
    else route_all<32>(a, bad);
  }
  __syncthreads();
  if (scal[0]) {
    write_error(a);
    return;
  }

  // ---- B. picks per expert
  for (int p = tid; p < P; p += NT) atomicAdd(&cnt[a.ids[p]], 1);
  __syncthreads();

  // ---- C. hit / miss flags (packed, one scan), pick hits
  int my_pick_hits = 0;
  for (int e = tid; e < E; e += NT) {
    const bool used = cnt[e] > 0;
    const bool hit = used && es0[e] >= 0;
    const bool miss = used && es0[e] < 0;
    code[e] = (hit ? 1 : 0) | (miss ? 1 << 16 : 0);
    if (hit) my_pick_hits += cnt[e];
    if (used) a.usage[e] += (uint32_t)cnt[e];
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my_pick_hits += __shfl_xor_sync(0xffffffffu, my_pick_hits, o);
  if (lane == 0 && my_pick_hits) atomicAdd(&scal[1], my_pick_hits);
  __syncthreads();
  const int tot = block_scan_array<int>(code, E, ws);
  const int nH = tot & 0xFFFF, nM = tot >> 16, nU = nH + nM;
  const int n0 = (nU <= S) ? nM : (S - nH);
  const int n_later = nM - n0;
  // adopt (policy 2), a call of more than one stage: misses lowest rank first
  // (rank: picks in this call descending, then expert id ascending), and the
  // later stages stream through C slots, as many stages as LRU takes
  const bool adopt = a.policy == 2 && n_later > 0;
  const int G = (n_later + S - 1) / S;
  const int C = adopt ? (n_later + G - 1) / G : S;
  const int n_stages = n_later > 0 ? 1 + (n_later + C - 1) / C : 1;

  // ---- D. hits keep their slot; misses in ascending order (adopt: lowest
  // rank first); stage-0 victim ranks: empty slots (by index) first, then
  // slots whose expert the call does not pick, by (stamp, index)
  for (int e = tid; e < E; e += NT) {
    if (cnt[e] == 0) { item_of[e] = -1; continue; }
    const int s0 = es0[e];
    if (s0 >= 0) {
      e_slot[e] = s0;
      e_stage[e] = 0;
      touched[s0] = 1;
      item_of[e] = code[e] & 0xFFFF;
    } else {
      int mr = code[e] >> 16;
      if (adopt) {
        mr = 0;
        for (int f = 0; f < E; ++f)
          mr += cnt[f] > 0 && es0[f] < 0 && (cnt[f] < cnt[e] || (cnt[f] == cnt[e] && f > e));
      }
      M[mr] = e;
      item_of[e] = nH + mr;
    }
  }
  for (int i = tid; i < S; i += NT) {
    const int ei = se0[i];
    vclass[i] = ei < 0 ? 0 : (cnt[ei] == 0 ? 1 : -1);
  }
  __syncthreads();
  for (int i = tid; i < S; i += NT) {
    const int cli = vclass[i];
    int rank = -1;
    if (cli >= 0) {
      rank = 0;
      const unsigned long long ti = cli ? stamp0[i] : 0ull;
      for (int j = 0; j < S; ++j) {
        const int clj = vclass[j];
        if (clj < 0 || j == i) continue;
        const unsigned long long tj = clj ? stamp0[j] : 0ull;
        rank += (clj < cli) || (clj == cli && (tj < ti || (tj == ti && j < i)));
      }
      victim[rank] = i;
    }
    vpos[i] = rank;
  }
  __syncthreads();

  // ---- E. slot contents after stage 0
  for (int i = tid; i < S; i += NT) {
    const int r = vpos[i];
    const bool v0 = r >= 0 && r < n0;
    occ0[i] = v0 ? M[r] : se0[i];
    if (v0) touched[i] = 1;
  }
  __syncthreads();

  // ---- E2. slots of the later stages: LRU all S, slot i at position i; adopt
  // keeps the S - C slots whose stage-0 expert ranks highest (after stage 0
  // every slot holds an expert of the call), the others in ascending index
  if (adopt) {
    for (int i = tid; i < S; i += NT) {
      const int ei = occ0[i];
      int above = ei < 0 ? S : 0;  // (an empty slot cannot occur here; it would rank last)
      for (int j2 = 0; j2 < S && ei >= 0; ++j2) {
        const int ej = occ0[j2];
        above += ej >= 0 && (cnt[ej] > cnt[ei] || (cnt[ej] == cnt[ei] && ej < ei));
      }
      vpos[i] = above < S - C ? 1 : 0;  // kept (vpos is free after E)
    }
    __syncthreads();
    for (int i = tid; i < S; i += NT) {
      int q = -1;
      if (!vpos[i]) {
        q = 0;
        for (int j2 = 0; j2 < i; ++j2) q += vpos[j2] ? 0 : 1;
        qslot[q] = i;
      }
      qpos[i] = q;
    }
  } else {
    for (int i = tid; i < S; i += NT) {
      qpos[i] = i;
      qslot[i] = i;
    }
  }
  __syncthreads();

  // ---- F. miss list, final slot contents and stamps
  int my_evict = 0;
  for (int i = tid; i < nM; i += NT) {
    const MissItem m = miss_record(i, n0, C, M, victim, qslot, se0, occ0);
    e_slot[m.expert] = m.slot;
    e_stage[m.expert] = m.stage;
    my_evict += m.evicted >= 0;
    a.miss[i] = m;
  }
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) my_evict += __shfl_xor_sync(0xffffffffu, my_evict, o);
  if (lane == 0 && my_evict) atomicAdd(&scal[2], my_evict);
  for (int i = tid; i < S; i += NT) {
    int f = occ0[i];
    const int q = qpos[i];
    if (q >= 0 && n_later > q) f = M[n0 + q + C * ((n_later - 1 - q) / C)];
    a.slot_expert[i] = f;
    if (touched[i] || n_later > 0) a.slot_stamp[i] = now;
    if (f >= 0) new_es[f] = i;
  }
  __syncthreads();

  // ---- G. per-pair slot/stage, new expert->slot table, item sizes
  for (int e = tid; e < E; e += NT) a.expert_slot[e] = new_es[e];
  // the pairs' ids loaded four at a time before their stores, so the loads
  // are in flight together
  for (int p0 = tid; p0 < P; p0 += 4 * NT) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) ev[u] = p0 + u * NT < P ? a.ids[p0 + u * NT] : 0;
#pragma unroll
    for (int u = 0; u < 4; ++u) {
      if (p0 + u * NT < P) {
        a.gpu_slot[p0 + u * NT] = e_slot[ev[u]];
        a.stage[p0 + u * NT] = e_stage[ev[u]];
      }
    }
  }
  for (int e = tid; e < E; e += NT) {
    const int it = item_of[e];
    if (it < 0) continue;
    const long long units = (cnt[e] + kTokPerUnit - 1) / kTokPerUnit;
    itm[it] = (long long)cnt[e] | (units << 32);
  }
  __syncthreads();
  for (int e = tid; e < E; e += NT) {
    const int it = item_of[e];
    if (it >= 0) gitm[it] = (cnt[e] + kGemmN - 1) / kGemmN;
  }
  const long long tot_iu = block_scan_array<long long>(itm, nU, ws64);
  const int n_units = (int)(tot_iu >> 32);
  if (tid == 0) itm[nU] = tot_iu;
  const int n_gunits = block_scan_array<int>(gitm, nU, ws);
  if (tid == 0) gitm[nU] = n_gunits;
  __syncthreads();

  // ---- H. items, units, stage ranges; perm = the pairs grouped by item
  for (int e = tid; e < E; e += NT) {
    const int it = item_of[e];
    if (it < 0) continue;
    WorkItem w;
    w.expert = e;
    w.slot = e_slot[e];
    w.stage = e_stage[e];
    w.is_miss = es0[e] < 0;
    w.pair_begin = (int)(itm[it] & 0xFFFFFFFFll);
    w.pair_count = cnt[e];
    a.items[it] = w;
    const int u0 = (int)(itm[it] >> 32);
    const int nun = (cnt[e] + kTokPerUnit - 1) / kTokPerUnit;
    for (int j = 0; j < nun; ++j) {
      WorkUnit u;
      u.item = it;
      u.pair_begin = w.pair_begin + j * kTokPerUnit;
      u.pair_count = min(kTokPerUnit, cnt[e] - j * kTokPerUnit);
      u.stage = w.stage;
      a.units[u0 + j] = u;
    }
    const int g0 = gitm[it], ngu = (cnt[e] + kGemmN - 1) / kGemmN;
    for (int j = 0; j < ngu; ++j) {
      WorkUnit u;
      u.item = it;
      u.pair_begin = w.pair_begin + j * kGemmN;
      u.pair_count = min(kGemmN, cnt[e] - j * kGemmN);
      u.stage = w.stage;
      a.gunits[g0 + j] = u;
    }
  }
  for (int j = tid; j <= n_stages; j += NT) {
    const int first_item = (j == 0) ? 0 : min(nU, nH + n0 + (j - 1) * C);
    a.unit_begin[j] = (int)(itm[first_item] >> 32);
    a.gunit_begin[j] = gitm[first_item];
  }
  const int hit_units = (int)(itm[nH] >> 32);
  const int hit_gunits = gitm[nH];

  // perm: each item's pairs in its range [pair_begin, pair_begin + count), in
  // an unspecified order (shared-memory counters): a pair's arithmetic does
  // not depend on its position among its item's pairs, so no stable sort is
  // needed (the outputs are the same bits in any order)
  for (int e = tid; e < E; e += NT) {
    const int it = item_of[e];
    if (it >= 0) cnt[e] = (int)(itm[it] & 0xFFFFFFFFll);  // cnt is free after H: the fill position
  }
  __syncthreads();
  for (int p0 = tid; p0 < P; p0 += 4 * NT) {
    int ev[4];
#pragma unroll
    for (int u = 0; u < 4; ++u) ev[u] = p0 + u * NT < P ? a.ids[p0 + u * NT] : 0;
#pragma unroll
    for (int u = 0; u < 4; ++u)
      if (p0 + u * NT < P) a.perm[atomicAdd(&cnt[ev[u]], 1)] = p0 + u * NT;
  }

  // ---- I. header, stats, clock, mailbox
  const int pick_hits = scal[1];
  if (tid == 0) {
    PlanHdr h = {};
    h.n_unique = nU;
    h.n_hits = nH;
    h.n_miss = nM;
    h.n_stage0_miss = n0;
    h.n_stages = n_stages;
    h.n_units = n_units;
    h.n_evict = scal[2];
    h.pick_hits = pick_hits;
    h.pick_misses = P - pick_hits;
    h.hit_units = hit_units;
    h.hit_gunits = hit_gunits;
    h.epoch = epoch;
    h.stage_cap = C;
    *a.epoch = epoch;
    *a.hdr = h;
    *a.clock = now;
    uint64_t *st = a.stats;
    st[0] += 1;
    st[1] += (uint64_t)pick_hits;
    st[2] += (uint64_t)(P - pick_hits);
    st[3] += (uint64_t)nH;
    st[4] += (uint64_t)nM;
    st[5] += (uint64_t)scal[2];
    st[6] += (uint64_t)nM * a.expert_bytes;
    st[7] += (uint64_t)n_stages;
    st[8] += n_stages > 1 ? 1ull : 0ull;
    if (a.mailbox) a.mailbox->hdr = h;
  }
  if (a.mailbox) {
    int32_t *mub = reinterpret_cast<int32_t *>(a.mailbox + 1);
    MissItem *mm = reinterpret_cast<MissItem *>(mub + a.mailbox_stage_cap);
    for (int j = tid; j <= n_stages; j += NT) {
      const int first_item = (j == 0) ? 0 : min(nU, nH + n0 + (j - 1) * C);
      mub[j] = (int)(itm[first_item] >> 32);
    }
    for (int i = tid; i < nM; i += NT) mm[i] = miss_record(i, n0, C, M, victim, qslot, se0, occ0);
    __threadfence_system();
    __syncthreads();
    if (tid == 0) {
      __threadfence_system();
      a.mailbox->seq = a.seq;
      __threadfence_system();
    }
  }
}


// Single-warp plan for small calls: at most 32 (token, pick) pairs, at most 256
// slots, and no more distinct experts possible than slots (one stage).  Same
// rule and outputs as plan_kernel, with warp-synchronous code only (small
// code: this kernel runs once per layer call, mostly from a cold instruction
// cache).
constexpr int kSmallMaxSlots = 256;
constexpr int kRouteGridMin = 8;  // calls with more tokens route in their own grid (one warp per token)

// POLICY: MOE_POLICY_LRU (0) or MOE_POLICY_SCORE (1); the LRU instance carries
// none of the score code or its shared memory.
template <int POLICY>
__global__ void __launch_bounds__(32, 1) plan_small_kernel(PlanArgs a) {
  const unsigned F = 0xffffffffu;
  const int E = a.E, S = a.S, k = a.k, T = a.T, P = T * k;
  const int lane = threadIdx.x;
  __shared__ int s_bad;
  __shared__ uint32_t s_pinned[kSmallMaxSlots / 32];
  __shared__ int s_se[kSmallMaxSlots];
  __shared__ unsigned long long s_st[kSmallMaxSlots];
  __shared__ int s_es[kMaxExperts];
  __shared__ unsigned long long s_pack[kMaxExperts];
  __shared__ unsigned long long s_key[kSmallMaxSlots];
  __shared__ int32_t s_ids[32];  // the routed ids, pair order (P <= 32)
  __shared__ float s_score[POLICY == 1 ? kMaxExperts : 1];  // policy 1: the layer's decayed usage scores
  __shared__ int s_fr[POLICY == 1 ? kSmallMaxSlots : 1];      // policy 1: empty slots, ascending
  // Launched as a programmatic dependent of the kernel before it: until
  // griddepcontrol.wait it reads only the layer's state and the handle's
  // counters, which only earlier plan kernels write (complete before that
  // kernel passed its own wait), and writes nothing.  The state goes to shared
  // memory by asynchronous copies that land while the router runs.
  for (int i = lane; i < S; i += 32) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(&s_se[i])), "l"(a.slot_expert + i)
                 : "memory");
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_addr(&s_st[i])), "l"(a.slot_stamp + i)
                 : "memory");
  }
  for (int i = lane; i < E; i += 32)
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(&s_es[i])), "l"(a.expert_slot + i)
                 : "memory");
  if constexpr (POLICY == 1)
    for (int i = lane; i < E; i += 32)
      asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(&s_score[i])), "l"(a.score + i)
                   : "memory");
  asm volatile("cp.async.commit_group;" ::: "memory");
  const unsigned long long now = *a.clock + 1ull;
  const uint32_t epoch = *a.epoch + 1u;  // loaded early: the header is the last thing written
  // the caller's logits, and scratch the kernel before may still read, only
  // after it has completed; this grid's dependent (the decode layer kernel)
  // may then start its plan-independent prologue
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
  float lg4[4], lg8[8];
  if (E <= 128) load_logits<4>(a.logits, E, lg4);
  else if (E <= 256) load_logits<8>(a.logits, E, lg8);
  if (lane == 0) s_bad = 0;
  if (lane < kSmallMaxSlots / 32) s_pinned[lane] = 0;
  for (int i = lane; i < a.sync_n; i += 32) a.sync[i] = 0;
  __syncwarp();
  for (int t = 0; t < T; ++t) {
    const float *row = a.logits + (size_t)t * E;
    if (E <= 128) {
      if (t > 0) load_logits<4>(row, E, lg4);
      route_values<4>(lg4, E, k, a.weight_mode, a.ids + t * k, a.w + t * k, &s_bad, s_ids + t * k);
    } else if (E <= 256) {
      if (t > 0) load_logits<8>(row, E, lg8);
      route_values<8>(lg8, E, k, a.weight_mode, a.ids + t * k, a.w + t * k, &s_bad, s_ids + t * k);
    } else {
      route_token<32>(row, E, k, a.weight_mode, a.ids + t * k, a.w + t * k, &s_bad, s_ids + t * k);
    }
  }
  asm volatile("cp.async.wait_all;" ::: "memory");
  __syncwarp();
  if (s_bad) {
    write_error(a);
    return;
  }

  // policy 1: token by token every score x0.9, then each pick +1 (fp32, each
  // operation rounded, none fused: the same bits as any plain evaluation)
  if constexpr (POLICY == 1) {
    for (int t = 0; t < T; ++t) {
      for (int i = lane; i < E; i += 32) s_score[i] = __fmul_rn(s_score[i], 0.9f);
      __syncwarp();
      if (lane < k) s_score[s_ids[t * k + lane]] = __fadd_rn(s_score[s_ids[t * k + lane]], 1.0f);
      __syncwarp();
    }
    for (int i = lane; i < E; i += 32) a.score[i] = s_score[i];
  }

  // distinct experts: one leader lane per expert
  const bool act = lane < P;
  const int e = act ? s_ids[lane] : -1 - lane;
  const unsigned same = __match_any_sync(F, e);
  const int leader = __ffs(same) - 1;
  const bool lead = act && leader == lane;
  const int cnt = __popc(same);
  const int es0 = lead ? s_es[e] : -1;
  const bool hit = lead && es0 >= 0, miss = lead && es0 < 0;
  const unsigned hmask = __ballot_sync(F, hit), mmask = __ballot_sync(F, miss);
  const int nH = __popc(hmask), nM = __popc(mmask), nU = nH + nM;
  const int my_hit = __shfl_sync(F, hit ? 1 : 0, leader);
  const int pick_hits = __popc(__ballot_sync(F, act && my_hit));
  if (hit) atomicOr(&s_pinned[es0 >> 5], 1u << (es0 & 31));

  // per-expert packed counts, 8 bits each: [hit leaders][miss leaders]
  // [hit pairs][miss pairs][hit units][miss units]; their prefix over expert
  // ids gives every leader its item rank, pair offset and unit offset in the
  // item order (hits ascending, then misses ascending)
  const int ucount = (cnt + kTokPerUnit - 1) / kTokPerUnit;
  uint64_t total, before;
  if (T == 1) {
    // one token: k distinct experts, one pair and one unit each, so an
    // expert's prefix is the number of hit and of miss experts of lower id
    // (the fields the scan below gives), from k shuffles
    int bh = 0, bm = 0;
    for (int jl = 0; jl < k; ++jl) {
      const int ej = __shfl_sync(F, e, jl);
      bh += ((hmask >> jl) & 1u) && ej < e;
      bm += ((mmask >> jl) & 1u) && ej < e;
    }
    auto pack = [](uint64_t h, uint64_t m) { return h | (m << 8) | (h << 16) | (m << 24) | (h << 32) | (m << 40); };
    total = pack((uint64_t)nH, (uint64_t)nM);
    before = pack((uint64_t)bh, (uint64_t)bm);
  } else {
    const int csz = (E + 31) / 32;  // experts per lane in the scan
    for (int i = lane; i < csz * 32; i += 32) s_pack[i] = 0ull;
    __syncwarp();
    if (lead)
      s_pack[e] = hit ? (1ull | ((uint64_t)cnt << 16) | ((uint64_t)ucount << 32))
                      : ((1ull << 8) | ((uint64_t)cnt << 24) | ((uint64_t)ucount << 40));
    __syncwarp();
    uint64_t part = 0;
    for (int i = 0; i < csz; ++i) part += s_pack[lane * csz + i];
    uint64_t incl = part;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const uint64_t y = __shfl_up_sync(F, incl, o);
      if (lane >= o) incl += y;
    }
    total = __shfl_sync(F, incl, 31);
    const int src = lead ? e / csz : 0;
    before = __shfl_sync(F, incl - part, src);  // exclusive prefix of my expert's chunk
    if (lead)
      for (int i = src * csz; i < e; ++i) before += s_pack[i];
  }
  auto field = [](uint64_t v, int f) { return (int)((v >> (8 * f)) & 0xffull); };
  const int tot_hit_pairs = field(total, 2), tot_hit_units = field(total, 4);
  const int hr = field(before, 0), mr = field(before, 1);

  int vslot = -1, evicted = -1;  // a miss leader's slot (-1: bypassed) and the expert it replaces
  if constexpr (POLICY == 1) {
    // decayed score with admission: rounds over the misses, strongest first
    // (score descending, lower id); each takes the next empty slot, else the
    // weakest slot whose expert the call does not pick (score ascending, lower
    // index) if strictly stronger, while the budget lasts; the first miss that
    // cannot be admitted ends the rounds (every later one is weaker: bypassed)
    const int kpl = (S + 31) / 32;
    int nf = 0;
    for (int c = 0; c < kpl; ++c) {
      const int sl = c * 32 + lane;
      const bool em = sl < S && s_se[sl] < 0;
      const unsigned m = __ballot_sync(F, em);
      if (em) s_fr[nf + __popc(m & ((1u << lane) - 1u))] = sl;
      nf += __popc(m);
    }
    uint32_t evbits = 0;  // this lane's evictable slots, bit c = slot c * 32 + lane
    for (int c = 0; c < kpl; ++c) {
      const int sl = c * 32 + lane;
      if (sl < S && s_se[sl] >= 0 && !((s_pinned[c] >> lane) & 1u)) {
        // sticky share: a slot is kept when fewer than n_sticky occupied slots
        // score higher (ties: lower index first)
        bool kept = false;
        if (a.n_sticky > 0) {
          const float sc = s_score[s_se[sl]];
          int above = 0;
          for (int s2 = 0; s2 < S; ++s2) {
            const int e2 = s_se[s2];
            above += e2 >= 0 && (s_score[e2] > sc || (s_score[e2] == sc && s2 < sl));
          }
          kept = above < a.n_sticky;
        }
        if (!kept) evbits |= 1u << c;
      }
    }
    __syncwarp();
    bool pend = miss;
    int remaining = a.admit_budget > 0 ? a.admit_budget : S + 1, used_free = 0;
    for (int r = 0; r < nM; ++r) {
      float bs = pend ? s_score[e] : -1.f;
      int bi = pend ? e : 0x7fffffff;
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) {
        const float os = __shfl_xor_sync(F, bs, o);
        const int oi = __shfl_xor_sync(F, bi, o);
        if (os > bs || (os == bs && oi < bi)) { bs = os; bi = oi; }
      }
      int slot = -1, old = -1;
      if (remaining > 0) {
        if (used_free < nf) {
          slot = s_fr[used_free++];
        } else {
          float ws = __int_as_float(0x7f800000);  // +inf
          int wsl = 0x7fffffff;
          for (int c = 0; c < kpl; ++c)
            if ((evbits >> c) & 1u) {
              const int sl = c * 32 + lane;
              const float sc = s_score[s_se[sl]];
              if (sc < ws || (sc == ws && sl < wsl)) { ws = sc; wsl = sl; }
            }
#pragma unroll
          for (int o = 16; o > 0; o >>= 1) {
            const float os = __shfl_xor_sync(F, ws, o);
            const int osl = __shfl_xor_sync(F, wsl, o);
            if (os < ws || (os == ws && osl < wsl)) { ws = os; wsl = osl; }
          }
          if (wsl != 0x7fffffff && bs > ws) {
            slot = wsl;
            old = s_se[wsl];
            if ((wsl & 31) == lane) evbits &= ~(1u << (wsl >> 5));
          }
        }
      }
      if (slot >= 0) --remaining;
      if (pend && e == bi) {
        vslot = slot;
        evicted = old;
        pend = false;
      }
      if (slot < 0) break;
    }
  } else {
    // stage-0 victims: empty slots (by index), then unpinned slots by (stamp, index);
    // miss rank r takes the r-th smallest key
    __syncwarp();
    unsigned long long key = ~0ull;
    for (int c = 0; c * 32 < S; ++c) {
      const int sl = c * 32 + lane;
      if (sl < S && !((s_pinned[c] >> lane) & 1u)) {
        const int se = s_se[sl];
        const unsigned long long kk =
            se < 0 ? (unsigned long long)sl : (1ull << 62) | ((unsigned long long)s_st[sl] << 11) | (unsigned)sl;
        key = kk < key ? kk : key;
      }
    }
    // lanes hold their smallest remaining key; keys beyond one per lane stay in s_key
    const int kpl = (S + 31) / 32;
    if (kpl > 1) {
      for (int c = 0; c < kpl; ++c) {
        const int sl = c * 32 + lane;
        unsigned long long kk = ~0ull;
        if (sl < S && !((s_pinned[c] >> lane) & 1u)) {
          const int se = s_se[sl];
          kk = se < 0 ? (unsigned long long)sl : (1ull << 62) | ((unsigned long long)s_st[sl] << 11) | (unsigned)sl;
        }
        s_key[sl] = kk;
      }
      __syncwarp();
    }
    int my_victim = -1;  // lane r holds the victim of miss rank r
    for (int r = 0; r < nM; ++r) {
      const unsigned hi = __reduce_min_sync(F, (unsigned)(key >> 32));
      const unsigned lo = __reduce_min_sync(F, (unsigned)(key >> 32) == hi ? (unsigned)key : 0xffffffffu);
      const unsigned long long best = ((unsigned long long)hi << 32) | lo;
      const int sl = (int)(best & 2047ull);
      if (lane == r) my_victim = sl;
      if (lane == (sl & 31)) {
        // the owner drops the taken key and exposes its next smallest
        if (kpl == 1) {
          key = ~0ull;
        } else {
          s_key[sl] = ~0ull;
          key = ~0ull;
          for (int c = 0; c < kpl; ++c) {
            const unsigned long long kk = s_key[c * 32 + lane];
            key = kk < key ? kk : key;
          }
        }
      }
    }
    const int v = __shfl_sync(F, my_victim, miss ? mr : 0);
    if (miss) {
      vslot = v;
      evicted = s_se[v];
    }
  }
  const int my_slot = hit ? es0 : (miss ? vslot : -1);
  const int n_bypass = __popc(__ballot_sync(F, miss && vslot < 0));
  const int n_evict = __popc(__ballot_sync(F, miss && evicted >= 0));
  __syncwarp();

  // new state (a bypassed miss changes nothing)
  if (miss && vslot >= 0) {
    a.slot_expert[vslot] = e;
    a.expert_slot[e] = vslot;
    a.slot_stamp[vslot] = now;
    if (evicted >= 0) a.expert_slot[evicted] = -1;
  }
  if (miss) a.miss[mr] = MissItem{e, vslot, evicted, 0};
  if (hit) a.slot_stamp[es0] = now;
  if (lead) a.usage[e] += (uint32_t)cnt;

  // per-pair slot and stage
  const int pslot = __shfl_sync(F, my_slot, leader);
  if (act) {
    a.gpu_slot[lane] = pslot;
    a.stage[lane] = 0;
  }

  // work items (hits ascending, then misses ascending), units, perm
  const int item = hit ? hr : (miss ? nH + mr : -1);
  const int pb = hit ? field(before, 2) : tot_hit_pairs + field(before, 3);
  const int ub = hit ? field(before, 4) : tot_hit_units + field(before, 5);
  const int n_units = tot_hit_units + field(total, 5);
  if (lead) {
    a.items[item] = WorkItem{e, my_slot, 0, miss ? 1 : 0, pb, cnt};
    for (int j = 0; j < ucount; ++j)
      a.units[ub + j] = WorkUnit{item, pb + j * kTokPerUnit, min(kTokPerUnit, cnt - j * kTokPerUnit), 0};
    a.gunits[item] = WorkUnit{item, pb, cnt, 0};  // at most 32 pairs: one GEMM unit per item
  }
  const int ppb = __shfl_sync(F, pb, leader);
  if (act) a.perm[ppb + __popc(same & ((1u << lane) - 1u))] = lane;
  if (lane == 0) {
    a.unit_begin[0] = 0;
    a.unit_begin[1] = n_units;
    a.gunit_begin[0] = 0;
    a.gunit_begin[1] = nU;
    PlanHdr h = {};
    h.n_unique = nU;
    h.n_hits = nH;
    h.n_miss = nM;
    h.n_stage0_miss = nM;
    h.n_stages = 1;
    h.n_units = n_units;
    h.n_evict = n_evict;
    h.pick_hits = pick_hits;
    h.pick_misses = P - pick_hits;
    h.hit_units = tot_hit_units;
    h.hit_gunits = nH;
    h.epoch = epoch;
    h.stage_cap = S;
    *a.epoch = epoch;
    *a.hdr = h;
    *a.clock = now;
    unsigned long long *st = reinterpret_cast<unsigned long long *>(a.stats);
    atomicAdd(st + 0, 1ull);
    atomicAdd(st + 1, (unsigned long long)pick_hits);
    atomicAdd(st + 2, (unsigned long long)(P - pick_hits));
    atomicAdd(st + 3, (unsigned long long)nH);
    atomicAdd(st + 4, (unsigned long long)nM);
    atomicAdd(st + 5, (unsigned long long)n_evict);
    atomicAdd(st + 6, (unsigned long long)nM * a.expert_bytes);
    atomicAdd(st + 7, 1ull);
    if (n_bypass) atomicAdd(st + 9, (unsigned long long)n_bypass);
    if (a.mailbox) {
      a.mailbox->hdr = h;
      int32_t *mub = reinterpret_cast<int32_t *>(a.mailbox + 1);
      mub[0] = 0;
      mub[1] = n_units;
    }
  }
  if (a.mailbox) {
    int32_t *mub = reinterpret_cast<int32_t *>(a.mailbox + 1);
    MissItem *mm = reinterpret_cast<MissItem *>(mub + a.mailbox_stage_cap);
    if (miss) mm[mr] = MissItem{e, vslot, evicted, 0};
    __threadfence_system();
    __syncwarp();
    if (lane == 0) {
      __threadfence_system();
      a.mailbox->seq = a.seq;
      __threadfence_system();
    }
  }
}

}  // namespace

size_t plan_smem_bytes(int E, int S) {
  auto r8 = [](size_t n) { return 8 * ((n + 1) / 2 * 2); };
  auto r4 = [](size_t n) { return 4 * ((n + 3) / 4 * 4); };
  size_t b = r8(S) + r8(E + 1) + r8(NW + 2);
  b += 8 * r4(E) + r4(E + 1);
  b += 8 * r4(S);
  b += r4(NW + 2) + r4(8);
  return b + 64;
}

bool plan_small_ok(int T, int E, int k, int S) {
  const int P = T * k;
  return P <= 32 && S <= kSmallMaxSlots && (E < P ? E : P) <= S;
}

cudaError_t launch_plan(const PlanArgs &a_in, cudaStream_t st) {
  if (plan_small_ok(a_in.T, a_in.E, a_in.k, a_in.S)) {
    // a programmatic dependent of the kernel before it (see plan_small_kernel)
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1);
    cfg.blockDim = dim3(32);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return a_in.policy == 1 ? cudaLaunchKernelEx(&cfg, plan_small_kernel<1>, a_in)
                            : cudaLaunchKernelEx(&cfg, plan_small_kernel<0>, a_in);
  }
  PlanArgs a = a_in;
  a.routed = 0;
  if (a.T > kRouteGridMin && a.route_bad) {
    // many tokens: route them grid-wide first (one warp per token)
    const dim3 grid((a.T + 7) / 8);
    if (a.E <= 128)
      route_kernel<4><<<grid, 256, 0, st>>>(a.logits, a.T, a.E, a.k, a.weight_mode, a.ids, a.w, a.route_bad);
    else if (a.E <= 256)
      route_kernel<8><<<grid, 256, 0, st>>>(a.logits, a.T, a.E, a.k, a.weight_mode, a.ids, a.w, a.route_bad);
    else
      route_kernel<32><<<grid, 256, 0, st>>>(a.logits, a.T, a.E, a.k, a.weight_mode, a.ids, a.w, a.route_bad);
    const cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) return e;
    a.routed = 1;
  }
  const size_t smem = plan_smem_bytes(a.E, a.S);
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(plan_kernel, smem, cur);
  if (e != cudaSuccess) return e;
  plan_kernel<<<1, NT, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace moe
