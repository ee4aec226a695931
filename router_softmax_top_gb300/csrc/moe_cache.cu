// Host runtime and C ABI of the routed-MoE expert-slot cache (see
// include/moe_cache.h for the contract of every entry point).
//
// Per layer call, on the caller's stream:
//   plan kernel (router + LRU slot map + work lists)
//   -> stage-0 hit gate/up (does not wait for any copy)
//   -> [fill] misses of the stage: cudaMemcpyAsync per block on the side stream
//      into staging, then a repack kernel into the slots (MOE_FILL_MEMCPY), or a
//      repack kernel reading the mapped host store directly (MOE_FILL_PULL)
//   -> miss gate/up -> down -> (next stage ...) -> weighted combine.
// The host learns the miss list from a mapped mailbox the plan kernel writes
// ("Longhaul MoE loading": one synchronisation per routed layer to discover the
// selected experts and populate missing slots).  A slot is only read by kernels
// ordered after its copy ("llama.cpp + MoE expert cache", "Keeping the cache
// fresh": publish after the copy completes).
#include <algorithm>
#include <atomic>
#include <chrono>
#include <cstdio>
#include <cstdlib>
#include <cmath>
#include <cstring>
#include <new>
#include <vector>

#include "common.cuh"
#include "moe_cache.h"
#include "plan_check.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

using namespace moe;

namespace {

struct TimingPool {
  bool on = false;
  std::vector<cudaEvent_t> ev;  // pairs
  std::vector<int> kind;
  int used = 0;
  double ms[K_NKINDS] = {};
  uint64_t n[K_NKINDS] = {};
};

}  // namespace

struct moe_cache {
  moe_cache_config cfg;
  moe_host_store store;
  int device = 0;
  bool registered = false;
  const uint8_t *host_dev = nullptr;  // device-visible alias of the host store
  SlotLayout lay;
  uint64_t expert_bytes = 0;
  int maxP = 0, maxU = 0, maxUnits = 0, maxStages = 0;

  // persistent device state
  uint8_t *d_slots = nullptr;
  uint8_t *d_stage_buf = nullptr;  // 2 x S blocks (slot layout): stages >= 1 of staged calls
  std::vector<int> fin_src;         // [S] after a staged call: the stage holding each slot's final block
  cudaEvent_t ev_fin = nullptr;
  int32_t *d_slot_expert = nullptr, *d_expert_slot = nullptr;
  uint64_t *d_slot_stamp = nullptr, *d_clock = nullptr, *d_stats = nullptr;
  float *d_score = nullptr;  // MOE_POLICY_SCORE: decayed usage per (layer, expert), fp32
  uint32_t *d_usage = nullptr;  // lifetime activation counts per (layer, expert)

  // per-call scratch
  int32_t *d_ids = nullptr, *d_gpu_slot = nullptr, *d_stage = nullptr, *d_perm = nullptr;
  int32_t *d_unit_begin = nullptr;
  float *d_w = nullptr, *d_h = nullptr, *d_y = nullptr;
  WorkItem *d_items = nullptr;
  WorkUnit *d_units = nullptr;
  MissItem *d_miss = nullptr;
  PlanHdr *d_hdr = nullptr;
  int32_t *d_sync = nullptr;  // per-call counters: queue head, per item, per (token, row tile)
  // decode layer kernel: gate/up outputs [2][maxPd][F] and down outputs [maxPd][H], each value
  // stored with the number of the call that wrote it (maxPd = pairs of 8 tokens)
  uint64_t *d_gut = nullptr, *d_yt = nullptr;
  uint32_t *d_epoch = nullptr;  // call counter, advanced by the plan
  int32_t *d_route_bad = nullptr;  // non-finite-logit flag of the grid router
  int n_sms = 0;
  WorkUnit *d_gunits = nullptr;
  int32_t *d_gunit_begin = nullptr;
  __nv_bfloat16 *d_h16 = nullptr;  // gate/up output of the GEMM path, pair-sorted rows [maxP, F]
  __nv_bfloat16 *d_xs = nullptr;   // activations in pair-sorted order [maxP, H]
  GemmMaps xs_maps, h16_maps;
  RawMaps slot_maps, stage_maps;  // the slot planes of all layers' slots, of the stage buffers
  int maxGunits = 0;
  uint8_t *d_staging = nullptr;
  int staging_blocks = 0;
  // memcpy fill through the decode layer kernel: [r] = call number once staging
  // block r has landed, written by a stream memory operation after the copy
  uint32_t *d_miss_ready = nullptr;
  using WriteValueFn = CUresult (*)(CUstream, CUdeviceptr, cuuint32_t, unsigned int);
  WriteValueFn write_value32 = nullptr;

  // mapped host words
  unsigned char *h_mail_raw = nullptr;
  Mailbox *h_mail = nullptr, *d_mail = nullptr;
  int32_t *h_mail_ub = nullptr;
  MissItem *h_mail_miss = nullptr;
  int mail_stage_cap = 0;
  int32_t *h_err = nullptr, *d_err = nullptr;
  uint32_t seq = 0;

  cudaStream_t side = nullptr;
  cudaStream_t side2 = nullptr;  // memcpy fill through the decode layer kernel: every second missed block
  cudaEvent_t ev_plan = nullptr;
  std::vector<cudaEvent_t> ev_up, ev_done;

  int poisoned = 0, last_error = MOE_OK, cuda_error = 0;
  int inject = 0;  // pending fault injection (moe_cache_inject)
  int copy_fail_in = 0;  // > 0: the copy_fail_in-th next fill copy fails before it is issued
  bool check_plans = false;  // MOE_CHECK_PLANS=1 at init: host check of every call's plan
  int last_layer = -1, last_T = 0;
  std::atomic<uint64_t> launches{0};
  TimingPool tp;
};

namespace {

const char *const kKindNames[K_NKINDS] = {"plan",        "repack",    "q4_gateup_gemv", "q4_down_gemv",
                                          "combine",     "gemm_gateup", "gemm_down",    "gather",
                                          "h2d_memcpy",  "fused_miss",  "decode_layer"};

// The handle's device error word: 1 = a non-finite router logit (the plan),
// anything else = a bounded device wait gave up.
int device_error_code(const moe_cache *c) {
  const int32_t e = __atomic_load_n(c->h_err, __ATOMIC_ACQUIRE);
  return e == 0 ? MOE_OK : e == 1 ? MOE_ERR_INVALID_ARG : MOE_ERR_TIMEOUT;
}

int poison(moe_cache *c, int code) {
  if (!c->poisoned) {
    c->poisoned = 1;
    c->last_error = code;
    if (code == MOE_ERR_CUDA) {
      const cudaError_t e = cudaGetLastError();
      if (!c->cuda_error) c->cuda_error = (int)e;
    }
  }
  return code;
}

int poison_cuda(moe_cache *c, cudaError_t e) {
  if (!c->poisoned && !c->cuda_error) c->cuda_error = (int)e;
  return poison(c, MOE_ERR_CUDA);
}

// --- timing: event pairs on the launching stream
void tp_flush(moe_cache *c) {
  TimingPool &t = c->tp;
  if (t.used == 0) return;
  cudaEventSynchronize(t.ev[2 * (t.used - 1) + 1]);
  for (int i = 0; i < t.used; ++i) {
    float ms = 0.f;
    if (cudaEventElapsedTime(&ms, t.ev[2 * i], t.ev[2 * i + 1]) == cudaSuccess) {
      t.ms[t.kind[i]] += ms;
      t.n[t.kind[i]] += 1;
    }
  }
  t.used = 0;
}

// Room for n more timed launches now (flushing waits for the device), so that
// no flush falls where the host must not block.
void tp_reserve(moe_cache *c, int n) {
  TimingPool &t = c->tp;
  if (t.on && t.used + n > (int)t.kind.size()) tp_flush(c);
}

int tp_begin(moe_cache *c, int kind, cudaStream_t st) {
  TimingPool &t = c->tp;
  if (!t.on) return -1;
  if (t.used == (int)t.kind.size()) tp_flush(c);
  const int i = t.used++;
  t.kind[i] = kind;
  cudaEventRecord(t.ev[2 * i], st);
  return i;
}

void tp_end(moe_cache *c, int i, cudaStream_t st) {
  if (i >= 0) cudaEventRecord(c->tp.ev[2 * i + 1], st);
}

struct Launch {
  moe_cache *c;
  cudaStream_t st;
  int idx;
  Launch(moe_cache *c_, int kind, cudaStream_t s) : c(c_), st(s) {
    idx = tp_begin(c, kind, s);
    if (kind != K_MEMCPY) c->launches.fetch_add(1, std::memory_order_relaxed);
  }
  ~Launch() { tp_end(c, idx, st); }
};

double now_us() {
  using namespace std::chrono;
  return (double)duration_cast<nanoseconds>(steady_clock::now().time_since_epoch()).count() * 1e-3;
}

// Wait for the plan kernel's mailbox write, bounded by cfg.timeout_us.
int wait_mailbox(moe_cache *c, uint32_t seq, cudaStream_t st) {
  const double t0 = now_us();
  uint32_t *p = const_cast<uint32_t *>(&c->h_mail->seq);
  for (uint64_t it = 0;; ++it) {
    if (__atomic_load_n(p, __ATOMIC_ACQUIRE) == seq) return MOE_OK;
    if ((it & 255) == 255) {
      const cudaError_t e = cudaStreamQuery(st);
      if (e != cudaSuccess && e != cudaErrorNotReady) return MOE_ERR_CUDA;
      if (e == cudaSuccess) {
        // the stream drained: the plan kernel has finished, so its mailbox write
        // must show up; give the host view a short grace period
        const double t1 = now_us();
        while (now_us() - t1 < 2000.0)
          if (__atomic_load_n(p, __ATOMIC_ACQUIRE) == seq) return MOE_OK;
        return MOE_ERR_CUDA;
      }
      if (now_us() - t0 > (double)c->cfg.timeout_us) return MOE_ERR_TIMEOUT;
    }
  }
}

int wait_stream(cudaStream_t st, int64_t timeout_us) {
  const double t0 = now_us();
  for (;;) {
    const cudaError_t e = cudaStreamQuery(st);
    if (e == cudaSuccess) return MOE_OK;
    if (e != cudaErrorNotReady) return MOE_ERR_CUDA;
    if (now_us() - t0 > (double)timeout_us) return MOE_ERR_TIMEOUT;
  }
}

// One host-to-device copy of a missed block (memcpy fill).  An injected
// failure (MOE_INJECT_MEMCPY_FAIL) makes the n-th such copy fail before it is
// issued, as a refused copy would.
cudaError_t fill_copy(moe_cache *c, void *dst, const void *src, size_t bytes, cudaStream_t st) {
  if (c->copy_fail_in > 0 && --c->copy_fail_in == 0) {
    if (!c->cuda_error) c->cuda_error = (int)cudaErrorUnknown;
    return cudaErrorUnknown;
  }
  return cudaMemcpyAsync(dst, src, bytes, cudaMemcpyHostToDevice, st);
}

template <typename T>
cudaError_t dalloc(T **p, size_t n) {
  return cudaMalloc(reinterpret_cast<void **>(p), sizeof(T) * (n ? n : 1));
}

void free_all(moe_cache *c) {
  cudaFree(c->d_slots);
  cudaFree(c->d_stage_buf);
  if (c->ev_fin) cudaEventDestroy(c->ev_fin);
  cudaFree(c->d_slot_expert);
  cudaFree(c->d_expert_slot);
  cudaFree(c->d_slot_stamp);
  cudaFree(c->d_clock);
  cudaFree(c->d_stats);
  cudaFree(c->d_score);
  cudaFree(c->d_usage);
  cudaFree(c->d_ids);
  cudaFree(c->d_gpu_slot);
  cudaFree(c->d_stage);
  cudaFree(c->d_perm);
  cudaFree(c->d_unit_begin);
  cudaFree(c->d_w);
  cudaFree(c->d_h);
  cudaFree(c->d_y);
  cudaFree(c->d_items);
  cudaFree(c->d_units);
  cudaFree(c->d_miss);
  cudaFree(c->d_hdr);
  cudaFree(c->d_sync);
  cudaFree(c->d_gut);
  cudaFree(c->d_yt);
  cudaFree(c->d_epoch);
  cudaFree(c->d_route_bad);
  cudaFree(c->d_gunits);
  cudaFree(c->d_gunit_begin);
  cudaFree(c->d_h16);
  cudaFree(c->d_xs);
  cudaFree(c->d_staging);
  cudaFree(c->d_miss_ready);
  if (c->h_mail_raw) cudaFreeHost(c->h_mail_raw);
  if (c->h_err) cudaFreeHost(c->h_err);
  if (c->side) cudaStreamDestroy(c->side);
  if (c->side2) cudaStreamDestroy(c->side2);
  if (c->ev_plan) cudaEventDestroy(c->ev_plan);
  for (auto e : c->ev_up) cudaEventDestroy(e);
  for (auto e : c->ev_done) cudaEventDestroy(e);
  for (auto e : c->tp.ev) cudaEventDestroy(e);
  if (c->registered) cudaHostUnregister(const_cast<void *>(c->store.base));
}

int check_config(const moe_cache_config *g) {
  if (g->n_layers < 1 || g->n_experts < 1 || g->n_experts > kMaxExperts) return MOE_ERR_INVALID_ARG;
  if (g->top_k < 1 || g->top_k > g->n_experts || g->top_k > kMaxTopK) return MOE_ERR_INVALID_ARG;
  if (g->slots_per_layer < 1 || g->slots_per_layer > g->n_experts) return MOE_ERR_INVALID_ARG;
  if (g->max_tokens < 1 || (int64_t)g->max_tokens * g->top_k > (1 << 22)) return MOE_ERR_INVALID_ARG;
  if (g->weight_mode != 0 && g->weight_mode != 1) return MOE_ERR_INVALID_ARG;
  if (g->act_dtype != 0 && g->act_dtype != 1) return MOE_ERR_INVALID_ARG;
  if (g->fill_mode != MOE_FILL_MEMCPY && g->fill_mode != MOE_FILL_PULL) return MOE_ERR_INVALID_ARG;
  if (g->gemm_min_tokens < 0 || g->timeout_us <= 0 || g->sticky_permille < 0 || g->sticky_permille > 1000 ||
      (g->sticky_permille != 0 && g->policy != MOE_POLICY_SCORE))
    return MOE_ERR_INVALID_ARG;
  if ((g->policy != MOE_POLICY_LRU && g->policy != MOE_POLICY_SCORE && g->policy != MOE_POLICY_ADOPT) ||
      g->admit_budget < 0)
    return MOE_ERR_INVALID_ARG;
  if (g->hidden < 64 || g->hidden % 64 || g->ffn < 64 || g->ffn % 64) return MOE_ERR_UNSUPPORTED;
  if (g->hidden > 16384 || g->ffn > 16384) return MOE_ERR_UNSUPPORTED;
  return MOE_OK;
}

}  // namespace

// ======================================================================= ABI

MOE_API uint64_t moe_expert_bytes(int32_t hidden, int32_t ffn) {
  if (hidden <= 0 || ffn <= 0) return 0;
  return 3ull * (uint64_t)ffn * (uint64_t)(hidden / 32) * 18ull;
}

MOE_API const char *moe_strerror(int code) {
  switch (code) {
    case MOE_OK: return "ok";
    case MOE_ERR_INVALID_ARG: return "invalid argument";
    case MOE_ERR_CUDA: return "CUDA error";
    case MOE_ERR_OOM: return "out of memory";
    case MOE_ERR_TIMEOUT: return "timed out";
    case MOE_ERR_HOST_STORE: return "host store invalid or not registrable";
    case MOE_ERR_POISONED: return "handle poisoned by an earlier failure";
    case MOE_ERR_UNSUPPORTED: return "unsupported shape";
    case MOE_ERR_CHECK: return "a debug check of a call's plan failed";
    default: return "unknown error";
  }
}

MOE_API int moe_cache_init(const moe_cache_config *cfg, const moe_host_store *store,
                           void *cuda_stream, moe_cache **out) {
  if (!out) return MOE_ERR_INVALID_ARG;
  *out = nullptr;
  if (!cfg || !store) return MOE_ERR_INVALID_ARG;
  int rc = check_config(cfg);
  if (rc != MOE_OK) return rc;
  const uint64_t eb = moe_expert_bytes(cfg->hidden, cfg->ffn);
  if (!store->base || store->expert_stride < eb || store->layer_stride == 0) return MOE_ERR_HOST_STORE;
  if ((uintptr_t)store->base % 16 || store->expert_stride % 16 || store->layer_stride % 16)
    return MOE_ERR_HOST_STORE;
  const uint64_t last = (uint64_t)(cfg->n_layers - 1) * store->layer_stride +
                        (uint64_t)(cfg->n_experts - 1) * store->expert_stride + eb;
  if (last > store->bytes) return MOE_ERR_HOST_STORE;

  moe_cache *c = new (std::nothrow) moe_cache();
  if (!c) return MOE_ERR_OOM;
  c->cfg = *cfg;
  c->store = *store;
  c->lay = make_slot_layout(cfg->hidden, cfg->ffn);
  c->expert_bytes = eb;
  const int E = cfg->n_experts, S = cfg->slots_per_layer, L = cfg->n_layers, k = cfg->top_k;
  c->maxP = cfg->max_tokens * k;
  c->maxU = std::min(E, c->maxP);
  c->maxUnits = c->maxU + (c->maxP + kTokPerUnit - 1) / kTokPerUnit + 1;
  c->maxStages = 2 + (c->maxU + S - 1) / S;
  cudaStream_t st = (cudaStream_t)cuda_stream;

  auto fail = [&](int code) {
    cudaGetLastError();
    free_all(c);
    delete c;
    return code;
  };
  {
    const char *v = getenv("MOE_CHECK_PLANS");
    c->check_plans = v && v[0] == '1';
  }
  if (cudaGetDevice(&c->device) != cudaSuccess ||
      cudaDeviceGetAttribute(&c->n_sms, cudaDevAttrMultiProcessorCount, c->device) != cudaSuccess)
    return fail(MOE_ERR_CUDA);

  // host store: pinned and mapped
  cudaPointerAttributes pa;
  if (cudaPointerGetAttributes(&pa, store->base) != cudaSuccess) {
    cudaGetLastError();
    pa.type = cudaMemoryTypeUnregistered;
  }
  if (pa.type != cudaMemoryTypeHost) {
    if (cudaHostRegister(const_cast<void *>(store->base), store->bytes,
                         cudaHostRegisterMapped | cudaHostRegisterPortable) != cudaSuccess)
      return fail(MOE_ERR_HOST_STORE);
    c->registered = true;
  }
  void *hd = nullptr;
  if (cudaHostGetDevicePointer(&hd, const_cast<void *>(store->base), 0) != cudaSuccess) {
    cudaGetLastError();
    if (cfg->fill_mode == MOE_FILL_PULL) return fail(MOE_ERR_HOST_STORE);
    hd = nullptr;
  }
  c->host_dev = static_cast<const uint8_t *>(hd);

  // device memory
  const size_t slot_bytes = (size_t)L * S * c->lay.stride;
  bool ok = cudaMalloc(&c->d_slots, slot_bytes) == cudaSuccess;
  // staged calls (more distinct experts than slots) are possible: stages >= 1
  // alternate between two stage buffers, so that a stage's fill overlaps the
  // previous stage's compute
  if (ok && std::min(E, cfg->max_tokens * cfg->top_k) > S) {
    ok = cudaMalloc(&c->d_stage_buf, (size_t)2 * S * c->lay.stride) == cudaSuccess;
    c->fin_src.assign(S, 0);
  }
  ok = ok && dalloc(&c->d_slot_expert, (size_t)L * S) == cudaSuccess;
  ok = ok && dalloc(&c->d_expert_slot, (size_t)L * E) == cudaSuccess;
  ok = ok && dalloc(&c->d_slot_stamp, (size_t)L * S) == cudaSuccess;
  ok = ok && dalloc(&c->d_clock, (size_t)L) == cudaSuccess;
  ok = ok && dalloc(&c->d_stats, (size_t)L * kNStat) == cudaSuccess;
  ok = ok && dalloc(&c->d_score, (size_t)L * E) == cudaSuccess &&
       cudaMemset(c->d_score, 0, sizeof(float) * L * E) == cudaSuccess;
  ok = ok && dalloc(&c->d_usage, (size_t)L * E) == cudaSuccess &&
       cudaMemset(c->d_usage, 0, sizeof(uint32_t) * L * E) == cudaSuccess;
  ok = ok && dalloc(&c->d_ids, c->maxP) == cudaSuccess;
  ok = ok && dalloc(&c->d_gpu_slot, c->maxP) == cudaSuccess;
  ok = ok && dalloc(&c->d_stage, c->maxP) == cudaSuccess;
  ok = ok && dalloc(&c->d_perm, c->maxP) == cudaSuccess;
  ok = ok && dalloc(&c->d_unit_begin, c->maxStages + 1) == cudaSuccess;
  ok = ok && dalloc(&c->d_w, c->maxP) == cudaSuccess;
  ok = ok && dalloc(&c->d_h, (size_t)c->maxP * cfg->ffn) == cudaSuccess;
  ok = ok && dalloc(&c->d_y, (size_t)c->maxP * cfg->hidden) == cudaSuccess;
  ok = ok && dalloc(&c->d_items, c->maxU) == cudaSuccess;
  ok = ok && dalloc(&c->d_units, c->maxUnits) == cudaSuccess;
  ok = ok && dalloc(&c->d_miss, c->maxU) == cudaSuccess;
  ok = ok && dalloc(&c->d_hdr, 1) == cudaSuccess;
  ok = ok && dalloc(&c->d_sync, (size_t)c->maxU + 2 + (size_t)cfg->max_tokens * (cfg->hidden / 32)) == cudaSuccess;
  const size_t maxPd = (size_t)std::min(cfg->max_tokens, kTokPerUnit) * cfg->top_k;
  ok = ok && dalloc(&c->d_gut, 2 * maxPd * cfg->ffn) == cudaSuccess;
  ok = ok && dalloc(&c->d_yt, maxPd * cfg->hidden) == cudaSuccess;
  ok = ok && dalloc(&c->d_epoch, 1) == cudaSuccess;
  ok = ok && dalloc(&c->d_route_bad, 1) == cudaSuccess &&
       cudaMemsetAsync(c->d_route_bad, 0, sizeof(int32_t), (cudaStream_t)cuda_stream) == cudaSuccess;
  c->maxGunits = c->maxU + (c->maxP + kGemmN - 1) / kGemmN + 1;
  ok = ok && dalloc(&c->d_gunits, c->maxGunits) == cudaSuccess;
  ok = ok && dalloc(&c->d_gunit_begin, c->maxStages + 1) == cudaSuccess;
  if (ok && cfg->gemm_min_tokens > 0 && cfg->act_dtype == 1) {
    ok = dalloc(&c->d_h16, (size_t)c->maxP * cfg->ffn) == cudaSuccess &&
         dalloc(&c->d_xs, (size_t)c->maxP * cfg->hidden) == cudaSuccess;
    if (ok && (make_gemm_maps(c->d_xs, cfg->hidden, c->maxP, &c->xs_maps) != cudaSuccess ||
               make_gemm_maps(c->d_h16, cfg->ffn, c->maxP, &c->h16_maps) != cudaSuccess ||
               make_raw_maps(c->d_slots, L * S, c->lay.stride, c->lay, &c->slot_maps) != cudaSuccess ||
               (c->d_stage_buf &&
                make_raw_maps(c->d_stage_buf, 2 * S, c->lay.stride, c->lay, &c->stage_maps) != cudaSuccess)))
      return fail(MOE_ERR_CUDA);
  }
  if (ok && cfg->fill_mode == MOE_FILL_MEMCPY) {
    c->staging_blocks = std::min(S, c->maxU);
    ok = cudaMalloc(&c->d_staging, (size_t)c->staging_blocks * eb) == cudaSuccess &&
         dalloc(&c->d_miss_ready, c->staging_blocks) == cudaSuccess &&
         cudaMemset(c->d_miss_ready, 0, sizeof(uint32_t) * c->staging_blocks) == cudaSuccess;
    // cuStreamWriteValue32 from the driver; without it the memcpy fill keeps
    // its event-ordered schedule
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuStreamWriteValue32", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess && fn)
      c->write_value32 = reinterpret_cast<moe_cache::WriteValueFn>(fn);
    else
      cudaGetLastError();
  } else if (ok) {
    c->staging_blocks = 1;  // used by the bandwidth probe only
    ok = cudaMalloc(&c->d_staging, eb) == cudaSuccess;
  }
  if (!ok) return fail(MOE_ERR_OOM);
  // the score policy plans every call as one stage in the small plan kernel and
  // runs it on the decode layer kernel (a bypassed miss is computed there from
  // the host store, or from staging, without taking a slot)
  if (cfg->policy == MOE_POLICY_SCORE) {
    const int T = cfg->max_tokens, k = cfg->top_k;
    const bool fill_ok = cfg->fill_mode == MOE_FILL_PULL || c->write_value32 != nullptr;
    const bool gemm_off = cfg->gemm_min_tokens == 0 || cfg->gemm_min_tokens > T;
    if (T > kTokPerUnit || T * k > std::min(S, 32) || !plan_small_ok(T, E, k, S) || !gemm_off || !fill_ok ||
        !decode_layer_supported(cfg->hidden, cfg->ffn, T))
      return fail(MOE_ERR_UNSUPPORTED);
  }

  // mapped mailbox and error word
  c->mail_stage_cap = c->maxStages + 1;
  const size_t mail_bytes = sizeof(Mailbox) + sizeof(int32_t) * c->mail_stage_cap +
                            sizeof(MissItem) * c->maxU;
  if (cudaHostAlloc(&c->h_mail_raw, mail_bytes, cudaHostAllocMapped) != cudaSuccess)
    return fail(MOE_ERR_OOM);
  memset(c->h_mail_raw, 0, mail_bytes);
  c->h_mail = reinterpret_cast<Mailbox *>(c->h_mail_raw);
  c->h_mail_ub = reinterpret_cast<int32_t *>(c->h_mail + 1);
  c->h_mail_miss = reinterpret_cast<MissItem *>(c->h_mail_ub + c->mail_stage_cap);
  void *dm = nullptr;
  if (cudaHostGetDevicePointer(&dm, c->h_mail_raw, 0) != cudaSuccess) return fail(MOE_ERR_CUDA);
  c->d_mail = static_cast<Mailbox *>(dm);
  if (cudaHostAlloc(&c->h_err, sizeof(int32_t) * 4, cudaHostAllocMapped) != cudaSuccess)
    return fail(MOE_ERR_OOM);
  memset(c->h_err, 0, sizeof(int32_t) * 4);
  if (cudaHostGetDevicePointer(&dm, c->h_err, 0) != cudaSuccess) return fail(MOE_ERR_CUDA);
  c->d_err = static_cast<int32_t *>(dm);

  // streams and events
  // the side stream carries the fills: highest priority, so that its kernels
  // get SMs ahead of the compute kernels they overlap
  int prio_lo = 0, prio_hi = 0;
  if (cudaDeviceGetStreamPriorityRange(&prio_lo, &prio_hi) != cudaSuccess ||
      cudaStreamCreateWithPriority(&c->side, cudaStreamNonBlocking, prio_hi) != cudaSuccess ||
      (cfg->fill_mode == MOE_FILL_MEMCPY &&
       cudaStreamCreateWithPriority(&c->side2, cudaStreamNonBlocking, prio_hi) != cudaSuccess) ||
      cudaEventCreateWithFlags(&c->ev_fin, cudaEventDisableTiming) != cudaSuccess)
    return fail(MOE_ERR_CUDA);
  if (cudaEventCreateWithFlags(&c->ev_plan, cudaEventDisableTiming) != cudaSuccess) return fail(MOE_ERR_CUDA);
  c->ev_up.resize(c->maxStages);
  c->ev_done.resize(c->maxStages);
  for (int i = 0; i < c->maxStages; ++i) {
    if (cudaEventCreateWithFlags(&c->ev_up[i], cudaEventDisableTiming) != cudaSuccess ||
        cudaEventCreateWithFlags(&c->ev_done[i], cudaEventDisableTiming) != cudaSuccess)
      return fail(MOE_ERR_CUDA);
  }
  const int pool = 2048;
  c->tp.ev.resize(2 * pool);
  c->tp.kind.resize(pool);
  for (auto &e : c->tp.ev)
    if (cudaEventCreate(&e) != cudaSuccess) return fail(MOE_ERR_CUDA);

  // empty cache
  bool okm = cudaMemsetAsync(c->d_slot_expert, 0xFF, sizeof(int32_t) * L * S, st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_expert_slot, 0xFF, sizeof(int32_t) * L * E, st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_slot_stamp, 0, sizeof(uint64_t) * L * S, st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_clock, 0, sizeof(uint64_t) * L, st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_stats, 0, sizeof(uint64_t) * L * kNStat, st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_hdr, 0, sizeof(PlanHdr), st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_epoch, 0, sizeof(uint32_t), st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_gut, 0, sizeof(uint64_t) * 2 * maxPd * cfg->ffn, st) == cudaSuccess;
  okm = okm && cudaMemsetAsync(c->d_yt, 0, sizeof(uint64_t) * maxPd * cfg->hidden, st) == cudaSuccess;
  okm = okm && cudaStreamSynchronize(st) == cudaSuccess;
  if (!okm) return fail(MOE_ERR_CUDA);
  *out = c;
  return MOE_OK;
}

MOE_API int moe_layer_forward(moe_cache *c, int32_t layer, const float *d_logits, const void *d_x,
                              int32_t n_tokens, float *d_out, void *cuda_stream) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (c->poisoned) return MOE_ERR_POISONED;
  if (const int de = device_error_code(c)) return poison(c, de);
  const moe_cache_config &g = c->cfg;
  if (layer < 0 || layer >= g.n_layers || n_tokens < 0 || n_tokens > g.max_tokens)
    return MOE_ERR_INVALID_ARG;
  if (n_tokens == 0) return MOE_OK;
  if (!d_logits || !d_x || !d_out) return MOE_ERR_INVALID_ARG;
  cudaStream_t st = (cudaStream_t)cuda_stream;
  const int E = g.n_experts, k = g.top_k, S = g.slots_per_layer, T = n_tokens;
  const int P = T * k;
  const int maxU = std::min(E, P);
  const int maxUnits = maxU + (P + kTokPerUnit - 1) / kTokPerUnit;
  const bool use_gemm = g.gemm_min_tokens > 0 && T >= g.gemm_min_tokens && g.act_dtype == 1 &&
                        c->d_h16 != nullptr;
  const bool need_host = g.fill_mode == MOE_FILL_MEMCPY || maxU > S || use_gemm;

  c->seq += 1;
  if (c->seq == 0) c->seq = 1;
  PlanArgs pa;
  pa.logits = d_logits;
  pa.T = T;
  pa.E = E;
  pa.k = k;
  pa.S = S;
  pa.weight_mode = g.weight_mode;
  pa.slot_expert = c->d_slot_expert + (size_t)layer * S;
  pa.expert_slot = c->d_expert_slot + (size_t)layer * E;
  pa.slot_stamp = c->d_slot_stamp + (size_t)layer * S;
  pa.clock = c->d_clock + layer;
  pa.stats = c->d_stats + (size_t)layer * kNStat;
  pa.expert_bytes = c->expert_bytes;
  pa.ids = c->d_ids;
  pa.w = c->d_w;
  pa.gpu_slot = c->d_gpu_slot;
  pa.stage = c->d_stage;
  pa.perm = c->d_perm;
  pa.items = c->d_items;
  pa.units = c->d_units;
  pa.unit_begin = c->d_unit_begin;
  pa.gunits = c->d_gunits;
  pa.gunit_begin = c->d_gunit_begin;
  pa.miss = c->d_miss;
  pa.hdr = c->d_hdr;
  pa.err_flag = c->d_err;
  pa.sync = c->d_sync;
  pa.route_bad = c->d_route_bad;
  pa.routed = 0;
  pa.epoch = c->d_epoch;
  pa.policy = g.policy;
  pa.admit_budget = g.admit_budget;
  pa.score = c->d_score + (size_t)layer * E;
  pa.usage = c->d_usage + (size_t)layer * E;
  pa.n_sticky = (int)((int64_t)g.sticky_permille * S / 1000);
  const bool use_decode = !need_host && g.fill_mode == MOE_FILL_PULL && decode_layer_supported(g.hidden, g.ffn, T);
  // memcpy fill, one stage guaranteed (distinct experts <= slots), few tokens:
  // the decode layer kernel too, its misses read from staging as they land
  const bool use_decode_mc = g.fill_mode == MOE_FILL_MEMCPY && c->write_value32 && !use_gemm && maxU <= S &&
                             maxU <= c->staging_blocks && decode_layer_supported(g.hidden, g.ffn, T);
  pa.sync_n = 2 + maxU + ((use_decode || use_decode_mc) ? T * (g.hidden / 32) : 0);
  if (g.policy == MOE_POLICY_SCORE && !use_decode && !use_decode_mc) return MOE_ERR_UNSUPPORTED;
  pa.mailbox = need_host ? c->d_mail : nullptr;
  pa.mailbox_stage_cap = c->mail_stage_cap;
  pa.seq = c->seq;

  FfnArgs fa;
  fa.slots = c->d_slots + (size_t)layer * S * c->lay.stride;
  fa.slot_stride = c->lay.stride;
  fa.lay = c->lay;
  fa.H = g.hidden;
  fa.F = g.ffn;
  fa.k = k;
  fa.x = d_x;
  fa.x_bf16 = g.act_dtype == 1;
  fa.perm = c->d_perm;
  fa.items = c->d_items;
  fa.units = c->d_units;
  fa.unit_begin = c->d_unit_begin;
  fa.hdr = c->d_hdr;
  fa.h = c->d_h;
  fa.y = c->d_y;
  fa.max_tok = std::min(kTokPerUnit, T);
  fa.err = c->d_err;

  RepackArgs ra;
  ra.slots = c->d_slots + (size_t)layer * S * c->lay.stride;
  ra.slot_stride = c->lay.stride;
  ra.lay = c->lay;
  ra.miss = c->d_miss;
  ra.hdr = c->d_hdr;

  cudaError_t e;
#define MOE_LAUNCH(kind, expr)                          \
  do {                                                  \
    Launch _l(c, kind, st);                             \
    e = (expr);                                         \
    if (e != cudaSuccess) return poison_cuda(c, e);     \
  } while (0)

  MOE_LAUNCH(K_PLAN, launch_plan(pa, st));
  if (cudaEventRecord(c->ev_plan, st) != cudaSuccess) return poison(c, MOE_ERR_CUDA);
  const bool dc_ok = down_combine_supported(g.ffn, k);

  // Where stage j's misses live: stage 0 in their slots; later stages (whose
  // i-th miss takes slot i) alternately in the two stage buffers, so that the
  // fill of stage j + 1 overlaps the compute of stage j.
  uint8_t *const layer_slots = c->d_slots + (size_t)layer * S * c->lay.stride;
  auto stage_base = [&](int j) -> uint8_t * {
    return (j == 0 || !c->d_stage_buf) ? layer_slots : c->d_stage_buf + (size_t)(j & 1) * S * c->lay.stride;
  };
  // the event after which stage j's destination is free
  auto stage_free = [&](int j) -> cudaEvent_t { return j < 2 ? c->ev_plan : c->ev_done[j - 2]; };

  // fill of stage j's misses on the side stream: host copies (memcpy mode)
  // after `after`, the repack into the stage's destination after `dst_free`;
  // the main stream then waits for it.
  auto fill_stage = [&](int j, int nmiss, cudaEvent_t after, cudaEvent_t dst_free, int mlo,
                        bool from_mailbox) -> int {
    if (cudaStreamWaitEvent(c->side, after, 0) != cudaSuccess) return MOE_ERR_CUDA;
    ra.stage = j;
    ra.slots = stage_base(j);
    if (g.fill_mode == MOE_FILL_MEMCPY) {
      {
        Launch l(c, K_MEMCPY, c->side);
        const uint8_t *lbase = static_cast<const uint8_t *>(c->store.base) +
                               (size_t)layer * c->store.layer_stride;
        for (int i = mlo; i < mlo + nmiss; ++i) {
          const MissItem m = c->h_mail_miss[i];
          if (!from_mailbox || m.expert < 0 || m.expert >= E) return MOE_ERR_CUDA;
          if (fill_copy(c, c->d_staging + (size_t)(i - mlo) * c->expert_bytes,
                        lbase + (size_t)m.expert * c->store.expert_stride, c->expert_bytes, c->side) != cudaSuccess)
            return MOE_ERR_CUDA;
        }
      }
      ra.src_base = c->d_staging;
      ra.src_layer_off = 0;
      ra.src_expert_stride = 0;
      ra.src_slot_stride = c->expert_bytes;
      ra.by_expert = 0;
    } else {
      ra.src_base = c->host_dev;
      ra.src_layer_off = (uint64_t)layer * c->store.layer_stride;
      ra.src_expert_stride = c->store.expert_stride;
      ra.src_slot_stride = 0;
      ra.by_expert = 1;
    }
    if (dst_free != after && cudaStreamWaitEvent(c->side, dst_free, 0) != cudaSuccess) return MOE_ERR_CUDA;
    {
      Launch l(c, K_REPACK, c->side);
      if (launch_repack(ra, S, nmiss, c->side) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (cudaEventRecord(c->ev_up[j], c->side) != cudaSuccess ||
        cudaStreamWaitEvent(st, c->ev_up[j], 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  };
  // After a staged call: the blocks the final state maps live in the stage
  // buffers for stages >= 1.  Each slot's last miss (the miss list is in stage
  // order) names the stage whose buffer holds its final block; runs of
  // consecutive slots from the same buffer are copied into the layer's slots
  // in one piece, once stage 0's compute no longer reads the slots.  The main
  // stream waits.
  auto finalize_stages = [&](int n_st, int nM) -> int {
    if (n_st < 2 || !c->d_stage_buf) return MOE_OK;
    std::vector<int> &fin_src = c->fin_src;  // sized S at init
    std::fill(fin_src.begin(), fin_src.end(), 0);
    for (int i = 0; i < nM; ++i) {
      const MissItem m = c->h_mail_miss[i];
      if (m.slot < 0 || m.slot >= S || m.stage < 0 || m.stage >= n_st) return MOE_ERR_CUDA;
      fin_src[m.slot] = m.stage;
    }
    if (cudaStreamWaitEvent(c->side, c->ev_done[0], 0) != cudaSuccess) return MOE_ERR_CUDA;
    const size_t stride = c->lay.stride;
    for (int s0 = 0; s0 < S;) {
      int s1 = s0 + 1;
      while (s1 < S && fin_src[s1] == fin_src[s0]) ++s1;
      if (fin_src[s0] >= 1 &&
          cudaMemcpyAsync(layer_slots + (size_t)s0 * stride, stage_base(fin_src[s0]) + (size_t)s0 * stride,
                          (size_t)(s1 - s0) * stride, cudaMemcpyDeviceToDevice, c->side) != cudaSuccess)
        return MOE_ERR_CUDA;
      s0 = s1;
    }
    if (cudaEventRecord(c->ev_fin, c->side) != cudaSuccess || cudaStreamWaitEvent(st, c->ev_fin, 0) != cudaSuccess)
      return MOE_ERR_CUDA;
    return MOE_OK;
  };

  const bool fused_ok = T <= kTokPerUnit && fused_miss_supported(g.hidden, g.ffn);
  // the decode layer kernel's device waits give up after a quarter of
  // timeout_us (so that a host wait outlasts them), within [1 ms, 2 s]
  const uint64_t decode_wait_ns =
      (uint64_t)std::min<int64_t>(std::max<int64_t>(g.timeout_us / 4, 1000), 2000000) * 1000u;

  // misses of a single-stage call through the fused kernel on the side stream
  // (after `after`), the main stream waiting for it before the combine
  auto fused_stage0 = [&](cudaEvent_t after, int nmiss_max, bool copies) -> int {
    ra.slots = layer_slots;
    if (cudaStreamWaitEvent(c->side, after, 0) != cudaSuccess) return MOE_ERR_CUDA;
    if (g.fill_mode == MOE_FILL_MEMCPY) {
      if (copies) {
        Launch l(c, K_MEMCPY, c->side);
        const uint8_t *lbase = static_cast<const uint8_t *>(c->store.base) +
                               (size_t)layer * c->store.layer_stride;
        for (int i = 0; i < nmiss_max; ++i) {
          const MissItem m = c->h_mail_miss[i];
          if (m.expert < 0 || m.expert >= E) return MOE_ERR_CUDA;
          if (fill_copy(c, c->d_staging + (size_t)i * c->expert_bytes,
                        lbase + (size_t)m.expert * c->store.expert_stride, c->expert_bytes, c->side) != cudaSuccess)
            return MOE_ERR_CUDA;
        }
      }
      ra.src_base = c->d_staging;
      ra.src_layer_off = 0;
      ra.src_expert_stride = 0;
      ra.src_slot_stride = c->expert_bytes;
      ra.by_expert = 0;
    } else {
      ra.src_base = c->host_dev;
      ra.src_layer_off = (uint64_t)layer * c->store.layer_stride;
      ra.src_expert_stride = c->store.expert_stride;
      ra.src_slot_stride = 0;
      ra.by_expert = 1;
    }
    ra.stage = 0;
    {
      Launch l(c, K_FUSED, c->side);
      const int grid = std::max(1, std::min(128, nmiss_max * (g.ffn / 32 + g.hidden / 32)));
      if (launch_fused_miss(fa, ra, c->d_sync, grid, c->side) != cudaSuccess) return MOE_ERR_CUDA;
    }
    if (cudaEventRecord(c->ev_up[0], c->side) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
  };

  if (use_decode) {
    // pull fill, single stage, few tokens: the whole layer in one launch after
    // the plan (misses from the mapped host store, hits from their slots)
    const uint8_t *host_layer = static_cast<const uint8_t *>(c->host_dev) + (size_t)layer * c->store.layer_stride;
    const int inject = c->inject == MOE_INJECT_DECODE_WAIT;
    c->inject = 0;
    MOE_LAUNCH(K_DECODE, launch_decode_layer(fa, host_layer, c->store.expert_stride, nullptr, c->d_w, c->d_gut,
                                             c->d_yt, static_cast<float *>(d_out), c->d_sync, 2 + maxU, T,
                                             c->n_sms, decode_wait_ns, inject, st));
  } else if (use_decode_mc) {
    // memcpy fill, one stage: the decode layer kernel starts on the hits at
    // once; its misses wait, each for its staging block.  The host reads the
    // miss list from the mailbox and, on the side stream, copies each missed
    // block into staging (cudaMemcpyAsync) and then writes the call number
    // into that block's ready word (a stream memory write, fenced after the copy).
    // Nothing between the kernel's launch and the last copy may wait for the
    // device (the kernel waits for the copies): the timing pool is made roomy first.
    tp_reserve(c, 2);
    const int inject = c->inject == MOE_INJECT_DECODE_WAIT;
    c->inject = 0;
    MOE_LAUNCH(K_DECODE, launch_decode_layer(fa, c->d_staging, c->expert_bytes, c->d_miss_ready, c->d_w,
                                             c->d_gut, c->d_yt, static_cast<float *>(d_out), c->d_sync, 2 + maxU,
                                             T, c->n_sms, decode_wait_ns, inject, st));
    int rc = wait_mailbox(c, c->seq, st);
    if (rc != MOE_OK) return poison(c, rc);
    const PlanHdr hdr = c->h_mail->hdr;
    if (hdr.error) return poison(c, MOE_ERR_INVALID_ARG);
    if (hdr.n_stages != 1 || hdr.n_miss > c->staging_blocks) return poison(c, MOE_ERR_CUDA);
    if (hdr.n_miss > 0) {
      // the missed blocks alternate between two side streams, so that a block's
      // copy does not queue behind the previous block's ready-word write
      if (cudaStreamWaitEvent(c->side, c->ev_plan, 0) != cudaSuccess ||
          (hdr.n_miss > 1 && cudaStreamWaitEvent(c->side2, c->ev_plan, 0) != cudaSuccess))
        return poison(c, MOE_ERR_CUDA);
      Launch l(c, K_MEMCPY, c->side);
      const uint8_t *lbase = static_cast<const uint8_t *>(c->store.base) + (size_t)layer * c->store.layer_stride;
      for (int i = 0; i < hdr.n_miss; ++i) {
        const MissItem m = c->h_mail_miss[i];
        if (m.expert < 0 || m.expert >= E) return poison(c, MOE_ERR_CUDA);
        cudaStream_t cs = (i & 1) ? c->side2 : c->side;
        if (fill_copy(c, c->d_staging + (size_t)i * c->expert_bytes,
                      lbase + (size_t)m.expert * c->store.expert_stride, c->expert_bytes, cs) != cudaSuccess ||
            c->write_value32(reinterpret_cast<CUstream>(cs),
                             reinterpret_cast<CUdeviceptr>(c->d_miss_ready + i), hdr.epoch, 0) != CUDA_SUCCESS)
          return poison(c, MOE_ERR_CUDA);
      }
    }
  } else if (!need_host && fused_ok) {
    // pull fill, single stage guaranteed, few tokens: misses read once from the
    // host store and computed on the way; hits computed beside them
    int rc = fused_stage0(c->ev_plan, maxU, false);
    if (rc != MOE_OK) return poison(c, rc);
    MOE_LAUNCH(K_GATEUP, launch_gateup(fa, 0, 0, maxUnits, st));
    MOE_LAUNCH(K_DOWN, launch_down(fa, 0, 0, maxUnits, st));
    if (cudaStreamWaitEvent(st, c->ev_up[0], 0) != cudaSuccess) return poison(c, MOE_ERR_CUDA);
    MOE_LAUNCH(K_COMBINE, launch_combine(c->d_y, c->d_w, c->d_hdr, T, k, g.hidden, d_out, st));
  } else if (!need_host) {
    // pull fill, single stage guaranteed: the fill overlaps the hit gate/up
    MOE_LAUNCH(K_GATEUP, launch_gateup(fa, 0, 0, maxUnits, st));
    int rc = fill_stage(0, maxU, c->ev_plan, c->ev_plan, 0, false);  // main waits for it from here on
    if (rc != MOE_OK) return poison(c, rc);
    MOE_LAUNCH(K_GATEUP, launch_gateup(fa, 1, 0, maxUnits, st));
    if (dc_ok) {
      MOE_LAUNCH(K_DOWN, launch_down_combine(fa, c->d_w, c->d_gpu_slot, T, d_out, st));
    } else {
      MOE_LAUNCH(K_DOWN, launch_down(fa, 2, 0, maxUnits, st));
      MOE_LAUNCH(K_COMBINE, launch_combine(c->d_y, c->d_w, c->d_hdr, T, k, g.hidden, d_out, st));
    }
  } else if (use_gemm) {
    // tensor-core grouped GEMM; stage-0 hits start before the copies are issued
    const int maxG = std::min(c->maxGunits, maxU + (P + kGemmN - 1) / kGemmN + 1);
    const __nv_bfloat16 *xb = static_cast<const __nv_bfloat16 *>(d_x);
    MOE_LAUNCH(K_GATHER, launch_gather_sorted(xb, c->d_perm, P, k, g.hidden, c->d_xs, st));
    MOE_LAUNCH(K_GEMM_GATEUP, launch_gemm_gateup(fa, c->xs_maps, c->slot_maps, layer * S, c->d_gunits,
                                                 c->d_gunit_begin, c->d_h16, 0, 0, maxG, st));
    int rc = wait_mailbox(c, c->seq, st);
    if (rc != MOE_OK) return poison(c, rc);
    const PlanHdr hdr = c->h_mail->hdr;
    if (hdr.error) return poison(c, MOE_ERR_INVALID_ARG);
    const int n_st = hdr.n_stages, n0 = hdr.n_stage0_miss, nM = hdr.n_miss, cap = hdr.stage_cap;
    if (n_st < 1 || n_st > c->maxStages - 1 || cap < 1 || cap > S || n0 < 0 || n0 > nM || nM > c->maxU)
      return poison(c, MOE_ERR_CUDA);
    for (int j = 0; j < n_st; ++j) {
      const int mlo = j == 0 ? 0 : n0 + (j - 1) * cap;
      const int mhi = j == 0 ? n0 : std::min(nM, n0 + j * cap);
      if (mhi > mlo) {
        rc = fill_stage(j, mhi - mlo, c->ev_plan, stage_free(j), mlo, true);
        if (rc != MOE_OK) return poison(c, rc);
      }
      FfnArgs fj = fa;
      fj.slots = stage_base(j);
      // the tensor maps of the slot array stage j reads, and its slot 0 there
      const bool in_layer = j == 0 || !c->d_stage_buf;
      const RawMaps &rm = in_layer ? c->slot_maps : c->stage_maps;
      const int slot0 = in_layer ? layer * S : (j & 1) * S;
      const int sg = std::min(maxG, S + (P + kGemmN - 1) / kGemmN + 1);  // units of one stage, bound
      MOE_LAUNCH(K_GEMM_GATEUP, launch_gemm_gateup(fj, c->xs_maps, rm, slot0, c->d_gunits, c->d_gunit_begin,
                                                   c->d_h16, 1, j, sg, st));
      MOE_LAUNCH(K_GEMM_DOWN,
                 launch_gemm_down(fj, c->h16_maps, rm, slot0, c->d_gunits, c->d_gunit_begin, 2, j, sg, st));
      if (cudaEventRecord(c->ev_done[j], st) != cudaSuccess) return poison(c, MOE_ERR_CUDA);
    }
    rc = finalize_stages(n_st, nM);
    if (rc != MOE_OK) return poison(c, rc);
    MOE_LAUNCH(K_COMBINE, launch_combine(c->d_y, c->d_w, c->d_hdr, T, k, g.hidden, d_out, st));
  } else {
    MOE_LAUNCH(K_GATEUP, launch_gateup(fa, 0, 0, maxUnits, st));
    int rc = wait_mailbox(c, c->seq, st);
    if (rc != MOE_OK) return poison(c, rc);
    const PlanHdr hdr = c->h_mail->hdr;
    if (hdr.error) return poison(c, MOE_ERR_INVALID_ARG);
    const int n_st = hdr.n_stages, n0 = hdr.n_stage0_miss, nM = hdr.n_miss, cap = hdr.stage_cap;
    if (n_st < 1 || n_st > c->maxStages - 1 || cap < 1 || cap > S || n0 < 0 || n0 > nM || nM > c->maxU)
      return poison(c, MOE_ERR_CUDA);
    if (n_st == 1 && fused_ok) {
      if (nM > 0) {
        rc = fused_stage0(c->ev_plan, nM, true);
        if (rc != MOE_OK) return poison(c, rc);
      }
      MOE_LAUNCH(K_DOWN, launch_down(fa, 0, 0, std::max(1, hdr.hit_units), st));
      if (nM > 0 && cudaStreamWaitEvent(st, c->ev_up[0], 0) != cudaSuccess)
        return poison(c, MOE_ERR_CUDA);
      MOE_LAUNCH(K_COMBINE, launch_combine(c->d_y, c->d_w, c->d_hdr, T, k, g.hidden, d_out, st));
    } else {
      for (int j = 0; j < n_st; ++j) {
        const int mlo = j == 0 ? 0 : n0 + (j - 1) * cap;
        const int mhi = j == 0 ? n0 : std::min(nM, n0 + j * cap);
        if (mhi > mlo) {
          rc = fill_stage(j, mhi - mlo, c->ev_plan, stage_free(j), mlo, true);
          if (rc != MOE_OK) return poison(c, rc);
        }
        FfnArgs fj = fa;
        fj.slots = stage_base(j);
        const int ulo = j == 0 ? hdr.hit_units : c->h_mail_ub[j];
        const int uhi = c->h_mail_ub[j + 1];
        if (uhi > ulo) MOE_LAUNCH(K_GATEUP, launch_gateup(fj, 1, j, uhi - ulo, st));
        if (n_st == 1 && dc_ok) {
          MOE_LAUNCH(K_DOWN, launch_down_combine(fj, c->d_w, c->d_gpu_slot, T, d_out, st));
        } else {
          const int dlo = c->h_mail_ub[j];
          if (uhi > dlo) MOE_LAUNCH(K_DOWN, launch_down(fj, 2, j, uhi - dlo, st));
          if (cudaEventRecord(c->ev_done[j], st) != cudaSuccess) return poison(c, MOE_ERR_CUDA);
        }
      }
      rc = finalize_stages(n_st, nM);
      if (rc != MOE_OK) return poison(c, rc);
      if (n_st > 1 || !dc_ok)
        MOE_LAUNCH(K_COMBINE, launch_combine(c->d_y, c->d_w, c->d_hdr, T, k, g.hidden, d_out, st));
    }
  }
#undef MOE_LAUNCH
  c->last_layer = layer;
  c->last_T = T;
  if (c->check_plans) {
    // debug runs: wait for the call, then check its plan and the layer's state
    // on the host (skipped while the stream is being captured)
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    if (cudaStreamIsCapturing(st, &cs) != cudaSuccess) return poison(c, MOE_ERR_CUDA);
    if (cs == cudaStreamCaptureStatusNone) {
      int rc = wait_stream(st, g.timeout_us);
      if (rc == MOE_OK) rc = wait_stream(c->side, g.timeout_us);
      if (rc == MOE_OK && c->side2) rc = wait_stream(c->side2, g.timeout_us);
      if (rc != MOE_OK) return poison(c, rc);
      if (const int de = device_error_code(c)) return poison(c, de);
      PlanHdr h;
      std::vector<int32_t> ids(P), gs(P), sg(P), se(S), es(E);
      std::vector<MissItem> mi(std::max(1, maxU));
      bool ok = cudaMemcpy(&h, c->d_hdr, sizeof(h), cudaMemcpyDeviceToHost) == cudaSuccess &&
                cudaMemcpy(ids.data(), c->d_ids, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess &&
                cudaMemcpy(gs.data(), c->d_gpu_slot, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess &&
                cudaMemcpy(sg.data(), c->d_stage, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess &&
                cudaMemcpy(se.data(), pa.slot_expert, 4 * S, cudaMemcpyDeviceToHost) == cudaSuccess &&
                cudaMemcpy(es.data(), pa.expert_slot, 4 * E, cudaMemcpyDeviceToHost) == cudaSuccess;
      ok = ok && h.n_miss >= 0 && h.n_miss <= maxU &&
           (h.n_miss == 0 ||
            cudaMemcpy(mi.data(), c->d_miss, sizeof(MissItem) * h.n_miss, cudaMemcpyDeviceToHost) == cudaSuccess);
      if (!ok) return poison(c, MOE_ERR_CUDA);
      if (h.error) return poison(c, MOE_ERR_INVALID_ARG);
      if (plan_check(T, k, E, S, h.n_stages, h.n_miss, ids.data(), gs.data(), sg.data(),
                     reinterpret_cast<const int32_t *>(mi.data()), se.data(), es.data()) != 0)
        return poison(c, MOE_ERR_CHECK);
    }
  }
  return MOE_OK;
}

MOE_API int moe_cache_sync(moe_cache *c, void *cuda_stream) {
  if (!c) return MOE_ERR_INVALID_ARG;
  int rc = wait_stream((cudaStream_t)cuda_stream, c->cfg.timeout_us);
  if (rc == MOE_OK) rc = wait_stream(c->side, c->cfg.timeout_us);
  if (rc == MOE_OK && c->side2) rc = wait_stream(c->side2, c->cfg.timeout_us);
  if (rc != MOE_OK) return poison(c, rc);
  if (const int de = device_error_code(c)) return poison(c, de);
  return c->poisoned ? c->last_error : MOE_OK;
}

MOE_API int moe_cache_stats(const moe_cache *cc, int32_t layer, moe_cache_stats_t *out) {
  moe_cache *c = const_cast<moe_cache *>(cc);
  if (!c || !out || layer < -1 || layer >= c->cfg.n_layers) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    poison(c, MOE_ERR_CUDA);
  }
  std::vector<uint64_t> st((size_t)c->cfg.n_layers * kNStat);
  if (cudaMemcpy(st.data(), c->d_stats, sizeof(uint64_t) * st.size(), cudaMemcpyDeviceToHost) !=
      cudaSuccess) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  uint64_t acc[kNStat] = {};
  for (int l = 0; l < c->cfg.n_layers; ++l) {
    if (layer >= 0 && l != layer) continue;
    for (int i = 0; i < kNStat; ++i) acc[i] += st[(size_t)l * kNStat + i];
  }
  out->calls = acc[0];
  out->pick_hits = acc[1];
  out->pick_misses = acc[2];
  out->unique_hits = acc[3];
  out->unique_misses = acc[4];
  out->evictions = acc[5];
  out->bytes_uploaded = acc[6];
  out->stages = acc[7];
  out->staged_calls = acc[8];
  out->bypassed = acc[9];
  if (const int de = device_error_code(c)) poison(c, de);
  out->poisoned = c->poisoned;
  out->last_error = c->last_error;
  out->cuda_error = c->cuda_error;
  out->reserved = 0;
  return MOE_OK;
}

MOE_API int moe_layer_last_plan(const moe_cache *cc, int32_t layer, int32_t *ids, float *w,
                                int32_t *gpu_slot, int32_t *stage, int32_t *miss_expert,
                                int32_t *miss_slot, int32_t *miss_evicted, int32_t *miss_stage,
                                int32_t *n_miss, int32_t *n_stages) {
  moe_cache *c = const_cast<moe_cache *>(cc);
  if (!c || layer != c->last_layer || c->last_T <= 0) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  const size_t P = (size_t)c->last_T * c->cfg.top_k;
  PlanHdr h;
  bool ok = cudaMemcpy(&h, c->d_hdr, sizeof(h), cudaMemcpyDeviceToHost) == cudaSuccess;
  if (ok && ids) ok = cudaMemcpy(ids, c->d_ids, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (ok && w) ok = cudaMemcpy(w, c->d_w, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (ok && gpu_slot) ok = cudaMemcpy(gpu_slot, c->d_gpu_slot, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (ok && stage) ok = cudaMemcpy(stage, c->d_stage, 4 * P, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  if (h.error) return MOE_ERR_INVALID_ARG;
  std::vector<MissItem> m(std::max(1, h.n_miss));
  if (h.n_miss > 0 && cudaMemcpy(m.data(), c->d_miss, sizeof(MissItem) * h.n_miss,
                                 cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  for (int i = 0; i < h.n_miss; ++i) {
    if (miss_expert) miss_expert[i] = m[i].expert;
    if (miss_slot) miss_slot[i] = m[i].slot;
    if (miss_evicted) miss_evicted[i] = m[i].evicted;
    if (miss_stage) miss_stage[i] = m[i].stage;
  }
  if (n_miss) *n_miss = h.n_miss;
  if (n_stages) *n_stages = h.n_stages;
  return MOE_OK;
}

MOE_API int moe_cache_set_timing(moe_cache *c, int32_t enable) {
  if (!c) return MOE_ERR_INVALID_ARG;
  if (enable) {
    tp_flush(c);
    for (int i = 0; i < K_NKINDS; ++i) { c->tp.ms[i] = 0; c->tp.n[i] = 0; }
    c->tp.on = true;
  } else {
    c->tp.on = false;
  }
  return MOE_OK;
}

MOE_API int moe_cache_timing(moe_cache *c, const char **names, uint64_t *launches, double *ms,
                             int32_t cap, int32_t *n) {
  if (!c || cap < 0) return MOE_ERR_INVALID_ARG;
  tp_flush(c);
  int m = std::min(cap, (int)K_NKINDS);
  for (int i = 0; i < m; ++i) {
    if (names) names[i] = kKindNames[i];
    if (launches) launches[i] = c->tp.n[i];
    if (ms) ms[i] = c->tp.ms[i];
  }
  if (n) *n = K_NKINDS;
  return MOE_OK;
}

namespace {

// Copies the blocks named by items (expert, slot) of layer l from the host
// store into their slots: the fill kernel reads the mapped store, or each chunk
// goes through staging when the store has no device mapping.  d_list holds S
// items, d_h one header.  Stream-ordered on st; waits for st after each chunk
// (the host lists are reused).  Returns MOE_OK or MOE_ERR_CUDA.
int fill_layer_slots(moe_cache *c, int l, const std::vector<MissItem> &items, MissItem *d_list, PlanHdr *d_h,
                     cudaStream_t st) {
  const int S = c->cfg.slots_per_layer;
  const int chunk = c->host_dev ? S : std::max(1, c->staging_blocks);
  const int m = (int)items.size();
  const uint8_t *lbase = static_cast<const uint8_t *>(c->store.base) + (size_t)l * c->store.layer_stride;
  for (int lo = 0; lo < m; lo += chunk) {
    const int n = std::min(chunk, m - lo);
    PlanHdr h = {};
    h.n_stages = 1;
    h.n_stage0_miss = n;
    h.n_miss = n;
    h.stage_cap = S;
    RepackArgs ra;
    ra.slots = c->d_slots + (size_t)l * S * c->lay.stride;
    ra.slot_stride = c->lay.stride;
    ra.lay = c->lay;
    ra.miss = d_list;
    ra.hdr = d_h;
    ra.stage = 0;
    bool ok = cudaMemcpyAsync(d_list, items.data() + lo, sizeof(MissItem) * n, cudaMemcpyHostToDevice, st) ==
                  cudaSuccess &&
              cudaMemcpyAsync(d_h, &h, sizeof(PlanHdr), cudaMemcpyHostToDevice, st) == cudaSuccess;
    if (c->host_dev) {
      ra.src_base = c->host_dev;
      ra.src_layer_off = (uint64_t)l * c->store.layer_stride;
      ra.src_expert_stride = c->store.expert_stride;
      ra.src_slot_stride = 0;
      ra.by_expert = 1;
    } else {
      // staging block i holds the chunk's i-th item (the repack reads its
      // source by list position and writes the item's slot)
      for (int i = 0; ok && i < n; ++i)
        ok = fill_copy(c, c->d_staging + (size_t)i * c->expert_bytes,
                       lbase + (size_t)items[lo + i].expert * c->store.expert_stride, c->expert_bytes, st) ==
             cudaSuccess;
      ra.src_base = c->d_staging;
      ra.src_layer_off = 0;
      ra.src_expert_stride = 0;
      ra.src_slot_stride = c->expert_bytes;
      ra.by_expert = 0;
    }
    ok = ok && launch_repack(ra, S, n, st) == cudaSuccess;
    ok = ok && cudaStreamSynchronize(st) == cudaSuccess;
    if (!ok) return MOE_ERR_CUDA;
  }
  return MOE_OK;
}

// Device lists for fill_layer_slots, freed with the object.
struct FillLists {
  MissItem *list = nullptr;
  PlanHdr *hdr = nullptr;
  bool alloc(int S) { return dalloc(&list, (size_t)S) == cudaSuccess && dalloc(&hdr, 1) == cudaSuccess; }
  ~FillLists() {
    cudaFree(list);
    cudaFree(hdr);
  }
};

}  // namespace

MOE_API int moe_cache_preload(moe_cache *c, const uint32_t *counts, void *cuda_stream) {
  if (!c || !counts) return MOE_ERR_INVALID_ARG;
  if (c->poisoned) return MOE_ERR_POISONED;
  const int L = c->cfg.n_layers, E = c->cfg.n_experts, S = c->cfg.slots_per_layer;
  cudaStream_t st = (cudaStream_t)cuda_stream;
  // the new state: per layer the S most-used experts, by (count desc, id asc),
  // in slots 0, 1, ...
  std::vector<int32_t> se((size_t)L * S, -1), es((size_t)L * E, -1);
  FillLists fl;
  if (!fl.alloc(S)) return MOE_ERR_OOM;
  int rc = MOE_OK;
  for (int l = 0; l < L && rc == MOE_OK; ++l) {
    const uint32_t *cnt = counts + (size_t)l * E;
    std::vector<int32_t> order;
    for (int e = 0; e < E; ++e)
      if (cnt[e] > 0) order.push_back(e);
    std::stable_sort(order.begin(), order.end(), [&](int32_t x, int32_t y) { return cnt[x] > cnt[y]; });
    if ((int)order.size() > S) order.resize(S);
    std::vector<MissItem> items;
    for (int i = 0; i < (int)order.size(); ++i) {
      se[(size_t)l * S + i] = order[i];
      es[(size_t)l * E + order[i]] = i;
      items.push_back(MissItem{order[i], i, -1, 0});
    }
    rc = fill_layer_slots(c, l, items, fl.list, fl.hdr, st);
  }
  if (rc == MOE_OK &&
      (cudaMemcpyAsync(c->d_slot_expert, se.data(), sizeof(int32_t) * se.size(), cudaMemcpyHostToDevice, st) !=
           cudaSuccess ||
       cudaMemcpyAsync(c->d_expert_slot, es.data(), sizeof(int32_t) * es.size(), cudaMemcpyHostToDevice, st) !=
           cudaSuccess ||
       cudaMemsetAsync(c->d_slot_stamp, 0, sizeof(uint64_t) * (size_t)L * S, st) != cudaSuccess ||
       cudaStreamSynchronize(st) != cudaSuccess))
    rc = MOE_ERR_CUDA;
  if (rc != MOE_OK) {
    cudaGetLastError();
    return poison(c, rc);
  }
  return MOE_OK;
}

MOE_API int moe_cache_usage(const moe_cache *cc, uint32_t *counts) {
  moe_cache *c = const_cast<moe_cache *>(cc);
  if (!c || !counts) return MOE_ERR_INVALID_ARG;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    poison(c, MOE_ERR_CUDA);
  }
  if (cudaMemcpy(counts, c->d_usage, sizeof(uint32_t) * (size_t)c->cfg.n_layers * c->cfg.n_experts,
                 cudaMemcpyDeviceToHost) != cudaSuccess) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  return MOE_OK;
}

namespace {

// Byte offsets of the arrays of a saved state (see moe_cache_state_header).
struct StateLayout {
  uint64_t clock, stamp, expert, score, usage, total;
  StateLayout(uint64_t L, uint64_t E, uint64_t S) {
    clock = sizeof(moe_cache_state_header);
    stamp = clock + 8 * L;
    expert = stamp + 8 * L * S;
    score = expert + 4 * L * S;
    usage = score + 4 * L * E;
    total = usage + 4 * L * E;
  }
};

}  // namespace

MOE_API int moe_cache_state_size(const moe_cache *c, uint64_t *bytes) {
  if (!c || !bytes) return MOE_ERR_INVALID_ARG;
  *bytes = StateLayout(c->cfg.n_layers, c->cfg.n_experts, c->cfg.slots_per_layer).total;
  return MOE_OK;
}

MOE_API int moe_cache_save_state(const moe_cache *cc, void *buf, uint64_t cap) {
  moe_cache *c = const_cast<moe_cache *>(cc);
  if (!c || !buf) return MOE_ERR_INVALID_ARG;
  const uint64_t L = c->cfg.n_layers, E = c->cfg.n_experts, S = c->cfg.slots_per_layer;
  const StateLayout o(L, E, S);
  if (cap < o.total) return MOE_ERR_INVALID_ARG;
  if (c->poisoned) return MOE_ERR_POISONED;
  if (cudaDeviceSynchronize() != cudaSuccess) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  if (const int de = device_error_code(c)) return poison(c, de);
  uint8_t *b = static_cast<uint8_t *>(buf);
  moe_cache_state_header h = {};
  h.magic = MOE_STATE_MAGIC;
  h.version = MOE_STATE_VERSION;
  h.n_layers = (int32_t)L;
  h.n_experts = (int32_t)E;
  h.slots_per_layer = (int32_t)S;
  h.policy = c->cfg.policy;
  h.expert_bytes = c->expert_bytes;
  h.total_bytes = o.total;
  std::memcpy(b, &h, sizeof(h));
  const bool ok =
      cudaMemcpy(b + o.clock, c->d_clock, 8 * L, cudaMemcpyDeviceToHost) == cudaSuccess &&
      cudaMemcpy(b + o.stamp, c->d_slot_stamp, 8 * L * S, cudaMemcpyDeviceToHost) == cudaSuccess &&
      cudaMemcpy(b + o.expert, c->d_slot_expert, 4 * L * S, cudaMemcpyDeviceToHost) == cudaSuccess &&
      cudaMemcpy(b + o.score, c->d_score, 4 * L * E, cudaMemcpyDeviceToHost) == cudaSuccess &&
      cudaMemcpy(b + o.usage, c->d_usage, 4 * L * E, cudaMemcpyDeviceToHost) == cudaSuccess;
  if (!ok) {
    cudaGetLastError();
    return poison(c, MOE_ERR_CUDA);
  }
  return MOE_OK;
}

MOE_API int moe_cache_load_state(moe_cache *c, const void *buf, uint64_t size, void *cuda_stream) {
  if (!c || !buf || size < sizeof(moe_cache_state_header)) return MOE_ERR_INVALID_ARG;
  if (c->poisoned) return MOE_ERR_POISONED;
  const int L = c->cfg.n_layers, E = c->cfg.n_experts, S = c->cfg.slots_per_layer;
  const StateLayout o(L, E, S);
  const uint8_t *b = static_cast<const uint8_t *>(buf);
  moe_cache_state_header h;
  std::memcpy(&h, b, sizeof(h));
  if (h.magic != MOE_STATE_MAGIC || h.version != MOE_STATE_VERSION || h.n_layers != L || h.n_experts != E ||
      h.slots_per_layer != S || h.expert_bytes != c->expert_bytes || h.total_bytes != o.total || size != o.total)
    return MOE_ERR_INVALID_ARG;
  // copies of the arrays (the buffer need not be aligned)
  std::vector<uint64_t> clock(L), stamp((size_t)L * S);
  std::vector<int32_t> se((size_t)L * S), es((size_t)L * E, -1);
  std::vector<float> score((size_t)L * E);
  std::vector<uint32_t> usage((size_t)L * E);
  std::memcpy(clock.data(), b + o.clock, 8 * clock.size());
  std::memcpy(stamp.data(), b + o.stamp, 8 * stamp.size());
  std::memcpy(se.data(), b + o.expert, 4 * se.size());
  std::memcpy(score.data(), b + o.score, 4 * score.size());
  std::memcpy(usage.data(), b + o.usage, 4 * usage.size());
  for (int l = 0; l < L; ++l) {
    if (clock[l] >= (1ull << 48)) return MOE_ERR_INVALID_ARG;  // stamps are packed below 2^51 in the plan
    for (int s = 0; s < S; ++s) {
      const int32_t e = se[(size_t)l * S + s];
      if (e < -1 || e >= E) return MOE_ERR_INVALID_ARG;
      if (e < 0) continue;
      if (es[(size_t)l * E + e] >= 0 || stamp[(size_t)l * S + s] > clock[l]) return MOE_ERR_INVALID_ARG;
      es[(size_t)l * E + e] = s;
    }
    for (int e = 0; e < E; ++e) {
      const float v = score[(size_t)l * E + e];
      if (!(v >= 0.f) || std::isinf(v)) return MOE_ERR_INVALID_ARG;
    }
  }
  cudaStream_t st = (cudaStream_t)cuda_stream;
  FillLists fl;
  if (!fl.alloc(S)) return MOE_ERR_OOM;
  int rc = MOE_OK;
  for (int l = 0; l < L && rc == MOE_OK; ++l) {
    std::vector<MissItem> items;
    for (int s = 0; s < S; ++s)
      if (se[(size_t)l * S + s] >= 0) items.push_back(MissItem{se[(size_t)l * S + s], s, -1, 0});
    rc = fill_layer_slots(c, l, items, fl.list, fl.hdr, st);
  }
  if (rc == MOE_OK &&
      (cudaMemcpyAsync(c->d_slot_expert, se.data(), 4 * se.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaMemcpyAsync(c->d_expert_slot, es.data(), 4 * es.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaMemcpyAsync(c->d_slot_stamp, stamp.data(), 8 * stamp.size(), cudaMemcpyHostToDevice, st) !=
           cudaSuccess ||
       cudaMemcpyAsync(c->d_clock, clock.data(), 8 * clock.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaMemcpyAsync(c->d_score, score.data(), 4 * score.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaMemcpyAsync(c->d_usage, usage.data(), 4 * usage.size(), cudaMemcpyHostToDevice, st) != cudaSuccess ||
       cudaStreamSynchronize(st) != cudaSuccess))
    rc = MOE_ERR_CUDA;
  if (rc != MOE_OK) {
    cudaGetLastError();
    return poison(c, rc);
  }
  return MOE_OK;
}

MOE_API int moe_cache_inject(moe_cache *c, int32_t what) {
  if (!c) return MOE_ERR_INVALID_ARG;
  const int code = what & 0xFF, n = what >> 8;
  if (what == 0) {
    c->inject = 0;
    c->copy_fail_in = 0;
  } else if (what == MOE_INJECT_DECODE_WAIT) {
    c->inject = what;
  } else if (code == MOE_INJECT_MEMCPY_FAIL && n >= 0) {
    c->copy_fail_in = n == 0 ? 1 : n;
  } else {
    return MOE_ERR_INVALID_ARG;
  }
  return MOE_OK;
}

MOE_API int moe_cache_probe_h2d(moe_cache *c, int32_t iters, double *gbps) {
  if (!c || iters < 1 || !gbps) return MOE_ERR_INVALID_ARG;
  if (c->poisoned) return MOE_ERR_POISONED;
  cudaEvent_t a, b;
  if (cudaEventCreate(&a) != cudaSuccess || cudaEventCreate(&b) != cudaSuccess) return MOE_ERR_CUDA;
  std::vector<double> v;
  const uint8_t *base = static_cast<const uint8_t *>(c->store.base);
  int rc = MOE_OK;
  // one untimed pass over the same blocks first (first-touch effects), then timed
  for (int i = 0; i < 2 * iters && rc == MOE_OK; ++i) {
    const int e = i % iters % c->cfg.n_experts;
    cudaEventRecord(a, c->side);
    if (cudaMemcpyAsync(c->d_staging, base + (size_t)e * c->store.expert_stride, c->expert_bytes,
                        cudaMemcpyHostToDevice, c->side) != cudaSuccess) {
      rc = MOE_ERR_CUDA;
      break;
    }
    cudaEventRecord(b, c->side);
    rc = wait_stream(c->side, c->cfg.timeout_us);
    float ms = 0.f;
    if (i >= iters && rc == MOE_OK && cudaEventElapsedTime(&ms, a, b) == cudaSuccess && ms > 0.f)
      v.push_back((double)c->expert_bytes / (ms * 1e-3) / 1e9);
  }
  cudaEventDestroy(a);
  cudaEventDestroy(b);
  if (rc != MOE_OK) return poison(c, rc);
  if (v.empty()) return MOE_ERR_CUDA;
  std::sort(v.begin(), v.end());
  *gbps = v[v.size() / 2];
  return MOE_OK;
}

MOE_API uint64_t moe_cache_launch_count(const moe_cache *c) {
  return c ? c->launches.load(std::memory_order_relaxed) : 0;
}

MOE_API void moe_cache_destroy(moe_cache *c) {
  if (!c) return;
  cudaDeviceSynchronize();
  cudaGetLastError();
  free_all(c);
  delete c;
}
