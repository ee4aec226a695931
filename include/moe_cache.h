/*
 * moe_cache.h — C ABI of the routed Mixture-of-Experts layer over a
 * GPU-resident expert-slot cache (one GB300 GPU, sm_103a).
 *
 * What one layer call computes (sources, by page title and section):
 *  1. Router: the top-k experts of each token and their weights
 *     ("llama.cpp + MoE expert cache", "The idea: cache the hot experts on the
 *     GPU", step 1).  Top-k of the raw fp32 logits, descending, ties to the lower
 *     expert id; weight = softmax probability over all E experts
 *     (weight_mode 0) or renormalised over the chosen k (weight_mode 1).
 *  2. Slot table, -1 = not cached (same section, step 2), kept per layer with
 *     least-recently-used replacement under a fixed budget of slots
 *     ("Longhaul MoE loading", opening paragraph).  The call's experts are
 *     planned as one batch: experts it needs are never evicted by it, and each
 *     distinct expert is loaded at most once (same page, the paragraph on
 *     expert IDs planned as a batch).
 *  3. Missing experts are copied from the host store into their slots
 *     ("llama.cpp + MoE expert cache", "Keeping the cache fresh": a slot is
 *     published only after its copy completes).
 *  4. Each (token, expert) pair is computed exactly once from its slot
 *     (same page, "The idea", step 3): Q4_0 SwiGLU FFN, h = silu(W_gate x) *
 *     (W_up x), y = W_down h ("Limitations": merged gate/up, SiLU).
 *  5. Weighted sum out_t = sum_k w[t,k] y[t,k], ascending k ("The idea", step 4).
 *  If one call needs more distinct experts than there are slots, the call runs
 *  in stages and the partial results are summed ("Longhaul MoE loading", the
 *  paragraph on --ubatch-size and stages).
 *
 * Weights: Q4_0, 18 bytes per 32 values ("Multi-GPU LLM Calculator: VRAM Split
 * and RAM Offload", "Memory placement"): fp16 scale d (little-endian), then 16
 * bytes whose low nibbles are values 0..15 and high nibbles values 16..31,
 * w = (q - 8) * d.  One expert block = [gate: F rows x H/32 blocks]
 * [up: F rows x H/32 blocks][down: H rows x F/32 blocks], rows row-major
 * (row r = output feature r, blocks along the input dimension).
 *
 * Conventions for every entry point:
 *  - Return value: MOE_OK (0) or one of the MOE_ERR_* codes; nothing else
 *    crosses the ABI (no exceptions, no aborts).
 *  - "device" pointers are CUDA device memory owned by the caller; "host"
 *    pointers are ordinary host memory owned by the caller.
 *  - Work is stream-ordered on the caller's stream; results are valid when that
 *    stream reaches the end of the call.  A handle serves one stream/thread at a
 *    time (not re-entrant).
 *  - After an error detected during a call (a CUDA error, a non-finite logit, a
 *    timeout) the handle is poisoned: later forward calls return
 *    MOE_ERR_POISONED; stats remain readable; destroy still frees everything.
 */
#ifndef MOE_CACHE_H
#define MOE_CACHE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define MOE_OK 0
#define MOE_ERR_INVALID_ARG 1   /* bad argument or config; non-finite logit      */
#define MOE_ERR_CUDA 2          /* a CUDA runtime call failed                     */
#define MOE_ERR_OOM 3           /* device or pinned allocation failed             */
#define MOE_ERR_TIMEOUT 4       /* a bounded host or device wait gave up          */
#define MOE_ERR_HOST_STORE 5    /* host store invalid or could not be registered  */
#define MOE_ERR_POISONED 6      /* an earlier call on this handle failed          */
#define MOE_ERR_UNSUPPORTED 7   /* shape outside what the kernels implement       */
#define MOE_ERR_CHECK 8         /* debug runs (MOE_CHECK_PLANS=1 at init): a
                                   call's plan or the layer's slot table failed
                                   the host-side consistency check               */

/* Slot replacement policy.
 * MOE_POLICY_LRU: every miss takes a slot; victims are empty slots, then the
 *   least recently used slots whose expert the call does not pick.
 * MOE_POLICY_SCORE ("Keeping the cache fresh": a decayed usage score per
 *   expert, x0.9 per token; a miss that scores higher than the weakest slot is
 *   promoted, up to a budget of copies): per layer, token by token every
 *   expert's score is multiplied by 0.9 and each picked expert gains 1 (fp32).
 *   Misses, strongest first (score descending, then lower id), take an empty
 *   slot if any, else the weakest slot whose expert the call does not pick
 *   (score ascending, then lower index) if their score is strictly higher,
 *   while admit_budget lasts; other misses are bypassed: computed from the host
 *   store like any miss but not cached (miss_slot -1, counted in `bypassed`).
 *   With sticky_permille p (Fork A's option to never evict the most-used share
 *   of each layer's slots), once the call's scores are updated the
 *   floor(p x slots_per_layer / 1000) occupied slots with the highest scores
 *   (ties to the lower index) are not evictable in that call.
 *   Needs every call to fit one stage and the decode layer kernel: max_tokens x
 *   top_k <= min(slots_per_layer, 32), max_tokens <= 8, no tensor-core GEMM
 *   (gemm_min_tokens 0 or > max_tokens), and the pull fill or the memcpy fill
 *   with stream memory writes; otherwise init returns MOE_ERR_UNSUPPORTED.
 * MOE_POLICY_ADOPT ("Prefill preheat": a long prompt's most-used experts stay
 *   in the cache in place of cached experts it used less): LRU, except for
 *   calls of more than one stage.  There rank = (picks in the call descending,
 *   expert id ascending); misses are taken lowest rank first, so the most-used
 *   ones stream last; stage 0 as LRU; with m misses after stage 0 and
 *   G = ceil(m / S) later stages (as many as LRU), the S - C slots whose
 *   stage-0 expert ranks highest (C = ceil(m / G)) keep it, and the other C
 *   slots, in ascending index, take the later misses in turn.  Same uploads,
 *   stages and outputs as LRU; the call ends holding higher-ranked experts. */
#define MOE_POLICY_LRU 0
#define MOE_POLICY_SCORE 1
#define MOE_POLICY_ADOPT 2

/* How misses reach their slots. */
#define MOE_FILL_MEMCPY 0  /* cudaMemcpyAsync per missed block on a side stream into a
                              staging area, overlapped with hit compute; then a device
                              repack into the slot */
#define MOE_FILL_PULL 1    /* a kernel reads the missed blocks straight from the pinned,
                              mapped host store and writes the slot (no host round trip) */

typedef struct moe_cache moe_cache;

typedef struct {
    int32_t n_layers;        /* L >= 1                                             */
    int32_t n_experts;       /* E, 1..1024                                         */
    int32_t top_k;           /* k, 1..min(E, 32)                                   */
    int32_t hidden;          /* H, multiple of 64, <= 16384                        */
    int32_t ffn;             /* F, multiple of 64, <= 16384                        */
    int32_t slots_per_layer; /* S, 1..E: the per-layer budget of device slots      */
    int32_t max_tokens;      /* largest n_tokens of any call, >= 1                 */
    int32_t weight_mode;     /* 0: softmax over all E (default); 1: over chosen k  */
    int32_t act_dtype;       /* 0: x is fp32 [T,H]; 1: x is bf16 [T,H]             */
    int32_t fill_mode;       /* MOE_FILL_MEMCPY or MOE_FILL_PULL                   */
    int32_t gemm_min_tokens; /* calls with n_tokens >= this use the tensor-core
                                grouped GEMM (bf16 activations only); 0 = never.
                                Shorter calls take the GEMV kernels.  Measured
                                on GB300 (hidden 2816, FFN 704, top-8, 32
                                slots): GEMV ahead up to 8 tokens, even at
                                12-16, GEMM ahead from 24; 16 is the switch   */
    int32_t policy;          /* slot replacement: MOE_POLICY_LRU (0),
                                MOE_POLICY_SCORE (1) or MOE_POLICY_ADOPT (2),
                                see above                                         */
    int32_t admit_budget;    /* MOE_POLICY_SCORE: admissions per call, 0 = no limit */
    int32_t sticky_permille; /* MOE_POLICY_SCORE: per mille of the slots, highest
                                scores first, that a call may not evict (0-1000;
                                0 = none; must be 0 under the other policies)      */
    int64_t timeout_us;      /* limit of every bounded host wait, > 0; the decode
                                layer kernel's device waits use a quarter of it,
                                clamped to [1 ms, 2 s] (other kernels: 2 s)        */
} moe_cache_config;

typedef struct {
    const void *base;        /* host memory holding canonical Q4_0 expert blocks   */
    uint64_t bytes;          /* size of the region at base                         */
    uint64_t layer_stride;   /* bytes between layer l and l+1                      */
    uint64_t expert_stride;  /* bytes between expert e and e+1 of one layer        */
} moe_host_store;

typedef struct {
    uint64_t calls;          /* forward calls that reached planning                */
    uint64_t pick_hits;      /* (token, pick) pairs whose expert was cached before */
    uint64_t pick_misses;
    uint64_t unique_hits;    /* distinct experts of a call already cached          */
    uint64_t unique_misses;  /* distinct experts uploaded (= uploads)              */
    uint64_t evictions;      /* uploads that replaced a cached expert              */
    uint64_t bytes_uploaded; /* unique_misses x expert block bytes                 */
    uint64_t stages;         /* sum over calls of the number of stages             */
    uint64_t staged_calls;   /* calls that needed more than one stage              */
    uint64_t bypassed;       /* misses computed without taking a slot (policy 1)   */
    int32_t poisoned;        /* 1 once a call on the handle has failed             */
    int32_t last_error;      /* the code that poisoned it (or MOE_OK)              */
    int32_t cuda_error;      /* the cudaError_t behind MOE_ERR_CUDA (0 if none)     */
    int32_t reserved;
} moe_cache_stats_t;

/*
 * Create a cache: per layer a fixed budget of slots_per_layer device slots,
 * managed least-recently-used, for a model whose expert weights do not all fit
 * ("Longhaul MoE loading", opening paragraph: a per-layer LRU cache of expert
 * slots under a fixed budget), over a host-resident store of every expert
 * ("llama.cpp + MoE expert cache", "The idea: cache the hot experts on the
 * GPU": the full expert set stays in host RAM, a subset is cached on the GPU).
 * cfg and store are read during the call only.
 * The host store must stay valid and unchanged until moe_cache_destroy.  If it
 * is not page-locked already, it is registered (cudaHostRegister, mapped) here
 * and unregistered at destroy; failure -> MOE_ERR_HOST_STORE.  Every (layer,
 * expert) block [base + l*layer_stride + e*expert_stride, + block bytes) must
 * lie inside [base, base + bytes).
 * The library allocates the slots (L x S blocks, repacked), the per-layer
 * state, the per-call scratch for max_tokens, a side stream and events.
 * cuda_stream: stream for the initial state set-up (NULL = legacy default).
 * *out receives the handle (NULL on error).
 */
int moe_cache_init(const moe_cache_config *cfg, const moe_host_store *store,
                   void *cuda_stream, moe_cache **out);

/*
 * One routed-MoE layer call (steps 1-5 above, staged when needed).
 * d_logits: device fp32 [n_tokens, E] row-major.
 * d_x:      device [n_tokens, H] row-major, fp32 or bf16 per cfg.act_dtype.
 * d_out:    device fp32 [n_tokens, H] row-major, overwritten.
 * n_tokens == 0: no-op, MOE_OK.  n_tokens > max_tokens or layer out of range:
 * MOE_ERR_INVALID_ARG.  A non-finite logit: MOE_ERR_INVALID_ARG, the layer's
 * state is left as it was and the handle is poisoned (with MOE_FILL_PULL the
 * check completes on the device; it is reported by the next call, by
 * moe_cache_sync or by moe_cache_stats).
 * Buffers must not alias each other.
 */
int moe_layer_forward(moe_cache *c, int32_t layer, const float *d_logits, const void *d_x,
                      int32_t n_tokens, float *d_out, void *cuda_stream);

/*
 * Wait (bounded by cfg.timeout_us) for the handle's outstanding work on
 * cuda_stream and its side stream, then report any error raised on the device.
 */
int moe_cache_sync(moe_cache *c, void *cuda_stream);

/* Counters of one layer, or the sum over all layers for layer == -1 (host out;
 * synchronises with the device).  The hit rate of the pages is the share of
 * routed picks whose expert was already cached, pick_hits / (pick_hits +
 * pick_misses) ("llama.cpp + MoE expert cache", "The idea: cache the hot
 * experts on the GPU": 70-80% of a token's expert picks were cached ones);
 * unique_* count distinct experts per call, unique_misses = uploads. */
int moe_cache_stats(const moe_cache *c, int32_t layer, moe_cache_stats_t *out);

/*
 * Test hook: the plan of the most recent forward call, which must have been on
 * `layer` (else MOE_ERR_INVALID_ARG).  All outputs are host arrays, any may be
 * NULL: ids/gpu_slot/stage [n_tokens*k], w [n_tokens*k] (fp32 router weights),
 * miss_* [n_miss] in ascending expert order (evicted = -1 for an empty slot),
 * n_miss, n_stages.  Synchronises with the device.
 */
int moe_layer_last_plan(const moe_cache *c, int32_t layer, int32_t *ids, float *w,
                        int32_t *gpu_slot, int32_t *stage, int32_t *miss_expert,
                        int32_t *miss_slot, int32_t *miss_evicted, int32_t *miss_stage,
                        int32_t *n_miss, int32_t *n_stages);

/*
 * Warm start from a usage profile ("Persistent hot experts": each layer's
 * most-used experts are preloaded before the first request).  counts: host
 * array [n_layers][n_experts] of usage counts (e.g. saved from an earlier
 * session).  Per layer, the experts with a non-zero count, by (count
 * descending, id ascending), the first slots_per_layer of them are copied from
 * the host store into slots 0, 1, ...; every other slot becomes empty; the
 * layer's recency stamps become 0.  The call counter, the scores of
 * MOE_POLICY_SCORE and the statistics do not change.  Stream-ordered on
 * cuda_stream (between calls, not during one) and synchronises with it before
 * returning.  NULL handle or counts: MOE_ERR_INVALID_ARG; a poisoned handle:
 * MOE_ERR_POISONED; CUDA failures poison the handle (MOE_ERR_CUDA).
 */
int moe_cache_preload(moe_cache *c, const uint32_t *counts, void *cuda_stream);

/*
 * Lifetime activation counts ("llama.cpp: fork with multi gpu acceleration
 * ...", "Persistent hot experts": the cache keeps how often each expert was
 * used, an n_layer x n_expert u32 array, saves it at shutdown and preloads the
 * most-used experts at the next start).  counts: host array
 * [n_layers][n_experts]; counts[l][e] = routed (token, pick) pairs of expert e
 * in layer l over every accepted forward call since init (or since the state
 * the handle was loaded from), whatever their slot outcome (hit, miss,
 * bypass); u32, wrapping.  The array is a valid `counts` for
 * moe_cache_preload.  Synchronises with the device; readable on a poisoned
 * handle.  NULL handle or counts: MOE_ERR_INVALID_ARG.
 */
int moe_cache_usage(const moe_cache *c, uint32_t *counts);

/*
 * Saved cache state.  The pages persist usage counts only; resuming the slot
 * tables themselves has no counterpart there: a handle that loads a state
 * plans its next calls exactly as the saved handle would have.  Layout, host
 * byte order, L = n_layers, S = slots_per_layer, E = n_experts:
 *   moe_cache_state_header          48 bytes
 *   uint64_t clock[L]               calls planned per layer
 *   uint64_t slot_stamp[L][S]       each slot's last use, a value of its clock
 *   int32_t  slot_expert[L][S]      expert held by each slot, -1 = empty
 *   float    score[L][E]            decayed usage scores (MOE_POLICY_SCORE)
 *   uint32_t usage[L][E]            lifetime activation counts
 * Slot contents are not saved: loading copies each held expert's block from
 * the handle's host store into its slot.
 */
#define MOE_STATE_MAGIC 0x53454F4Du /* "MOES" */
#define MOE_STATE_VERSION 1u
typedef struct {
  uint32_t magic, version;
  int32_t n_layers, n_experts, slots_per_layer;
  int32_t policy;         /* the saving handle's policy (not checked on load) */
  uint64_t expert_bytes;  /* bytes of one expert block (checked on load) */
  uint64_t total_bytes;   /* header + arrays */
  uint64_t reserved;      /* 0 */
} moe_cache_state_header;

/* Bytes of this handle's saved state.  NULL argument: MOE_ERR_INVALID_ARG. */
int moe_cache_state_size(const moe_cache *c, uint64_t *bytes);

/*
 * Writes the state into buf (host, cap bytes).  Includes every call issued
 * before it (synchronises with the device).  cap below moe_cache_state_size:
 * MOE_ERR_INVALID_ARG, nothing written; a poisoned handle: MOE_ERR_POISONED
 * (a failed call may have left the tables half-updated).
 */
int moe_cache_save_state(const moe_cache *c, void *buf, uint64_t cap);

/*
 * Replaces every layer's slot table, stamps, clock, scores and usage counts by
 * a saved state (host buf, size bytes) and fills the held slots from the host
 * store.  Stream-ordered on cuda_stream, between calls as for
 * moe_cache_preload, and synchronises with it before returning; statistics
 * and the call counter do not change.  Rejected with MOE_ERR_INVALID_ARG, the
 * handle unchanged: wrong magic, version or size; another shape (layers,
 * experts, slots, expert bytes); an expert id outside [-1, E) or one expert in
 * two slots of a layer; an occupied slot stamped after its layer's clock; a
 * clock of 2^48 or more (the decode plan orders slots by stamps packed below
 * 2^51; a handle reaches such a clock only after 2^48 calls of one layer); a
 * negative or non-finite score.  A poisoned handle: MOE_ERR_POISONED.  CUDA
 * failures while filling poison the handle (MOE_ERR_CUDA).
 */
int moe_cache_load_state(moe_cache *c, const void *buf, uint64_t size, void *cuda_stream);

/*
 * Debug runs: with MOE_CHECK_PLANS=1 in the environment when a handle is
 * created, every forward call on it waits for its own completion (not while
 * the stream is being captured) and checks on the host that its plan and the
 * layer's slot table are consistent: ids in [0, E) and distinct per token,
 * slots in [-1, S), stages and miss records in range, no expert in two slots,
 * each pair's expert in the slot its plan names.  A failed check poisons the
 * handle with MOE_ERR_CHECK.
 *
 * Test hook: fault injection without a GPU fault.  what = MOE_INJECT_DECODE_WAIT
 * makes the next call that runs the decode layer kernel (pull fill, one stage,
 * <= 8 tokens) wait, in its down items, for a gate value carrying a call number
 * that is never written: the wait can only end by its limit (timeout_us / 4,
 * clamped as above), after which the kernel ends every other wait, finishes,
 * and records the failure; the next forward or sync returns MOE_ERR_TIMEOUT and
 * the handle is poisoned.  what = 0 clears a pending injection.  Returns
 * MOE_ERR_INVALID_ARG for an unknown `what`.
 */
#define MOE_INJECT_DECODE_WAIT 1
/* what = MOE_INJECT_MEMCPY_FAIL | (n << 8), n >= 1 (0 reads as 1): the n-th next
 * host-to-device copy of a missed block (memcpy fill, preload through staging)
 * fails before it is issued, as a refused copy would.  The call that meets it
 * returns MOE_ERR_CUDA and poisons the handle (stats stay readable, cuda_error
 * reads cudaErrorUnknown); kernels of that call already launched finish, those
 * waiting for the missing block by their bounded wait. */
#define MOE_INJECT_MEMCPY_FAIL 2
int moe_cache_inject(moe_cache *c, int32_t what);

/*
 * Per-kernel timing with CUDA events on the streams the kernels run on.
 * enable = 1 starts recording (resets the totals), 0 stops.  moe_cache_timing
 * fills, for up to `cap` kernel kinds, the name (static string), the number of
 * launches and the summed device milliseconds; returns the number of kinds in
 * *n.  Synchronises with the device.
 */
int moe_cache_set_timing(moe_cache *c, int32_t enable);
int moe_cache_timing(moe_cache *c, const char **names, uint64_t *launches, double *ms,
                     int32_t cap, int32_t *n);

/*
 * Measured host->device bandwidth of one expert block: `iters` cudaMemcpyAsync
 * of one block from the pinned store into the staging area on the side stream,
 * each timed with events; *gbps receives the median in GB/s (1e9 B/s).
 */
int moe_cache_probe_h2d(moe_cache *c, int32_t iters, double *gbps);

/* Bytes of one expert block (3 * F * H / 32 * 18) and of one device slot. */
uint64_t moe_expert_bytes(int32_t hidden, int32_t ffn);

/*
 * One expert's Q4_0 SwiGLU FFN on up to 8 tokens, allocating nothing.
 * (No counterpart on the pages: an addition for callers that cannot allocate.)
 * Callers that cannot call cudaMalloc -- code inside a CUDA graph being
 * captured, real-time or signal-handling paths that must not block on an
 * allocator, plugins that do not own the process's memory pool -- pass their
 * inputs and outputs and get y without any per-call or per-handle allocation:
 * the only intermediate (h, the tokens' SwiGLU activations, and two work
 * counters) lives in a fixed array compiled into the library, 128 KiB + 256 B
 * on every GPU that loads it, held until the process exits.
 *   d_expert_block: one canonical expert block [gate | up | down] (layout as
 *                   above), in device memory or mapped pinned host memory,
 *                   16-byte aligned, 3 * ffn * hidden / 32 * 18 bytes.
 *   d_x: device fp32 [n_tokens, hidden]; d_y: device fp32 [n_tokens, hidden],
 *        overwritten with y_t = W_down (silu(W_gate x_t) * (W_up x_t)).
 * Limits: 0 <= n_tokens <= 8 (0 = no-op), hidden and ffn multiples of 64 and
 * <= 4096; beyond them MOE_ERR_UNSUPPORTED.  Null or misaligned pointers:
 * MOE_ERR_INVALID_ARG.  Stream-ordered on cuda_stream.
 * All calls on a device share the fixed array and its contents persist between
 * calls (the counters are cleared at the start of each call): calls that
 * overlap on the GPU race and must be serialised by the caller.  The first
 * call on each device looks up the array's device address (with that device
 * current), and the first call in the process page-locks a 64 KiB status page
 * compiled into the library (no allocation); make that first call before any
 * stream capture.
 * Failures on the device: each down tile waits, bounded (2 s), for the call's
 * gate/up tiles.  If that wait gives up, the tile's rows of d_y become NaN for
 * every token and the failure is recorded; the first call issued after the
 * failed kernel has finished returns MOE_ERR_TIMEOUT without launching
 * anything, and clears the record.
 * Cost: when hidden or ffn is large (e.g. 4096 and 1536 at 8 tokens) the
 * tokens' inputs are staged in groups that fit shared memory, and each group
 * decodes the weight tiles again.
 */
int moe_expert_ffn_static(const void *d_expert_block, int32_t hidden, int32_t ffn,
                          const float *d_x, int32_t n_tokens, float *d_y, void *cuda_stream);

/* Number of kernel launches the library issued since init (all streams). */
uint64_t moe_cache_launch_count(const moe_cache *c);

/* Free everything the handle owns (waits for its outstanding work first). */
void moe_cache_destroy(moe_cache *c);

/* Static description of a return code. */
const char *moe_strerror(int code);

#ifdef __cplusplus
}
#endif
#endif /* MOE_CACHE_H */
