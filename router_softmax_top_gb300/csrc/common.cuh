// Internal declarations shared by the library's translation units (not part
// of the C ABI).
#pragma once

#include <atomic>
#include <cuda.h>  // CUtensorMap (types only; the encoder is fetched from the driver)
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace moe {

// ---------------------------------------------------------------- limits
constexpr int kMaxExperts = 1024;
constexpr int kMaxTopK = 32;
constexpr int kPlanThreads = 256;
constexpr int kNStat = 10;  // calls, pick_hits, pick_misses, unique_hits, unique_misses,
                            // evictions, bytes_uploaded, stages, staged_calls, bypassed
constexpr int kTokPerUnit = 8;  // tokens of one expert handled by one GEMV work unit
constexpr int kGemmN = 128;     // routed pairs of one expert per tensor-core GEMM tile

// ------------------------------------------------------------ plan records
// Header of one call's plan, written by the plan kernel into device scratch and
// mirrored into the host mailbox.
struct PlanHdr {
  int32_t error;      // 0 ok, 1 non-finite logit (state untouched)
  int32_t n_unique;   // |U|
  int32_t n_hits;     // cached before the call
  int32_t n_miss;     // uploads
  int32_t n_stage0_miss;
  int32_t n_stages;
  int32_t n_units;    // GEMV work units (all stages)
  int32_t n_evict;
  int32_t pick_hits;
  int32_t pick_misses;
  int32_t hit_units;  // GEMV units of the stage-0 hits: [0, hit_units)
  int32_t hit_gunits; // GEMM units of the stage-0 hits: [0, hit_gunits)
  uint32_t epoch;     // call number of the handle (1, 2, ...): tags the decode layer kernel's outputs
  int32_t stage_cap;  // misses per stage after stage 0 (the last may hold fewer): S, or fewer
                      // under the adopt policy
  int32_t pad[2];
};

// A work item = one distinct expert of the call.  Items are ordered: stage-0
// hits (ascending expert), then misses in stage order (ascending expert; under
// the adopt policy a staged call's misses lowest rank first).
struct WorkItem {
  int32_t expert;
  int32_t slot;
  int32_t stage;
  int32_t is_miss;
  int32_t pair_begin;  // into perm
  int32_t pair_count;
};

// A GEMV work unit = up to kTokPerUnit pairs of one work item.  Units follow
// the item order, so each stage's units (and stage 0's hit units) are a range.
struct WorkUnit {
  int32_t item;
  int32_t pair_begin;  // into perm
  int32_t pair_count;
  int32_t stage;
};

struct MissItem {
  int32_t expert;
  int32_t slot;
  int32_t evicted;
  int32_t stage;
};

// Host-visible mailbox (pinned, mapped) filled by the plan kernel at its end.
// Followed in memory by int32 unit_begin[stage_cap] (units of stage j are
// [unit_begin[j], unit_begin[j+1])) and MissItem miss[max distinct experts].
struct Mailbox {
  volatile uint32_t seq;  // written last
  int32_t pad[3];
  PlanHdr hdr;
};

// ------------------------------------------------ repacked slot layout
// Each matrix of R rows x C columns (nb = C/32 blocks per row) is stored as a
// nibble plane followed by a scale plane, both ordered by 32-row tiles:
//   nibbles: [R/32 tiles][nb blocks][32 rows][16 bytes]
//   scales:  [R/32 tiles][nb blocks][32 rows] fp16
// so one tile of 32 rows is two contiguous regions (nb*512 and nb*64 bytes)
// that a single bulk copy each brings into shared memory, and the 32 rows of
// one block are 512 consecutive bytes (one 16-byte load per lane).  The 16
// nibble bytes of a block keep their canonical order.
__host__ __device__ inline uint64_t tile_elem(int r, int b, int nb) {
  return ((uint64_t)(r >> 5) * nb + b) * 32 + (r & 31);
}

struct MatLayout {
  uint64_t nib_off, sc_off;  // byte offsets inside the slot
  int32_t rows, nb;
};

struct SlotLayout {
  MatLayout gate, up, down;
  uint64_t bytes;   // = canonical expert bytes
  uint64_t stride;  // slot stride in device memory (bytes, 256-aligned)
};

inline SlotLayout make_slot_layout(int H, int F) {
  SlotLayout s;
  uint64_t mg = (uint64_t)F * (H / 32);
  uint64_t md = (uint64_t)H * (F / 32);
  s.gate = {0, mg * 16, F, H / 32};
  s.up = {mg * 18, mg * 18 + mg * 16, F, H / 32};
  s.down = {2 * mg * 18, 2 * mg * 18 + md * 16, H, F / 32};
  s.bytes = 2 * mg * 18 + md * 18;
  s.stride = (s.bytes + 255) / 256 * 256;
  return s;
}

// The dynamic shared memory limit a kernel has been raised to, per device
// (the attribute belongs to the kernel on each device).
struct DynSmemLimit {
  static constexpr int kDevices = 64;
  std::atomic<size_t> bytes[kDevices] = {};
};

// Raise a kernel's dynamic shared memory limit on the current device to
// `bytes` when needed (the limit plus the kernel's static shared memory must
// stay within the opt-in maximum, so it is raised to what a launch needs, not
// to the maximum).
template <typename Kern>
inline cudaError_t ensure_dyn_smem(Kern kernel, size_t bytes, DynSmemLimit &limit) {
  if (bytes <= 48 * 1024) return cudaSuccess;
  int dev = -1;
  const cudaError_t ge = cudaGetDevice(&dev);
  if (ge != cudaSuccess) return ge;
  std::atomic<size_t> *cur = (dev >= 0 && dev < DynSmemLimit::kDevices) ? &limit.bytes[dev] : nullptr;
  if (cur && bytes <= cur->load(std::memory_order_relaxed)) return cudaSuccess;
  const cudaError_t e =
      cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
  if (e == cudaSuccess && cur) {
    size_t seen = cur->load(std::memory_order_relaxed);
    while (seen < bytes && !cur->compare_exchange_weak(seen, bytes, std::memory_order_relaxed)) {
    }
  }
  return e;
}

// ------------------------------------------------------------ launchers
struct PlanArgs {
  const float *logits;  // [T, E]
  int T, E, k, S, weight_mode;
  // per-layer state
  int32_t *slot_expert;  // [S]
  int32_t *expert_slot;  // [E]
  uint64_t *slot_stamp;  // [S]
  uint64_t *clock;       // [1]
  uint64_t *stats;       // [kNStat]
  uint32_t *usage;       // [E] lifetime activation counts: + picks per expert of every accepted call
  uint64_t expert_bytes;
  // per-call outputs
  int32_t *ids;       // [T*k]
  float *w;           // [T*k]
  int32_t *gpu_slot;  // [T*k]
  int32_t *stage;     // [T*k]
  int32_t *perm;      // [T*k] pair ids grouped by work item
  WorkItem *items;    // [min(E, T*k)]
  WorkUnit *units;    // [min(E,T*k) + T*k/kTokPerUnit + 1]
  int32_t *unit_begin;  // [n_stages + 1] (capacity min(E,T*k) + 2)
  WorkUnit *gunits;     // GEMM units (up to kGemmN pairs of one item), item order
  int32_t *gunit_begin; // [n_stages + 1]
  MissItem *miss;     // [min(E, T*k)]
  PlanHdr *hdr;
  int32_t *err_flag;  // sticky device error word of the handle
  int32_t *sync;      // per-call counters, the first sync_n zeroed here
  int sync_n;
  int32_t *route_bad; // device word for the grid router's non-finite flag (zero between calls)
  int routed;         // set by launch_plan when route_kernel produced ids and w
  Mailbox *mailbox;   // device alias of the mapped host mailbox, or null
  int mailbox_stage_cap;  // capacity of the mailbox's unit_begin array
  uint32_t seq;
  uint32_t *epoch;    // the handle's call counter (device), advanced by every accepted call
  int policy;         // 0 LRU, 1 decayed score with admission (plan_small_kernel only),
                      // 2 LRU whose staged calls keep their most-used experts (plan_kernel)
  int admit_budget;   // policy 1: admissions per call, 0 = no limit
  float *score;       // policy 1: the layer's decayed usage scores [E] (fp32)
  int n_sticky;       // policy 1: occupied slots of highest score that may not be evicted
};
bool plan_small_ok(int T, int E, int k, int S);

cudaError_t launch_plan(const PlanArgs &a, cudaStream_t st);
size_t plan_smem_bytes(int E, int S);

struct FfnArgs {
  const uint8_t *slots;  // layer's slot 0
  uint64_t slot_stride;
  SlotLayout lay;
  int H, F, k;
  const void *x;  // [T, H] fp32 or bf16
  int x_bf16;
  const int32_t *perm;
  const WorkItem *items;
  const WorkUnit *units;
  const int32_t *unit_begin;
  const PlanHdr *hdr;
  float *h;  // [T*k, F]
  float *y;  // [T*k, H]
  int max_tok;  // largest pair count of one work unit this call can have (<= kTokPerUnit)
  int32_t *err;  // mapped error word: set on a device-side failure
};

// Units [unit_lo, unit_hi) are read from unit_begin on the device:
// range_kind 0: stage-0 hit units; 1: stage `stage` units that are misses;
// 2: all units of stage `stage`.
cudaError_t launch_gateup(const FfnArgs &a, int range_kind, int stage, int max_units,
                          cudaStream_t st);
cudaError_t launch_down(const FfnArgs &a, int range_kind, int stage, int max_units,
                        cudaStream_t st);
cudaError_t launch_combine(const float *y, const float *w, const PlanHdr *hdr, int T, int k,
                           int H, float *out, cudaStream_t st);
// Down projection of all picks of each token plus the weighted sum, for calls
// that run in one stage (out[T, H] written directly).
cudaError_t launch_down_combine(const FfnArgs &a, const float *w, const int32_t *gpu_slot, int T,
                                float *out, cudaStream_t st);
bool down_combine_supported(int F, int k);

struct RepackArgs {
  const uint8_t *src_base;  // canonical source: staging (device) or mapped host store
  uint64_t src_layer_off;   // host store: layer offset; staging: 0
  uint64_t src_expert_stride;  // host store: expert stride; staging: 0 (use src_slot_stride)
  uint64_t src_slot_stride;    // staging: bytes per staged block
  int by_expert;               // 1: source indexed by expert id; 0: by miss index in stage
  uint8_t *slots;
  uint64_t slot_stride;
  SlotLayout lay;
  const MissItem *miss;
  const PlanHdr *hdr;
  int stage;  // misses of this stage
};
cudaError_t launch_repack(const RepackArgs &a, int S, int max_miss, cudaStream_t st);
// Misses of a single-stage call of at most 8 tokens: fill + gate/up + down in
// one kernel (y of the miss pairs written to FfnArgs::y).  sync: per-call
// counters zeroed by the plan kernel ([0] queue head, [1 + m] per miss).
cudaError_t launch_fused_miss(const FfnArgs &a, const RepackArgs &r, int32_t *sync, int grid,
                              cudaStream_t st);
bool fused_miss_supported(int H, int F);
// Tensor-core grouped GEMM (bf16 activations).  The activations of the routed
// pairs are first copied into pair-sorted order (xs[pos] = x[perm[pos] / k]),
// so that the rows of one GEMM unit are contiguous and a TMA tensor copy loads
// them; gate/up writes h16 in the same sorted order, and down writes y by pair.
// GemmMaps: 2-D tensor maps (bf16, [rows][K], 128-byte swizzle) over one
// sorted buffer, with boxes of 64 columns x 16, 32, 64 and 128 rows.
struct GemmMaps {
  CUtensorMap box[4];
};
cudaError_t make_gemm_maps(const __nv_bfloat16 *base, int K, int rows, GemmMaps *out);
// RawMaps: the slot planes of an array of n_slots slots (tiled layout) as
// 32-bit-word tensors, so that one TMA copy brings a GEMM chunk (2 blocks of 4
// consecutive 32-row tiles) of gate and up, or of down:
//   gu_nib [slot][mat 2][tile][block][128 words]  box {128, 2, 4, 2, 1}
//   gu_sc  [slot][mat 2][tile][block][16 words]   box {16, 2, 4, 2, 1}
//   dn_nib [slot][tile][block][128 words]         box {128, 2, 4, 1}
//   dn_sc  [slot][tile][block][16 words]          box {16, 2, 4, 1}
// (tiles past the matrix read as zeros).
struct RawMaps {
  CUtensorMap gu_nib, gu_sc, dn_nib, dn_sc;
};
cudaError_t make_raw_maps(const uint8_t *base, int n_slots, uint64_t slot_stride, const SlotLayout &lay,
                          RawMaps *out);
cudaError_t launch_gather_sorted(const __nv_bfloat16 *x, const int32_t *perm, int P, int k, int H,
                                 __nv_bfloat16 *xs, cudaStream_t st);
// raw, slot0: the maps of the slot array that holds a.slots, and the index of
// a.slots' slot 0 in it
cudaError_t launch_gemm_gateup(const FfnArgs &a, const GemmMaps &xs_maps, const RawMaps &raw, int slot0,
                               const WorkUnit *gunits, const int32_t *gunit_begin, __nv_bfloat16 *h16s,
                               int range_kind, int stage, int max_gunits, cudaStream_t st);
cudaError_t launch_gemm_down(const FfnArgs &a, const GemmMaps &h16s_maps, const RawMaps &raw, int slot0,
                             const WorkUnit *gunits, const int32_t *gunit_begin, int range_kind, int stage,
                             int max_gunits, cudaStream_t st);

// Whole expert FFN + combine of a single-stage call of at most 8 tokens with the
// pull fill, in one persistent launch (misses read from the mapped host store
// and written into their slots on the way).
bool decode_layer_supported(int H, int F, int T);
// gu: tagged gate then up outputs (2 x T*k rows of F), yt: tagged down outputs
// (T*k rows of H); sync: [0], [1] queue heads, [2] abort word, [cbase + t*H/32 + r]
// picks done of token t, row tile r (zeroed by the plan)
// host_layer, expert_stride: where missed blocks are read (the layer's experts in
// the mapped host store, or the staging buffer with miss_ready set: block r of
// staging holds miss r once miss_ready[r] carries the call number).
// wait_ns: limit of every bounded device wait; inject: down items wait for a
// gate value that is never written (fault injection: the limit ends the wait)
cudaError_t launch_decode_layer(const FfnArgs &a, const uint8_t *host_layer, uint64_t expert_stride,
                                const uint32_t *miss_ready, const float *w, uint64_t *gu, uint64_t *yt, float *out,
                                int32_t *sync, int cbase, int T, int n_sms, uint64_t wait_ns, int inject,
                                cudaStream_t st);

enum KernelKind { K_PLAN = 0, K_REPACK, K_GATEUP, K_DOWN, K_COMBINE, K_GEMM_GATEUP, K_GEMM_DOWN,
                  K_GATHER, K_MEMCPY, K_FUSED, K_DECODE, K_NKINDS };

}  // namespace moe
