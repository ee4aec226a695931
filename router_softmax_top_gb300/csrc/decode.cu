// Decode layer kernel: the whole expert FFN and the weighted combine of one
// single-stage layer call of at most 8 tokens in one persistent launch, for
// the pull fill (the host store is read in place through its mapped address).
//
// Missed experts are read once from the host store over the host link and
// written into their slots on the way ("Multi-GPU LLM Calculator: VRAM Split
// and RAM Offload", "RAM offload": weights stream from host RAM when they do
// not fit); cached experts are read from their slots in HBM; both are computed
// by the same CTAs.  Work items are 32-row tiles of gate or of up, and groups
// of up to 2 consecutive 32-row tiles of down, of one expert.  Two queues hold
// them in dependency order: misses (gate/up tiles, then down groups) and hits
// (likewise).  When the call has misses, 48 CTAs serve the miss queue, each
// with one item at a time, so the host link is busy from the start and no
// compute of a miss CTA runs beside its own copy from the host; they then turn
// to the hit queue.  The other CTAs serve the hit queue only, so that no hit
// waits in a ring behind a copy from the host.  A down group needs the gate/up tiles of
// its expert, which come earlier in the same queue; a CTA claims items only
// while it runs, processes them in claim order, and takes from its second
// queue only once its first is exhausted, so every waited-for tile is held by
// a running CTA that reaches it.  Each CTA keeps its next items loading (bulk
// copies, a producer warp) while its compute warps work.
//
// Outputs that other CTAs read (gate, up and down rows) are stored as 64-bit
// words: the fp32 value and the number of the call that wrote it.  A reader
// polls each word until it carries this call's number, so no producer fences
// its stores (a GPU-scope fence would also wait for the CTA's copies in flight
// on the host link) and a down group starts on block b of h as soon as the
// gate and up values of that block exist: each warp forms h = silu(g) * u of
// its own blocks, with the same expression the other kernels use.
// The weighted sum over a token's picks is done by whichever down tile of
// that token and row tile is counted last (a per-(token, tile) counter): it
// adds the k down rows in ascending pick order ("The idea: cache the hot
// experts on the GPU", step 4).  Every value is reduced in the canonical order
// of the Q4_0 GEMV kernels, so results are bitwise those of the
// tile-GEMV + combine path.
#include "q4_math.cuh"

namespace moe {
namespace {

using namespace q4;

constexpr int kPubSlots = 4;
// per CTA: GROUPS groups of 8 compute warps (each group works on its own
// items), a producer warp and a publisher warp
__host__ __device__ constexpr int decode_threads(int groups) { return groups * kThreads + 64; }
constexpr int kHitQueue = 1 << 30;                 // claim code flag: item of the hit queue
constexpr int kMissCtas = 48;                      // CTAs that serve the miss queue first
constexpr int kMaxDG = 4;                          // 32-row down tiles per down item, at most
constexpr int kMissDG = 2;                         // ... of the miss queue, at most
constexpr int kHitDG = 2;                          // ... of the hit queue, at most

struct DecodeJob {
  const uint8_t *host;     // device alias of this layer's experts in the mapped host store, or
                           // the staging buffer (miss_ready set)
  uint64_t expert_stride;  // bytes between experts in the store (between blocks in staging)
  const uint32_t *miss_ready;  // staging mode: [r] carries the call number once miss r's block
                               // has landed in staging block r (copied from the host by the
                               // copy engine); null: misses read from the mapped store
  uint8_t *slots;          // layer's slot 0
  uint64_t slot_stride;
  SlotLayout lay;
  const PlanHdr *hdr;
  const WorkItem *items;   // hits [0, nH), then misses
  const int32_t *perm;
  const float *w;
  const void *x;
  int x_bf16;
  int T, k, H, F;
  int DG;                  // 32-row down tiles per down item (1, 2 or 4)
  uint64_t *g, *u;         // [T*k, F] tagged gate and up outputs
  uint64_t *y;             // [T*k, H] tagged down outputs
  float *out;              // [T, H]
  int32_t *sync;           // [0] miss queue head, [1] hit queue head, [2] abort word (a wait gave
                           // up), [cbase + t * H/32 + r] picks done of token t, row tile r
  int cbase;
  uint64_t wait_ns;        // limit of every bounded wait
  int inject;              // down items wait for a gate value that is never written
  int32_t *err;
};

__device__ __forceinline__ uint64_t now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Tagged values: the fp32 bits in the low word, the call number in the high word.
__device__ __forceinline__ void st_tagged(uint64_t *p, float v, uint32_t ep) {
  const uint64_t w = ((uint64_t)ep << 32) | __float_as_uint(v);
  asm volatile("st.relaxed.gpu.global.b64 [%0], %1;" ::"l"(p), "l"(w) : "memory");
}
__device__ __forceinline__ uint64_t ld_tagged(const uint64_t *p) {
  uint64_t w;
  asm volatile("ld.relaxed.gpu.global.b64 %0, [%1];" : "=l"(w) : "l"(p) : "memory");
  return w;
}
__device__ __forceinline__ int ld_relaxed(const int32_t *p) {
  int v;
  asm volatile("ld.relaxed.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Value at p once it carries call number ep.  Bounded: gives up after
// limit_ns, or soon after any CTA has given up (the abort word), and then
// returns false.
__device__ __forceinline__ bool wait_tagged(const uint64_t *p, uint32_t ep, int32_t *abort_word, float &v,
                                            uint64_t limit_ns) {
  uint64_t w = ld_tagged(p);
  uint64_t t0 = 0;
  for (uint32_t i = 0; (uint32_t)(w >> 32) != ep; ++i) {
    if ((i & 31u) == 31u) {
      const uint64_t t = now_ns();
      if (t0 == 0) t0 = t;
      if (ld_relaxed(abort_word) || t - t0 > limit_ns || i >= kSpinLimit) {
        atomicExch(abort_word, 1);
        v = 0.f;
        return false;
      }
    }
    __nanosleep(128);  // a poll is an L2 round trip: keep the request rate low
    w = ld_tagged(p);
  }
  v = __uint_as_float((uint32_t)w);
  return true;
}

// Inputs are staged with each 32-value block interleaved: value j at position
// 2j for j < 16, 2(j - 16) + 1 otherwise, so that values j and 16 + j sit side
// by side for the paired FMA below.
__device__ __forceinline__ int ilv(int j) { return ((j & 15) << 1) | (j >> 4); }
__device__ __forceinline__ unsigned long long pack2(float lo, float hi) {
  unsigned long long r;
  asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
  return r;
}
__device__ __forceinline__ unsigned long long ffma2(unsigned long long a, unsigned long long b,
                                                    unsigned long long c) {
  unsigned long long d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
// dot32 over an interleaved block: the two partial sums (values 0..15 and
// 16..31, each in ascending order) advance together in one paired FMA per
// step, then are added: bitwise the canonical dot32.
__device__ __forceinline__ float dot32_ilv(const float f[32], const float *xi) {
  unsigned long long s = 0ull;
#pragma unroll
  for (int i = 0; i < 16; i += 2) {
    const float4 a = *reinterpret_cast<const float4 *>(xi + 2 * i);  // x[i], x[16+i], x[i+1], x[17+i]
    s = ffma2(pack2(f[i], f[16 + i]), pack2(a.x, a.y), s);
    s = ffma2(pack2(f[i + 1], f[17 + i]), pack2(a.z, a.w), s);
  }
  float lo, hi;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(s));
  return lo + hi;
}

// A claimed item: work item, matrix (0 gate, 1 up, 2 down), first 32-row tile
// and number of tiles, source.
struct Work {
  int iu, mat, tile, nt;
  bool miss;
};
struct QueueShape {
  int nH, nM, tF, tH;
  int DGh, dGh, DGm, dGm;  // per queue (hits, misses): 32-row tiles per down item, down items per expert
  __device__ int misses() const { return nM * (2 * tF + dGm); }
  __device__ int hits() const { return nH * (2 * tF + dGh); }
};
// Queue position -> item.  Each queue: all gate/up tiles, then all down groups.
__device__ __forceinline__ Work decode_claim(int code, const QueueShape &q) {
  Work w;
  const bool hitq = code & kHitQueue;
  const int pos = code & (kHitQueue - 1);
  const int n_exp = hitq ? q.nH : q.nM, base = hitq ? 0 : q.nH;
  const int A = n_exp * 2 * q.tF;
  w.miss = !hitq;
  if (pos < A) {
    w.iu = base + pos / (2 * q.tF);
    const int r = pos % (2 * q.tF);
    w.mat = r / q.tF;
    w.tile = r % q.tF;
    w.nt = 1;
  } else {
    const int i = pos - A;
    const int DG = hitq ? q.DGh : q.DGm, dG = hitq ? q.dGh : q.dGm;
    w.iu = base + i / dG;
    w.mat = 2;
    w.tile = (i % dG) * DG;
    w.nt = min(DG, q.tH - w.tile);
  }
  return w;
}

__host__ __device__ inline size_t decode_slot_bytes(int H, int F, int DG) {
  const size_t gu = (size_t)32 * (H / 32) * 18, dn = (size_t)DG * 32 * (F / 32) * 18;
  return gu > dn ? gu : dn;  // canonical and tiled forms have the same size
}
// Down tiles per item: the most of 4, 2, 1 whose bytes fit a gate/up tile's
// (one is always allowed).
int decode_down_group(int H, int F) {
  const size_t gu = (size_t)32 * (H / 32) * 18, dn = (size_t)32 * (F / 32) * 18;
  for (int g = 4; g > 1; g /= 2)
    if (g * dn <= gu) return g;
  return 1;
}
// shared memory: NB ring slots, the call's inputs [T][H] and their block sums,
// and per compute group one down item's inputs [T][F] and the warp partials
// [8][T][32] (rounded to 32 floats: each group's inputs are read with 16-byte loads)
__host__ __device__ inline size_t decode_group_floats(int F, int T) {
  const size_t n = (size_t)T * F + (size_t)kWarps * T * 32;
  return (n + 31) / 32 * 32;
}
size_t decode_smem(int H, int F, int T, int NB, int groups) {
  return (size_t)NB * decode_slot_bytes(H, F, decode_down_group(H, F)) +
         sizeof(float) * ((size_t)T * H + (size_t)T * (H / 32) + (size_t)groups * decode_group_floats(F, T));
}
constexpr size_t kDecodeSmemCap = 226 * 1024;

// Compute warps (0-7) synchronise among themselves with a named barrier; the
// producer (warp 8) and publisher (warp 9) run beside them on mbarriers.
__device__ __forceinline__ void group_sync(int group) {
  asm volatile("bar.sync %0, %1;" ::"r"(1 + group), "n"(kThreads) : "memory");
}
template <int GROUPS>
__device__ __forceinline__ void all_compute_sync() {
  asm volatile("bar.sync 3, %0;" ::"n"(GROUPS * kThreads) : "memory");
}

__device__ __forceinline__ bool ring_wait(uint64_t *bar, uint32_t parity, uint64_t limit_ns) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      const uint64_t t = now_ns();
      if (t0 == 0) t0 = t;
      else if (t - t0 > limit_ns) return false;
    }
  }
  return false;
}

// Block b of row `row` of the item's tiles (row = 32 * tile-in-item + lane):
// nibbles and scale bits; a miss also writes the block's tiled form into its
// slot (fill on the way), unless it has none (a bypassed miss).
__device__ __forceinline__ void load_block(const unsigned char *buf, bool miss, int nt, int row, int b, int nb,
                                           uint8_t *slot, const MatLayout &L, int tile0, uint4 &qv,
                                           unsigned short &db) {
  if (miss) {
    qv = canon_block(buf, row, b, nb, db);
    if (slot) {
      const uint64_t e = tile_elem(tile0 * 32 + row, b, nb);
      reinterpret_cast<uint4 *>(slot + L.nib_off)[e] = qv;
      reinterpret_cast<unsigned short *>(slot + L.sc_off)[e] = db;
    }
  } else {
    const int i = ((row >> 5) * nb + b) * 32 + (row & 31);
    qv = reinterpret_cast<const uint4 *>(buf)[i];
    db = reinterpret_cast<const unsigned short *>(buf + (size_t)nt * nb * 512)[i];
  }
}

// Launched as a programmatic dependent of the plan kernel: everything before
// griddepcontrol.wait (barriers, the staged inputs) overlaps the plan; nothing
// the plan writes is read before it.  Only after it (the plan complete) may
// the next call's plan kernel, a programmatic dependent of this grid, start
// its prologue (which reads the counters this call's plan wrote).
__device__ __forceinline__ void wait_plan() {
  asm volatile("griddepcontrol.wait;" ::: "memory");
  asm volatile("griddepcontrol.launch_dependents;");
}

template <int NB, int TMAX, int GROUPS>
__global__ void __launch_bounds__(decode_threads(GROUPS), 1) decode_layer_kernel(const DecodeJob j) {
  const PlanHdr *hd = j.hdr;
  QueueShape qs;
  qs.nH = 0;
  qs.nM = 0;
  qs.tF = j.F / 32;
  qs.tH = j.H / 32;
  qs.DGh = min(j.DG, kHitDG);
  qs.dGh = (qs.tH + qs.DGh - 1) / qs.DGh;
  qs.DGm = min(j.DG, kMissDG);
  qs.dGm = (qs.tH + qs.DGm - 1) / qs.DGm;
  const int T = j.T, nbH = j.H / 32, tH = qs.tH;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const size_t slot_bytes = decode_slot_bytes(j.H, j.F, j.DG);

  extern __shared__ __align__(128) unsigned char sm[];
  unsigned char *ring = sm;
  float *xs = reinterpret_cast<float *>(sm + NB * slot_bytes);  // [T][H]: the call's inputs
  float *xsum = xs + (size_t)T * j.H;                           // [T][H/32]
  float *gbase = xsum + (size_t)T * nbH;                        // per compute group, below
  __shared__ __align__(8) uint64_t full[NB], empty[NB], pub[kPubSlots], pubfree[kPubSlots];
  __shared__ int s_item[NB], s_pub[kPubSlots];
  // each ring slot's work item and its pairs' rows (perm), written by the
  // producer with the claim, and the same handed on to the publisher: no
  // compute or combine step waits for a round trip to fetch them
  __shared__ WorkItem s_work[NB];
  __shared__ int s_prow[NB][TMAX], s_pub_n[kPubSlots], s_pub_prow[kPubSlots][TMAX];
  __shared__ int s_grow[GROUPS][TMAX];  // the current item's pair rows, per compute group
  __shared__ int s_ok[GROUPS];  // decisions of a group's thread 0, read after a barrier

  auto mat_of = [&](int mat) -> const MatLayout & {
    return mat == 0 ? j.lay.gate : mat == 1 ? j.lay.up : j.lay.down;
  };
  if (tid == 0) {
    for (int s = 0; s < NB; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    for (int p = 0; p < kPubSlots; ++p) {
      mbar_init(&pub[p], kThreads);
      mbar_init(&pubfree[p], 1);
    }
    fence_mbar_init();
    for (int g = 0; g < GROUPS; ++g) s_ok[g] = 1;
  }
  __syncthreads();

  if (warp == GROUPS * kWarps) {
    // ---- producer: claim items in order, bulk-copy each one's tiles into the ring
    wait_plan();
    if (hd->error) return;
    qs.nH = hd->n_hits;
    qs.nM = hd->n_stage0_miss;
    const uint32_t ep = hd->epoch;
    if (lane == 0) {
      // miss CTAs serve the miss queue, then help with the hits; hit CTAs serve
      // the hit queue only.  A miss CTA claims one item at a time: the next
      // claim waits until the compute warps have issued every store of the
      // previous item, so no copy from the host is in flight while they compute
      // (their stores would queue behind it), and a hit item taken after a
      // miss is never queued behind it
      const int n_miss_ctas = qs.nM ? min((int)gridDim.x / 3, kMissCtas) : 0;
      const bool hit_first = (int)blockIdx.x >= n_miss_ctas;
      bool second = false, prev_miss = false;
      for (int c = 0;; ++c) {
        const int s = c % NB;
        if (c >= NB && !ring_wait(&empty[s], (uint32_t)((c / NB) - 1) & 1u, j.wait_ns)) {
          // the compute warps stopped: no copy may still be landing when the CTA exits
          flag_error(j.err, 3);
          for (int c2 = c - NB; c2 < c; ++c2) (void)ring_wait(&full[c2 % NB], (uint32_t)(c2 / NB) & 1u, j.wait_ns);
          break;
        }
        bool gate_ok = true, waited = false;
        int code = -1;
        for (;;) {
          const bool hitq = hit_first != second;
          if (c >= 1 && (!hitq || prev_miss) && !waited) {
            const int c2 = c - 1;
            waited = true;
            gate_ok = ring_wait(&pub[c2 % kPubSlots], (uint32_t)(c2 / kPubSlots) & 1u, j.wait_ns);
            if (!gate_ok) {
              flag_error(j.err, 3);
              break;
            }
          }
          const int size = hitq ? qs.hits() : qs.misses();
          const int pos = size > 0 ? atomicAdd(&j.sync[hitq ? 1 : 0], 1) : size;
          if (pos < size) {
            code = pos | (hitq ? kHitQueue : 0);
            prev_miss = !hitq;
            break;
          }
          if (second || hit_first) break;
          second = true;
        }
        if (code < 0) {
          // the end of the list, once for each compute group
          for (int c2 = c; c2 < c + GROUPS; ++c2) {
            const int s2 = c2 % NB;
            if (c2 > c && c2 >= NB && !ring_wait(&empty[s2], (uint32_t)((c2 / NB) - 1) & 1u, j.wait_ns)) break;
            s_item[s2] = -1;
            mbar_arrive(&full[s2]);
          }
          break;
        }
        s_item[s] = code;
        const Work wk = decode_claim(code, qs);
        const WorkItem it = j.items[wk.iu];
        const MatLayout &L = mat_of(wk.mat);
        const int nb = L.nb;
        unsigned char *dst = ring + (size_t)s * slot_bytes;
        if (wk.miss) {
          // canonical rows [32 tile, 32 (tile + nt)) of the matrix: one contiguous run,
          // from the mapped store, or from staging block r once it has landed
          uint64_t src = (uint64_t)it.expert;
          if (j.miss_ready) {
            const int r = wk.iu - qs.nH;
            src = (uint64_t)r;
            uint64_t t0 = 0;
            for (uint32_t i = 0; (uint32_t)ld_acquire(reinterpret_cast<const int32_t *>(j.miss_ready + r)) != ep; ++i) {
              __nanosleep(256);
              if ((i & 15u) == 15u) {
                const uint64_t t = now_ns();
                if (t0 == 0) t0 = t;
                if (ld_relaxed(j.sync + 2) || t - t0 > j.wait_ns || i >= kSpinLimit) {
                  atomicExch(j.sync + 2, 1);
                  flag_error(j.err, 3);
                  break;
                }
              }
            }
          }
          const uint32_t bytes = (uint32_t)(32 * nb * 18);
          mbar_expect_tx_only(&full[s], bytes * wk.nt);
          bulk_g2s(dst, j.host + src * j.expert_stride + L.nib_off + (uint64_t)wk.tile * bytes, bytes * wk.nt,
                   &full[s]);
        } else {
          // tiled slot planes: nibbles [tiles][nb][32][16 B], then scales [tiles][nb][32]
          const uint8_t *slot = j.slots + (uint64_t)it.slot * j.slot_stride;
          const uint32_t bn = (uint32_t)nb * 512, bs = (uint32_t)nb * 64;
          mbar_expect_tx_only(&full[s], (bn + bs) * wk.nt);
          bulk_g2s(dst, slot + L.nib_off + (uint64_t)wk.tile * bn, bn * wk.nt, &full[s]);
          bulk_g2s(dst + (size_t)bn * wk.nt, slot + L.sc_off + (uint64_t)wk.tile * bs, bs * wk.nt, &full[s]);
        }
        // while the tiles are in flight: the item and its pairs' rows, then the
        // arrival that (with the bytes) completes the slot's phase
        s_work[s] = it;
#pragma unroll
        for (int q = 0; q < TMAX; ++q) s_prow[s][q] = q < it.pair_count ? j.perm[it.pair_begin + q] : 0;
        mbar_arrive(&full[s]);
      }
    }
    return;
  }

  if (warp == GROUPS * kWarps + 1) {
    // ---- publisher: counts each down item's rows per (token, row tile); the
    // last one counted does that tile's weighted sum
    wait_plan();
    if (hd->error) return;
    qs.nH = hd->n_hits;
    qs.nM = hd->n_stage0_miss;
    const uint32_t ep = hd->epoch;
    // lane q holds the router weight of pick q of token t in wreg[t] (k <= 32)
    float wreg[TMAX];
#pragma unroll
    for (int t = 0; t < TMAX; ++t) wreg[t] = (t < j.T && lane < j.k) ? j.w[t * j.k + lane] : 0.f;
    for (int c = 0;; ++c) {
      const int p = c % kPubSlots;
      int ok = 1;
      if (lane == 0) ok = ring_wait(&pub[p], (uint32_t)(c / kPubSlots) & 1u, j.wait_ns) ? 1 : 0;
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) {
        if (lane == 0) flag_error(j.err, 3);
        break;
      }
      (void)mbar_try_wait(&pub[p], (uint32_t)(c / kPubSlots) & 1u);  // completed phase: acquire
      const int code = s_pub[p];
      const int pc = s_pub_n[p];  // the item's pairs
      const int prq = lane < TMAX ? s_pub_prow[p][lane] : 0;  // lane q: row of the item's pair q
      __syncwarp();
      if (lane == 0) mbar_arrive(&pubfree[p]);
      if (code < 0) break;
      const Work wk = decode_claim(code, qs);
      if (wk.mat == 2) {
        // bit (tt * 8 + i): pick i of this item completed row tile tile + tt.
        // One counter per lane, all in flight together; meanwhile the first
        // two combinations' first 8 down rows are loaded on speculation (the
        // common single-token case: the tail of the call is then one round trip)
        const int ncomb = wk.nt * pc;
        const int tl = __shfl_sync(0xffffffffu, prq, lane % pc) / j.k;
        int old = -1;
        if (lane < ncomb) old = atomicAdd(&j.sync[j.cbase + tl * tH + wk.tile + lane / pc], 1);
        uint64_t spec[2][8];
#pragma unroll
        for (int c2 = 0; c2 < 2; ++c2)
          if (c2 < ncomb) {
            const int t = __shfl_sync(0xffffffffu, prq, c2 % pc) / j.k, r = (wk.tile + c2 / pc) * 32 + lane;
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2)
              if (i2 < j.k) spec[c2][i2] = ld_tagged(j.y + ((size_t)t * j.k + i2) * j.H + r);
          }
        const unsigned last = __ballot_sync(0xffffffffu, old == j.k - 1);
        // weighted sum over the picks of each completed (token, row tile), ascending
        for (int c2 = 0; c2 < ncomb; ++c2) {
          if (!(last >> c2 & 1u)) continue;
          const int t = __shfl_sync(0xffffffffu, prq, c2 % pc) / j.k, r = (wk.tile + c2 / pc) * 32 + lane;
          float wt = wreg[0];
#pragma unroll
          for (int tt = 1; tt < TMAX; ++tt)
            if (t == tt) wt = wreg[tt];
          float o = 0.f;
          bool yok = true;
          // the k rows' words 8 at a time, all in flight together; one that does
          // not carry this call's number yet is polled
          for (int q0 = 0; q0 < j.k; q0 += 8) {
            uint64_t yw[8];
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2)
              if (q0 + i2 < j.k) {
                if (q0 == 0 && c2 < 2) yw[i2] = c2 == 0 ? spec[0][i2] : spec[1][i2];
                else yw[i2] = ld_tagged(j.y + ((size_t)t * j.k + q0 + i2) * j.H + r);
              }
#pragma unroll
            for (int i2 = 0; i2 < 8; ++i2)
              if (q0 + i2 < j.k) {
                const float wq = __shfl_sync(0xffffffffu, wt, q0 + i2);
                float yv = __uint_as_float((uint32_t)yw[i2]);
                if ((uint32_t)(yw[i2] >> 32) != ep)
                  yok = wait_tagged(j.y + ((size_t)t * j.k + q0 + i2) * j.H + r, ep, j.sync + 2, yv, j.wait_ns) && yok;
                o = fmaf(wq, yv, o);
              }
          }
          if (!yok) flag_error(j.err, 3);
          j.out[(size_t)t * j.H + r] = o;
        }
      }
    }
    return;
  }

  // ---- compute warps: the call's inputs once (the staging of stage_rows),
  // blocks interleaved
  for (int t = 0; t < T; ++t) {
    float *dst = xs + (size_t)t * j.H;
    if (j.x_bf16) {
      const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(j.x) + (size_t)t * j.H;
      for (int c = tid; c < j.H; c += GROUPS * kThreads) dst[(c & ~31) + ilv(c & 31)] = __bfloat162float(src[c]);
    } else {
      const float4 *src = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(j.x) + (size_t)t * j.H);
      for (int c = tid; c < j.H / 4; c += GROUPS * kThreads) {
        const float4 v = src[c];
        const int e = 4 * c, base = e & ~31, jj = e & 31;
        dst[base + ilv(jj)] = v.x;
        dst[base + ilv(jj + 1)] = v.y;
        dst[base + ilv(jj + 2)] = v.z;
        dst[base + ilv(jj + 3)] = v.w;
      }
    }
  }
  all_compute_sync<GROUPS>();
  for (int i = warp; i < T * nbH; i += GROUPS * kWarps) {
    float v = xs[(size_t)i * 32 + ilv(lane)];  // lane j holds value j
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) xsum[i] = v;
  }
  all_compute_sync<GROUPS>();
  // this warp's group, and its thread and warp index within the group
  const int group = warp / kWarps;
  const int gtid = tid - group * kThreads;
  const int gwarp = warp - group * kWarps;
  float *hs = gbase + (size_t)group * decode_group_floats(j.F, T);  // [T][F]: one down item's inputs
  float *red = hs + (size_t)T * j.F;                                 // [warps][T][32]
  wait_plan();
  if (hd->error) return;
  qs.nH = hd->n_hits;
  qs.nM = hd->n_stage0_miss;
  const uint32_t ep = hd->epoch;
  int32_t *const abort_word = j.sync + 2;

  int c = group;
  for (;; c += GROUPS) {
    const int s = c % NB;
    const uint32_t parity = (uint32_t)(c / NB) & 1u;
    // one thread waits (bounded) and shares the decision, so that every
    // compute thread leaves the loop together
    if (gtid == 0) s_ok[group] = ring_wait(&full[s], parity, j.wait_ns) ? 1 : 0;
    group_sync(group);
    if (!s_ok[group]) {
      flag_error(j.err, 3);
      break;
    }
    (void)mbar_try_wait(&full[s], parity);  // completed phase: each thread's acquire of the tiles
    const int code = s_item[s];
    if (code < 0) break;
    const Work wk = decode_claim(code, qs);
    const int it_slot = s_work[s].slot, n = s_work[s].pair_count;
    // the pairs' rows outlive the ring slot: kept for the group (read after its
    // next barrier, rewritten only after the loop-top barrier of its next item)
    if (gtid == 0)
#pragma unroll
      for (int q = 0; q < TMAX; ++q) s_grow[group][q] = s_prow[s][q];
    const MatLayout &L = mat_of(wk.mat);
    const bool is_down = wk.mat == 2;
    const int nb = L.nb, K = 32 * nb;
    const unsigned char *buf = ring + (size_t)s * slot_bytes;
    uint8_t *slot = it_slot >= 0 ? j.slots + (uint64_t)it_slot * j.slot_stride : nullptr;

    if (!is_down) {
      // ---- one 32-row tile of gate or up: inputs are the call's staged rows
      int qrow[TMAX];
#pragma unroll
      for (int q = 0; q < TMAX; ++q) qrow[q] = q < n ? s_prow[s][q] / j.k : 0;
      const int row = lane;
      // blocks warp, warp + 8, ... in ascending order, two at a time; each is
      // added exactly as block_term adds it
      float acc[TMAX];
#pragma unroll
      for (int q = 0; q < TMAX; ++q) acc[q] = 0.f;
#pragma unroll 1
      for (int b = gwarp; b < nb; b += 2 * kWarps) {
        const int b2 = b + kWarps;
        const bool two = b2 < nb;
        uint4 q0, q1 = make_uint4(0, 0, 0, 0);
        unsigned short d0b, d1b = 0;
        load_block(buf, wk.miss, 1, row, b, nb, slot, L, wk.tile, q0, d0b);
        if (two) load_block(buf, wk.miss, 1, row, b2, nb, slot, L, wk.tile, q1, d1b);
        float f0[32], f1[32];
        decode_block(q0, f0);
        decode_block(q1, f1);
        const float d0 = half_bits(d0b), d1 = half_bits(d1b);
#pragma unroll
        for (int q = 0; q < TMAX; ++q) {
          if (q < n) {
            const float *xr = xs + (size_t)qrow[q] * K;
            const float t0 = dot32_ilv(f0, xr + 32 * b);
            const float t1 = two ? dot32_ilv(f1, xr + 32 * b2) : 0.f;
            acc[q] = fmaf(d0, fmaf(256.f, t0, -136.f * xsum[qrow[q] * nb + b]), acc[q]);
            if (two) acc[q] = fmaf(d1, fmaf(256.f, t1, -136.f * xsum[qrow[q] * nb + b2]), acc[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < TMAX; ++q)
        if (q < n) red[(gwarp * T + q) * 32 + lane] = acc[q];
      group_sync(group);
      if (gtid == 0) mbar_arrive(&empty[s]);  // the tile is no longer read
      uint64_t *dst = wk.mat == 0 ? j.g : j.u;
      for (int q = gwarp; q < n; q += kWarps) {
        float v = 0.f;
        for (int w2 = 0; w2 < kWarps; ++w2) v += red[(w2 * T + q) * 32 + lane];
        st_tagged(dst + (size_t)s_grow[group][q] * j.F + wk.tile * 32 + lane, v, ep);
      }
    } else {
      // ---- up to kMaxDG 32-row tiles of down.  Each warp takes its blocks b
      // (warp, warp + 8, ... ascending) one at a time: it forms block b of h
      // for every pair from the tagged gate and up values (waiting for them
      // where needed), then adds that block's term to each row of each tile.
      float acc[kMaxDG][TMAX];
#pragma unroll
      for (int tt = 0; tt < kMaxDG; ++tt)
#pragma unroll
        for (int q = 0; q < TMAX; ++q) acc[tt][q] = 0.f;
      bool ok = true;
      // the pairs' rows, and the tagged gate/up words of the warp's next block:
      // loaded one block ahead, so that they are in flight while the current
      // block is computed (a word whose store has not landed yet is polled)
      int prow[TMAX];
      uint64_t gw[TMAX], uw[TMAX];
#pragma unroll
      for (int q = 0; q < TMAX; ++q) prow[q] = q < n ? s_prow[s][q] : 0;
      auto fetch = [&](int b) {
#pragma unroll
        for (int q = 0; q < TMAX; ++q)
          if (q < n) {
            const size_t e = (size_t)prow[q] * j.F + 32 * b + lane;
            gw[q] = ld_tagged(j.g + e);
            uw[q] = ld_tagged(j.u + e);
          }
      };
      if (gwarp < nb) fetch(gwarp);
#pragma unroll 1
      for (int b = gwarp; b < nb; b += kWarps) {
        float hq[TMAX];
#pragma unroll
        for (int q = 0; q < TMAX; ++q) {
          hq[q] = 0.f;
          if (q < n) {
            const size_t e = (size_t)prow[q] * j.F + 32 * b + lane;
            float gv = __uint_as_float((uint32_t)gw[q]), uv = __uint_as_float((uint32_t)uw[q]);
            // injected fault: this call's number + 1 is never written
            const uint32_t ep_g = (j.inject && gwarp == 0 && b == 0 && q == 0) ? ep + 1u : ep;
            if ((uint32_t)(gw[q] >> 32) != ep_g) ok = wait_tagged(j.g + e, ep_g, abort_word, gv, j.wait_ns) && ok;
            if ((uint32_t)(uw[q] >> 32) != ep) ok = wait_tagged(j.u + e, ep, abort_word, uv, j.wait_ns) && ok;
            const float h = gv / (1.f + expf(-gv)) * uv;
            hs[q * K + 32 * b + ilv(lane)] = h;
            // block sum X_b: lane j holds value j, fixed xor tree
            float v = h;
#pragma unroll
            for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
            hq[q] = v;
          }
        }
        if (b + kWarps < nb) fetch(b + kWarps);
        __syncwarp();
        // the item's tiles two at a time for one token (two independent
        // decode/dot chains), one at a time for several (one chain per token)
        constexpr int kStep = TMAX == 1 ? 2 : 1;
#pragma unroll
        for (int tt = 0; tt < kMaxDG; tt += kStep) {
          if (tt < wk.nt) {
            const bool two = kStep == 2 && tt + 1 < wk.nt;
            uint4 q0, q1 = make_uint4(0, 0, 0, 0);
            unsigned short d0b, d1b = 0;
            load_block(buf, wk.miss, wk.nt, tt * 32 + lane, b, nb, slot, L, wk.tile, q0, d0b);
            if (two) load_block(buf, wk.miss, wk.nt, (tt + 1) * 32 + lane, b, nb, slot, L, wk.tile, q1, d1b);
            float f0[32], f1[32];
            decode_block(q0, f0);
            decode_block(q1, f1);
            const float d0 = half_bits(d0b), d1 = half_bits(d1b);
#pragma unroll
            for (int q = 0; q < TMAX; ++q)
              if (q < n) {
                const float *hb = hs + (size_t)q * K + 32 * b;
                const float t0 = dot32_ilv(f0, hb);
                const float t1 = two ? dot32_ilv(f1, hb) : 0.f;
                acc[tt][q] = fmaf(d0, fmaf(256.f, t0, -136.f * hq[q]), acc[tt][q]);
                if (two) acc[tt + 1][q] = fmaf(d1, fmaf(256.f, t1, -136.f * hq[q]), acc[tt + 1][q]);
              }
          }
        }
      }
      if (!ok) flag_error(j.err, 3);
#pragma unroll
      for (int tt = 0; tt < kMaxDG; ++tt) {
        if (tt < wk.nt) {
          if (tt > 0) group_sync(group);  // the previous tile's sums have been read
#pragma unroll
          for (int q = 0; q < TMAX; ++q)
            if (q < n) red[(gwarp * T + q) * 32 + lane] = acc[tt][q];
          group_sync(group);
          if (tt == wk.nt - 1 && gtid == 0) mbar_arrive(&empty[s]);  // the tiles are no longer read
          for (int q = gwarp; q < n; q += kWarps) {
            float v = 0.f;
            for (int w2 = 0; w2 < kWarps; ++w2) v += red[(w2 * T + q) * 32 + lane];
            st_tagged(j.y + (size_t)s_grow[group][q] * j.H + (wk.tile + tt) * 32 + lane, v, ep);
          }
        }
      }
    }
    // hand the item to the publisher once every compute thread's stores are issued
    const int p = c % kPubSlots;
    if (gtid == 0) {
      if (c >= kPubSlots && !ring_wait(&pubfree[p], (uint32_t)((c / kPubSlots) - 1) & 1u, j.wait_ns)) flag_error(j.err, 3);
      s_pub[p] = code;
      s_pub_n[p] = n;
#pragma unroll
      for (int q = 0; q < TMAX; ++q) s_pub_prow[p][q] = s_grow[group][q];
    }
    mbar_arrive(&pub[p]);
  }
  // end of the publisher's list
  {
    const int p = c % kPubSlots;
    if (gtid == 0) {
      if (c >= kPubSlots) (void)ring_wait(&pubfree[p], (uint32_t)((c / kPubSlots) - 1) & 1u, j.wait_ns);
      s_pub[p] = -1;
    }
    mbar_arrive(&pub[p]);
  }
}

}  // namespace

bool decode_layer_supported(int H, int F, int T) {
  if (T < 1 || T > kTokPerUnit || H % 32 || F % 32) return false;
  return decode_smem(H, F, T, 2, 1) <= kDecodeSmemCap;
}

cudaError_t launch_decode_layer(const FfnArgs &a, const uint8_t *host_layer, uint64_t expert_stride,
                                const uint32_t *miss_ready, const float *w, uint64_t *gu, uint64_t *yt, float *out,
                                int32_t *sync, int cbase, int T, int n_sms, uint64_t wait_ns, int inject,
                                cudaStream_t st) {
  if (!decode_layer_supported(a.H, a.F, T)) return cudaErrorInvalidValue;
  DecodeJob j;
  j.host = host_layer;
  j.expert_stride = expert_stride;
  j.miss_ready = miss_ready;
  j.slots = const_cast<uint8_t *>(a.slots);
  j.slot_stride = a.slot_stride;
  j.lay = a.lay;
  j.hdr = a.hdr;
  j.items = a.items;
  j.perm = a.perm;
  j.w = w;
  j.x = a.x;
  j.x_bf16 = a.x_bf16;
  j.T = T;
  j.k = a.k;
  j.H = a.H;
  j.F = a.F;
  j.DG = decode_down_group(a.H, a.F);
  j.g = gu;
  j.u = gu + (size_t)T * a.k * a.F;
  j.y = yt;
  j.out = out;
  j.sync = sync;
  j.cbase = cbase;
  j.wait_ns = wait_ns;
  j.inject = inject;
  j.err = a.err;
  // single-token calls: two compute groups and four items in flight per CTA;
  // two tokens: two groups and three items when they fit (with more tokens the
  // second group's registers spill and it loses); otherwise one group, three
  // items in flight when they fit, else two
  const bool two = T == 1 && decode_smem(a.H, a.F, T, 4, 2) <= kDecodeSmemCap;
  const bool two3 = !two && T == 2 && decode_smem(a.H, a.F, T, 3, 2) <= kDecodeSmemCap;
  const bool nb3 = decode_smem(a.H, a.F, T, 3, 1) <= kDecodeSmemCap;
  const size_t smem = two    ? decode_smem(a.H, a.F, T, 4, 2)
                      : two3 ? decode_smem(a.H, a.F, T, 3, 2)
                             : decode_smem(a.H, a.F, T, nb3 ? 3 : 2, 1);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sms);
  cfg.blockDim = dim3(decode_threads(two || two3 ? 2 : 1));
  cfg.dynamicSmemBytes = smem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  auto go = [&](auto kern, DynSmemLimit &cur) -> cudaError_t {
    const cudaError_t e = ensure_dyn_smem(kern, smem, cur);
    if (e != cudaSuccess) return e;
    return cudaLaunchKernelEx(&cfg, kern, j);
  };
  static DynSmemLimit c412, c322, c311, c211, c341, c381, c281;
  if (two) return go(decode_layer_kernel<4, 1, 2>, c412);
  if (two3) return go(decode_layer_kernel<3, 2, 2>, c322);
  if (T == 1) return nb3 ? go(decode_layer_kernel<3, 1, 1>, c311) : go(decode_layer_kernel<2, 1, 1>, c211);
  if (T <= 4 && nb3) return go(decode_layer_kernel<3, 4, 1>, c341);
  return nb3 ? go(decode_layer_kernel<3, kTokPerUnit, 1>, c381) : go(decode_layer_kernel<2, kTokPerUnit, 1>, c281);
}

}  // namespace moe
