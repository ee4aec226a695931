// Prefill path: token-sorted grouped GEMM of the expert FFN on the 5th-gen
// tensor cores (tcgen05.mma, kind::f16, bf16 operands, fp32 accumulators in
// TMEM), where one call routes many tokens to each expert and the FFN is a
// dense contraction (2 * 3 * H * F flops per routed pair, "Multi-GPU LLM
// Calculator: VRAM Split and RAM Offload", "Decode and prefill").
//
// One CTA computes one output tile: 128 output features (rows of W) x up to
// kGemmN routed pairs of one expert, looping over the input dimension in
// chunks of 64.  The pairs' activations were copied beforehand into
// pair-sorted order, so the tile's B operand is a contiguous row range that a
// TMA tensor copy lands directly in the 128-byte-swizzled K-major layout.
// Roles (11 warps):
//   warp 9     brings each chunk's Q4_0 weights into a raw ring with two TMA
//              tensor copies (nibbles, scales) over the slot planes viewed as
//              [slot][matrix][tile][block][words] (one instruction per plane
//              instead of one bulk copy per 1 KB run: issuing 16 bulk copies
//              took as long as a whole chunk's dequantisation and MMAs);
//   warp 10    brings each chunk's activation rows into a 6-deep ring with
//              TMA tensor copies;
//   warps 0-7  dequantise the raw chunk to bf16, w = (q - 8) * bf16(d) rounded
//              to bf16, built with bf16x2 operations from the nibble bits, into
//              the swizzled K-major layout the MMA reads;
//   warp 8     one thread issues the MMAs (gate and up share the activations
//              and accumulate into two TMEM regions) and commits each stage
//              back to its producers;
//   warps 0-7  finally read the accumulators from TMEM: gate/up -> h =
//              silu(g) * u rounded to bf16 (pair-sorted rows); down -> y in
//              fp32 (rows by pair).
// Stages are guarded by mbarriers; every wait is bounded and gives up early
// once another role has failed; on failure the CTA waits for its copies and
// MMAs in flight, sets the handle's error word, frees TMEM and returns.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kGemmM = 128;    // output features per tile
constexpr int kGemmK = 64;     // input features per pipeline stage (128 bytes of bf16)
constexpr int kAStages = 2;    // dequantised weight tiles
constexpr int kBStages = 6;    // activation tiles
constexpr int kRawStages = 4;  // raw Q4_0 chunks
constexpr int kDqThreads = 256;
constexpr int kMmaWarp = 8, kRawWarp = 9, kBWarp = 10;
constexpr int kGemmThreads = 352;
constexpr uint32_t kGemmSpin = 1u << 26;
constexpr uint64_t kGemmWaitNs = 2000000000ull;  // 2 s

__device__ __forceinline__ uint32_t gsa(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void g_mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(gsa(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void g_mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gsa(bar)) : "memory");
}
__device__ __forceinline__ uint64_t g_now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ bool g_mbar_test(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(gsa(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `bar` with the given parity: gives up (false)
// after kGemmWaitNs of wall time or kGemmSpin polls, or as soon as another role
// of the CTA has failed (fail != nullptr).
__device__ __forceinline__ bool g_mbar_wait(uint64_t *bar, uint32_t parity, const int *fail) {
  uint64_t t0 = 0;
  for (uint32_t i = 0; i < kGemmSpin; ++i) {
    if (g_mbar_test(bar, parity)) return true;
    if ((i & 255u) == 255u) {
      if (fail && *reinterpret_cast<const volatile int *>(fail)) return false;
      const uint64_t now = g_now_ns();
      if (t0 == 0) t0 = now;
      else if (now - t0 > kGemmWaitNs) return false;
    }
  }
  return false;
}

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 bytes apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFF) >> 4) | (1ull << 16) | (64ull << 32) | (1ull << 46) | (2ull << 61);
}

// Instruction descriptor, kind::f16: fp32 accumulate, bf16 A and B, both
// K-major, N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma(uint32_t tmem_d, uint64_t da, uint64_t db, uint32_t idesc,
                                     uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "l"(da), "l"(db), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(gsa(bar))
               : "memory");
}
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float v[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// Byte offset of 16-byte chunk c (0..7) of row r in a 128-byte-swizzled
// K-major tile (8-row groups of 1024 bytes).
__device__ __forceinline__ uint32_t sw128_off(int r, int c) {
  return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}


// TMA tensor copy of one 2-D box (x = column, y = row) into shared memory,
// completing on `bar` with the box's byte count.
__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int x, int y, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(gsa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x), "r"(y), "r"(gsa(bar))
      : "memory");
}
// TMA tensor copies of one 4-D / 5-D box (coordinates innermost first).
__device__ __forceinline__ void tma_load_4d(void *dst, const CUtensorMap *map, int x0, int x1, int x2, int x3,
                                            uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5}], [%6];" ::"r"(gsa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(gsa(bar))
      : "memory");
}
__device__ __forceinline__ void tma_load_5d(void *dst, const CUtensorMap *map, int x0, int x1, int x2, int x3,
                                            int x4, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.tensor.5d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4, "
      "%5, %6}], [%7];" ::"r"(gsa(dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(x0), "r"(x1), "r"(x2), "r"(x3), "r"(x4), "r"(gsa(bar))
      : "memory");
}
__device__ __forceinline__ void expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(gsa(bar)), "r"(bytes) : "memory");
}

struct GemmJob {
  int slot0;         // index of the layer's (or stage buffer's) slot 0 in the raw maps' slot array
  MatLayout m0, m1;  // gate, up (NMAT 2) or down (NMAT 1)
  int R, nb;         // output rows, input 32-blocks
  const int32_t *perm;
  const WorkItem *items;
  const WorkUnit *gunits;
  const int32_t *gunit_begin;
  const PlanHdr *hdr;
  int range_kind, stage;
  __nv_bfloat16 *h16s;  // gate/up output [sorted pairs, R]
  float *y;             // down output [pairs, R]
  int32_t *err;
};

__device__ __forceinline__ bool gunit_range(const PlanHdr *h, const int32_t *gb, int kind, int stage,
                                            int &lo, int &hi) {
  if (h->error || stage >= h->n_stages) return false;
  if (kind == 0) { lo = 0; hi = h->hit_gunits; }
  else if (kind == 1) { lo = stage == 0 ? h->hit_gunits : gb[stage]; hi = gb[stage + 1]; }
  else { lo = gb[stage]; hi = gb[stage + 1]; }
  return true;
}

constexpr size_t kBTileBytes = (size_t)kGemmN * 128;  // one chunk of up to 128 activation rows
template <int NMAT>
constexpr size_t a_stage_bytes() { return (size_t)NMAT * kGemmM * 128; }
// Q4_0 of one chunk (4 row tiles x 2 blocks per matrix), as the TMA boxes land:
// nibbles [matrix][tile][block][512 B], then scales [matrix][tile][block][64 B]
template <int NMAT>
constexpr size_t raw_stage_bytes() { return (size_t)NMAT * (4 * 1024 + 4 * 128); }
template <int NMAT>
constexpr size_t gemm_smem_bytes() {
  return kAStages * a_stage_bytes<NMAT>() + kBStages * kBTileBytes + kRawStages * raw_stage_bytes<NMAT>() + 1024;
}

// Dequantise block bi (32 inputs) of row r of one matrix from the raw chunk
// (nib: the matrix's nibbles [tile][block][32 rows][16 B], sc: its scales
// [tile][block][32 rows]) into the swizzled bf16 tile `a` (row r, 16-byte
// chunks 4 bi .. 4 bi + 3).
__device__ __forceinline__ void dequant_block(const unsigned char *nib, const unsigned char *sc, unsigned char *a,
                                              int r, int bi, bool valid) {
  uint4 q = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
  float d = 0.f;
  if (valid) {
    q = *reinterpret_cast<const uint4 *>(nib + (r >> 5) * 1024 + bi * 512 + (r & 31) * 16);
    d = __half2float(__ushort_as_half(
        *reinterpret_cast<const unsigned short *>(sc + (r >> 5) * 128 + bi * 64 + (r & 31) * 2)));
  }
  // two nibbles side by side under the bf16 exponent of 128: 0x4300|q is
  // 128 + q exactly; minus 136 gives q - 8 exactly; times d rounds once
  const __nv_bfloat162 d2 = __float2bfloat162_rn(d);
  const __nv_bfloat162 k136 = __float2bfloat162_rn(136.f);
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
  uint32_t lo_pk[8], hi_pk[8];  // values 0..15 (low nibbles), 16..31 (high nibbles)
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p01 = __byte_perm(w[i], 0u, 0x4140u);  // bytes 4i, 4i+1 in the two halves
    const uint32_t p23 = __byte_perm(w[i], 0u, 0x4342u);  // bytes 4i+2, 4i+3
    const uint32_t v[4] = {(p01 & 0x000F000Fu) | 0x43004300u, (p23 & 0x000F000Fu) | 0x43004300u,
                           ((p01 >> 4) & 0x000F000Fu) | 0x43004300u, ((p23 >> 4) & 0x000F000Fu) | 0x43004300u};
    __nv_bfloat162 o[4];
#pragma unroll
    for (int z = 0; z < 4; ++z) o[z] = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&v[z]), k136), d2);
    lo_pk[2 * i + 0] = *reinterpret_cast<const uint32_t *>(&o[0]);
    lo_pk[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&o[1]);
    hi_pk[2 * i + 0] = *reinterpret_cast<const uint32_t *>(&o[2]);
    hi_pk[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&o[3]);
  }
  *reinterpret_cast<uint4 *>(a + sw128_off(r, 4 * bi + 0)) = make_uint4(lo_pk[0], lo_pk[1], lo_pk[2], lo_pk[3]);
  *reinterpret_cast<uint4 *>(a + sw128_off(r, 4 * bi + 1)) = make_uint4(lo_pk[4], lo_pk[5], lo_pk[6], lo_pk[7]);
  *reinterpret_cast<uint4 *>(a + sw128_off(r, 4 * bi + 2)) = make_uint4(hi_pk[0], hi_pk[1], hi_pk[2], hi_pk[3]);
  *reinterpret_cast<uint4 *>(a + sw128_off(r, 4 * bi + 3)) = make_uint4(hi_pk[4], hi_pk[5], hi_pk[6], hi_pk[7]);
}

// Waits (bounded) until the last min(issued, stages) copies a loader issued
// into a ring of `stages` barriers have landed, so no copy is in flight when
// the CTA leaves; a no-op once all of them were consumed.
__device__ __forceinline__ void drain_ring(uint64_t *full, int stages, int issued) {
  for (int c = issued - stages < 0 ? 0 : issued - stages; c < issued; ++c)
    (void)g_mbar_wait(&full[c % stages], (uint32_t)(c / stages) & 1u, nullptr);
}

template <int NMAT>
__global__ void __launch_bounds__(kGemmThreads, 1)
    umma_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ RawMaps raw_maps,
                     const GemmJob j) {
  int lo, hi;
  if (!gunit_range(j.hdr, j.gunit_begin, j.range_kind, j.stage, lo, hi)) return;
  const int gu = lo + (int)blockIdx.y;
  if (gu >= hi) return;
  const WorkUnit wu = j.gunits[gu];
  const WorkItem it = j.items[wu.item];
  const int n = wu.pair_count;                 // 1..kGemmN
  const int nr = (n + 15) & ~15;               // MMA N: pairs rounded up to 16
  const int bsel = nr <= 16 ? 0 : nr <= 32 ? 1 : nr <= 64 ? 2 : 3;
  const uint32_t b_bytes = (uint32_t)(16 << bsel) * 128u;  // activation box of 16 << bsel rows
  const int m0 = blockIdx.x * kGemmM;
  const int rt0 = m0 >> 5, n_rt = min(4, (j.R >> 5) - rt0);  // valid 32-row tiles
  const int nb = j.nb, n_chunks = nb / 2;      // 64 inputs = 2 blocks per chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char *sm =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *sa_base = sm;
  unsigned char *sb_base = sa_base + kAStages * a_stage_bytes<NMAT>();
  unsigned char *raw = sb_base + kBStages * kBTileBytes;
  __shared__ __align__(8) uint64_t afull[kAStages], aempty[kAStages], bfull[kBStages], bempty[kBStages],
      rfull[kRawStages], rempty[kRawStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_rows[kGemmN];
  __shared__ int s_fail;

  constexpr uint32_t kCols = NMAT == 2 ? 2 * kGemmN : kGemmN;  // TMEM columns (power of 2)
  if (tid == 0) {
    for (int s = 0; s < kAStages; ++s) {
      g_mbar_init(&afull[s], kDqThreads);
      g_mbar_init(&aempty[s], 1);
    }
    for (int s = 0; s < kBStages; ++s) {
      g_mbar_init(&bfull[s], 1);
      g_mbar_init(&bempty[s], 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      g_mbar_init(&rfull[s], 1);
      g_mbar_init(&rempty[s], kDqThreads);
    }
    g_mbar_init(&done, 1);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kGemmN) s_rows[tid] = tid < n ? j.perm[wu.pair_begin + tid] : -1;
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(gsa(&tmem_base)),
                 "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  const int slot_ix = j.slot0 + it.slot;

  if (warp == kRawWarp) {
    // ---- raw Q4_0 loader: per chunk, blocks 2c, 2c+1 of row tiles rt0 .. rt0+3
    // of each matrix: one tensor copy of the nibbles, one of the scales (the
    // full boxes land, tiles past the matrix as zeros)
    if (lane == 0) {
      const CUtensorMap *mn = NMAT == 2 ? &raw_maps.gu_nib : &raw_maps.dn_nib;
      const CUtensorMap *ms = NMAT == 2 ? &raw_maps.gu_sc : &raw_maps.dn_sc;
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(mn)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(ms)) : "memory");
      int c = 0;
      for (; c < n_chunks; ++c) {
        const int s = c % kRawStages;
        if (c >= kRawStages && !g_mbar_wait(&rempty[s], (uint32_t)((c / kRawStages) - 1) & 1u, &s_fail)) {
          s_fail = 1;
          break;
        }
        unsigned char *rs = raw + (size_t)s * raw_stage_bytes<NMAT>();
        expect_tx(&rfull[s], (uint32_t)raw_stage_bytes<NMAT>());
        if (NMAT == 2) {
          tma_load_5d(rs, mn, 0, 2 * c, rt0, 0, slot_ix, &rfull[s]);
          tma_load_5d(rs + NMAT * 4096, ms, 0, 2 * c, rt0, 0, slot_ix, &rfull[s]);
        } else {
          tma_load_4d(rs, mn, 0, 2 * c, rt0, slot_ix, &rfull[s]);
          tma_load_4d(rs + NMAT * 4096, ms, 0, 2 * c, rt0, slot_ix, &rfull[s]);
        }
      }
      drain_ring(rfull, kRawStages, c);
    }
  } else if (warp == kBWarp) {
    // ---- activation loader: rows [pair_begin, pair_begin + box) of the sorted
    // buffer, columns [64 c, 64 c + 64), one TMA tensor copy per chunk
    if (lane == 0) {
      const CUtensorMap *map = &maps.box[bsel];
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
      int c = 0;
      for (; c < n_chunks; ++c) {
        const int s = c % kBStages;
        if (c >= kBStages && !g_mbar_wait(&bempty[s], (uint32_t)((c / kBStages) - 1) & 1u, &s_fail)) {
          s_fail = 1;
          break;
        }
        expect_tx(&bfull[s], b_bytes);
        tma_load_2d(sb_base + (size_t)s * kBTileBytes, map, c * kGemmK, wu.pair_begin, &bfull[s]);
      }
      drain_ring(bfull, kBStages, c);
    }
  } else if (warp == kMmaWarp) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kGemmM, nr);
      for (int c = 0; c < n_chunks; ++c) {
        const int sa = c % kAStages, sb = c % kBStages;
        if (!g_mbar_wait(&afull[sa], (uint32_t)(c / kAStages) & 1u, &s_fail) ||
            !g_mbar_wait(&bfull[sb], (uint32_t)(c / kBStages) & 1u, &s_fail)) {
          s_fail = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t b_addr = gsa(sb_base + (size_t)sb * kBTileBytes);
        const uint32_t a_base = gsa(sa_base + (size_t)sa * a_stage_bytes<NMAT>());
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint32_t a_addr = a_base + (uint32_t)(m * kGemmM * 128);
#pragma unroll
          for (int ks = 0; ks < kGemmK / 16; ++ks)
            umma(tmem + (uint32_t)(m * kGemmN), sw128_desc(a_addr + ks * 32), sw128_desc(b_addr + ks * 32), idesc,
                 (c > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&aempty[sa]);
        umma_commit(&bempty[sb]);
      }
      umma_commit(&done);  // also on failure: `done` then tracks the MMAs in flight
    }
  } else {
    // ---- dequant (warps 0-7): gate/up: thread = (matrix, row), both blocks;
    // down: thread = (block, row)
    const int r = tid & 127, hi_half = tid >> 7;
    const bool valid = (r >> 5) < n_rt;
    for (int c = 0; c < n_chunks; ++c) {
      const int sa = c % kAStages, rsi = c % kRawStages;
      if (c >= kAStages && !g_mbar_wait(&aempty[sa], (uint32_t)((c / kAStages) - 1) & 1u, &s_fail)) {
        s_fail = 1;
        break;
      }
      if (!g_mbar_wait(&rfull[rsi], (uint32_t)(c / kRawStages) & 1u, &s_fail)) {
        s_fail = 1;
        break;
      }
      const unsigned char *rs = raw + (size_t)rsi * raw_stage_bytes<NMAT>();
      unsigned char *st = sa_base + (size_t)sa * a_stage_bytes<NMAT>();
      if (NMAT == 2) {
        const unsigned char *nib = rs + hi_half * 4096, *sc = rs + NMAT * 4096 + hi_half * 512;
        unsigned char *a = st + (size_t)hi_half * kGemmM * 128;
        dequant_block(nib, sc, a, r, 0, valid);
        dequant_block(nib, sc, a, r, 1, valid);
      } else {
        dequant_block(rs, rs + NMAT * 4096, st, r, hi_half, valid);
      }
      g_mbar_arrive(&rempty[rsi]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      g_mbar_arrive(&afull[sa]);
    }
  }

  // ---- epilogue (warps 0-7): warp w reads TMEM lanes 32 (w % 4) .. + 31 (the
  // tile's rows) and the 16-column groups of parity w / 4
  const bool ok = warp < 8 && g_mbar_wait(&done, 0, &s_fail) && !s_fail;
  if (warp < 8 && ok) {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const int q = warp & 3, half = warp >> 2;
    const int row = m0 + q * 32 + lane;
    const uint32_t lane_addr = tmem + ((uint32_t)(q * 32) << 16);
    for (int c0 = half * 16; c0 < nr; c0 += 32) {
      float g[16], u[16];
      tmem_ld16(lane_addr + c0, g);
      if (NMAT == 2) tmem_ld16(lane_addr + kGemmN + c0, u);
      if (row < j.R) {
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int col = c0 + i;
          if (col < n) {
            if (NMAT == 2)
              j.h16s[(size_t)(wu.pair_begin + col) * j.R + row] = __float2bfloat16_rn(g[i] / (1.f + expf(-g[i])) * u[i]);
            else
              j.y[(size_t)s_rows[col] * j.R + row] = g[i];
          }
        }
      }
    }
  } else if (warp < 8 && !ok) {
    s_fail = 1;
  }
  // MMAs in flight must finish before TMEM is freed: `done` is committed on
  // every path of the issuer
  if (s_fail && warp == 0) (void)g_mbar_wait(&done, 0, nullptr);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (s_fail && tid == 0 && j.err) atomicExch(j.err, 4);
  if (warp == kMmaWarp) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
}

template <int NMAT>
cudaError_t launch_gemm_t(const GemmMaps &maps, const RawMaps &raw, const GemmJob &j, int max_gunits,
                          cudaStream_t st) {
  if (max_gunits <= 0) return cudaSuccess;
  if (j.nb % 2) return cudaErrorInvalidValue;
  const size_t smem = gemm_smem_bytes<NMAT>();
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(umma_gemm_kernel<NMAT>, smem, cur);
  if (e != cudaSuccess) return e;
  dim3 grid((j.R + kGemmM - 1) / kGemmM, max_gunits);
  umma_gemm_kernel<NMAT><<<grid, kGemmThreads, smem, st>>>(maps, raw, j);
  return cudaGetLastError();
}

// xs[pos] = x[perm[pos] / k], 16 bytes per thread
__global__ void gather_sorted_kernel(const uint4 *__restrict__ x, const int32_t *__restrict__ perm, int P, int k,
                                     int H8, uint4 *__restrict__ xs) {
  const int total = P * H8;
  for (int i = blockIdx.x * blockDim.x + threadIdx.x; i < total; i += gridDim.x * blockDim.x) {
    const int pos = i / H8, c = i - pos * H8;
    xs[i] = x[(size_t)(perm[pos] / k) * H8 + c];
  }
}

GemmJob base_job(const FfnArgs &a, int slot0, const WorkUnit *gunits, const int32_t *gunit_begin, int range_kind,
                 int stage) {
  GemmJob j;
  j.slot0 = slot0;
  j.perm = a.perm;
  j.items = a.items;
  j.gunits = gunits;
  j.gunit_begin = gunit_begin;
  j.hdr = a.hdr;
  j.range_kind = range_kind;
  j.stage = stage;
  j.h16s = nullptr;
  j.y = nullptr;
  j.err = a.err;
  return j;
}

}  // namespace

namespace {
using EncodeFn = CUresult (*)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                              const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                              CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
// cuTensorMapEncodeTiled from the driver (the runtime links no driver library)
EncodeFn tensor_map_encoder() {
  static EncodeFn encode = nullptr;
  if (!encode) {
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    const cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e == cudaSuccess && q == cudaDriverEntryPointSuccess && fn) encode = reinterpret_cast<EncodeFn>(fn);
  }
  return encode;
}
}  // namespace

cudaError_t make_gemm_maps(const __nv_bfloat16 *base, int K, int rows, GemmMaps *out) {
  const EncodeFn encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  if ((reinterpret_cast<uintptr_t>(base) & 15u) || K % kGemmK || rows <= 0) return cudaErrorInvalidValue;
  const cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)rows};
  const cuuint64_t strides[1] = {(cuuint64_t)K * sizeof(__nv_bfloat16)};
  const cuuint32_t elem[2] = {1, 1};
  for (int i = 0; i < 4; ++i) {
    const cuuint32_t box[2] = {(cuuint32_t)kGemmK, (cuuint32_t)(16 << i)};
    const CUresult r = encode(&out->box[i], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<__nv_bfloat16 *>(base), dims,
                              strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                              CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  }
  return cudaSuccess;
}

cudaError_t make_raw_maps(const uint8_t *base, int n_slots, uint64_t slot_stride, const SlotLayout &lay,
                          RawMaps *out) {
  const EncodeFn encode = tensor_map_encoder();
  if (!encode) return cudaErrorNotSupported;
  if (!base || n_slots <= 0 || (reinterpret_cast<uintptr_t>(base) & 15u) || (slot_stride & 15u))
    return cudaErrorInvalidValue;
  // planes of one matrix: nibbles [tiles][nb][32][16 B] = 128 words per (tile, block),
  // scales [tiles][nb][32] fp16 = 16 words; gate and up are mat_stride apart
  const uint64_t mat_stride = lay.up.nib_off - lay.gate.nib_off;
  if (lay.up.sc_off - lay.gate.sc_off != mat_stride || (mat_stride & 15u)) return cudaErrorInvalidValue;
  const cuuint32_t elem[5] = {1, 1, 1, 1, 1};
  auto enc = [&](CUtensorMap *m, uint64_t off, int rank, const cuuint64_t *dims, const cuuint64_t *strides,
                 const cuuint32_t *box) -> bool {
    if (off & 15u) return false;
    return encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, (cuuint32_t)rank, const_cast<uint8_t *>(base) + off, dims,
                  strides, box, elem, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
  };
  const int gnb = lay.gate.nb, gt = lay.gate.rows / 32, dnb = lay.down.nb, dt = lay.down.rows / 32;
  bool ok = true;
  {
    const cuuint64_t dims[5] = {128, (cuuint64_t)gnb, (cuuint64_t)gt, 2, (cuuint64_t)n_slots};
    const cuuint64_t strides[4] = {512, (cuuint64_t)gnb * 512, mat_stride, slot_stride};
    const cuuint32_t box[5] = {128, 2, 4, 2, 1};
    ok = ok && enc(&out->gu_nib, lay.gate.nib_off, 5, dims, strides, box);
  }
  {
    const cuuint64_t dims[5] = {16, (cuuint64_t)gnb, (cuuint64_t)gt, 2, (cuuint64_t)n_slots};
    const cuuint64_t strides[4] = {64, (cuuint64_t)gnb * 64, mat_stride, slot_stride};
    const cuuint32_t box[5] = {16, 2, 4, 2, 1};
    ok = ok && enc(&out->gu_sc, lay.gate.sc_off, 5, dims, strides, box);
  }
  {
    const cuuint64_t dims[4] = {128, (cuuint64_t)dnb, (cuuint64_t)dt, (cuuint64_t)n_slots};
    const cuuint64_t strides[3] = {512, (cuuint64_t)dnb * 512, slot_stride};
    const cuuint32_t box[4] = {128, 2, 4, 1};
    ok = ok && enc(&out->dn_nib, lay.down.nib_off, 4, dims, strides, box);
  }
  {
    const cuuint64_t dims[4] = {16, (cuuint64_t)dnb, (cuuint64_t)dt, (cuuint64_t)n_slots};
    const cuuint64_t strides[3] = {64, (cuuint64_t)dnb * 64, slot_stride};
    const cuuint32_t box[4] = {16, 2, 4, 1};
    ok = ok && enc(&out->dn_sc, lay.down.sc_off, 4, dims, strides, box);
  }
  return ok ? cudaSuccess : cudaErrorInvalidValue;
}

cudaError_t launch_gather_sorted(const __nv_bfloat16 *x, const int32_t *perm, int P, int k, int H,
                                 __nv_bfloat16 *xs, cudaStream_t st) {
  if (P <= 0) return cudaSuccess;
  if (H % 8) return cudaErrorInvalidValue;
  const int H8 = H / 8, total = P * H8;
  const int grid = std::min((total + 255) / 256, 152 * 8);
  gather_sorted_kernel<<<grid, 256, 0, st>>>(reinterpret_cast<const uint4 *>(x), perm, P, k, H8,
                                             reinterpret_cast<uint4 *>(xs));
  return cudaGetLastError();
}

cudaError_t launch_gemm_gateup(const FfnArgs &a, const GemmMaps &xs_maps, const RawMaps &raw, int slot0,
                               const WorkUnit *gunits, const int32_t *gunit_begin, __nv_bfloat16 *h16s,
                               int range_kind, int stage, int max_gunits, cudaStream_t st) {
  GemmJob j = base_job(a, slot0, gunits, gunit_begin, range_kind, stage);
  j.m0 = a.lay.gate;
  j.m1 = a.lay.up;
  j.R = a.F;
  j.nb = a.H / 32;
  j.h16s = h16s;
  return launch_gemm_t<2>(xs_maps, raw, j, max_gunits, st);
}

cudaError_t launch_gemm_down(const FfnArgs &a, const GemmMaps &h16s_maps, const RawMaps &raw, int slot0,
                             const WorkUnit *gunits, const int32_t *gunit_begin, int range_kind, int stage,
                             int max_gunits, cudaStream_t st) {
  GemmJob j = base_job(a, slot0, gunits, gunit_begin, range_kind, stage);
  j.m0 = a.lay.down;
  j.m1 = a.lay.down;
  j.R = a.H;
  j.nb = a.F / 32;
  j.y = a.y;
  return launch_gemm_t<1>(h16s_maps, raw, j, max_gunits, st);
}

}  // namespace moe
