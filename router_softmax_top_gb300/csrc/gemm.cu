// Prefill path: token-sorted grouped GEMM of the expert FFN on the 5th-gen
// tensor cores (tcgen05.mma, kind::f16, bf16 operands, fp32 accumulators in
// TMEM), where one call routes many tokens to each expert and the FFN is a
// dense contraction (2 * 3 * H * F flops per routed pair, "Multi-GPU LLM
// Calculator: VRAM Split and RAM Offload", "Decode and prefill").
//
// Persistent kernel: one CTA per SM walks the call's output tiles, each
// 128 output features (rows of W) x up to kGemmN routed pairs of one expert,
// looping over the input dimension in chunks of 64; one pipeline runs on
// across the CTA's tiles, so a tile's loads start while the previous tile is
// still being multiplied and no tile pays for set-up.  The pairs' activations
// were copied beforehand into pair-sorted order, so a tile's B operand is a
// contiguous row range that a TMA tensor copy lands directly in the
// 128-byte-swizzled K-major layout.  Roles:
//   raw loader  brings each chunk's Q4_0 weights into a raw ring (10 deep for
//               gate/up, 8 for down) with two TMA tensor copies (nibbles,
//               scales) over the slot planes viewed as
//               [slot][matrix][tile][block][words] (one instruction per plane:
//               issuing one bulk copy per 1 KB run took as long as a whole
//               chunk's dequantisation and MMAs);
//   B loader    brings each chunk's activation rows into shared memory with a
//               TMA tensor copy that completes on the stage's barrier;
//   dequant     two groups of 8 warps take the chunks in turn and dequantise
//               them to bf16, w = (q - 8) * bf16(d) rounded to bf16, built with
//               bf16x2 operations from the nibble bits, straight into the
//               stage's columns of tensor memory (tcgen05.st), so the weight
//               operand never passes through shared memory;
//   MMA         one thread waits for one barrier per chunk (the dequantised
//               weights and the activations) and issues the MMAs -- A from
//               tensor memory, B from shared memory; gate and up share the
//               activations and accumulate into two TMEM regions -- then
//               commits the stage back to both producers;
//   epilogue    4 warps read the accumulators from TMEM: gate/up -> h =
//               silu(g) * u rounded to bf16 (pair-sorted rows); down -> y in
//               fp32 (rows by pair), while the next tile's chunks already load
//               and dequantise (down: while the next tile accumulates into the
//               second accumulator buffer).
// Stages are guarded by mbarriers; every wait is bounded and gives up early
// once another role has failed; on failure the CTA waits for its copies and
// MMAs in flight, sets the handle's error word, frees TMEM and returns.
#include <algorithm>

#include "common.cuh"

namespace moe {
namespace {

constexpr int kGemmM = 128;    // output features per tile
constexpr int kGemmK = 64;     // input features per pipeline stage (128 bytes of bf16)
constexpr int kDqThreads = 256;  // one group of dequantising warps
constexpr int kGemmDqg = 2;      // groups of dequantising warps
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
__device__ __forceinline__ bool g_mbar_done(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(gsa(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Bounded wait for the phase of `bar` with the given parity: gives up (false)
// after kGemmWaitNs of wall time or kGemmSpin polls, or as soon as another role
// of the CTA has failed (fail != nullptr).  A phase that has completed already
// is seen by a non-blocking test first (a potentially suspending try_wait costs
// a few hundred cycles even then, which the MMA issuer cannot afford per chunk).
__device__ __forceinline__ bool g_mbar_wait(uint64_t *bar, uint32_t parity, const int *fail) {
  if (g_mbar_done(bar, parity)) return true;
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

// The same wait by every lane of a warp, agreed by a vote: the lanes leave
// their polling loops at different polls, and the warp-collective tcgen05
// instructions that follow (.sync.aligned: ld, st, wait) need the warp
// converged.  true only if every lane saw the phase complete.
__device__ __forceinline__ bool g_mbar_wait_warp(uint64_t *bar, uint32_t parity, const int *fail) {
  const bool ok = g_mbar_wait(bar, parity, fail);
  return __all_sync(0xffffffffu, ok);
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

// One MMA: D (tensor memory) += A x B, A in tensor memory (rows in lanes, K
// along the columns, two bf16 per 32-bit column), B in shared memory.
__device__ __forceinline__ void umma_ts(uint32_t tmem_d, uint32_t tmem_a, uint64_t db, uint32_t idesc,
                                        uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n" ::"r"(
          tmem_d),
      "r"(tmem_a), "l"(db), "r"(idesc), "r"(accumulate));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(gsa(bar))
               : "memory");
}
// The warp's 32 lanes x 16 consecutive 32-bit columns of tensor memory into
// registers; the values may be used only after tmem_ld_wait().
__device__ __forceinline__ void tmem_ld16_issue(uint32_t addr, uint32_t r[16]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(addr));
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_ld16(uint32_t addr, float v[16]) {
  uint32_t r[16];
  tmem_ld16_issue(addr, r);
  tmem_ld_wait();
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// The warp's 32 lanes x 16 consecutive 32-bit columns of tensor memory from
// registers (each thread its lane).
__device__ __forceinline__ void tmem_st16(uint32_t addr, const uint32_t v[16]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};" ::"r"(
          addr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]), "r"(v[9]),
      "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15])
      : "memory");
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
// Q4_0 of one chunk (4 row tiles x 2 blocks per matrix), as the TMA boxes land:
// nibbles [matrix][tile][block][512 B], then scales [matrix][tile][block][64 B]
template <int NMAT>
constexpr size_t raw_stage_bytes() { return (size_t)NMAT * (4 * 1024 + 4 * 128); }

// Dequantise block bi (32 inputs) of row r of one matrix from the raw chunk
// (nib: the matrix's nibbles [tile][block][32 rows][16 B], sc: its scales
// [tile][block][32 rows]) into 16 bf16 pairs in input order: out[0..7] hold
// values (0,1) .. (14,15) (low nibbles), out[8..15] values (16,17) .. (30,31).
__device__ __forceinline__ void dequant_block(const unsigned char *nib, const unsigned char *sc, int r, int bi,
                                              bool valid, uint32_t out[16]) {
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
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t p01 = __byte_perm(w[i], 0u, 0x4140u);  // bytes 4i, 4i+1 in the two halves
    const uint32_t p23 = __byte_perm(w[i], 0u, 0x4342u);  // bytes 4i+2, 4i+3
    const uint32_t v[4] = {(p01 & 0x000F000Fu) | 0x43004300u, (p23 & 0x000F000Fu) | 0x43004300u,
                           ((p01 >> 4) & 0x000F000Fu) | 0x43004300u, ((p23 >> 4) & 0x000F000Fu) | 0x43004300u};
    __nv_bfloat162 o[4];
#pragma unroll
    for (int z = 0; z < 4; ++z) o[z] = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&v[z]), k136), d2);
    out[2 * i + 0] = *reinterpret_cast<const uint32_t *>(&o[0]);
    out[2 * i + 1] = *reinterpret_cast<const uint32_t *>(&o[1]);
    out[8 + 2 * i + 0] = *reinterpret_cast<const uint32_t *>(&o[2]);
    out[8 + 2 * i + 1] = *reinterpret_cast<const uint32_t *>(&o[3]);
  }
}

// Waits (bounded) until the last min(issued, stages) copies a loader issued
// into a ring of `stages` barriers have landed, so no copy is in flight when
// the CTA leaves; a no-op once all of them were consumed.
__device__ __forceinline__ void drain_ring(uint64_t *full, int stages, int issued) {
  for (int c = issued - stages < 0 ? 0 : issued - stages; c < issued; ++c)
    (void)g_mbar_wait(&full[c % stages], (uint32_t)(c / stages) & 1u, nullptr);
}

// Pipeline depths, tensor-memory layout and warp roles of the persistent
// kernel.  Tensor memory (512 columns x 128 lanes of 32 bits): accumulators in
// columns [0, 256) -- gate/up: one buffer, gate [0, 128) and up [128, 256);
// down: two buffers of 128 -- and the dequantised weight stages in [256, 512),
// each 64 inputs x 128 rows per matrix = 32 columns (two bf16 per column).
// Keeping A in tensor memory takes its writes and the MMAs' reads of it off
// shared memory, whose bandwidth otherwise bounds the chunk rate.
template <int NMAT, int DQG>
struct GemmCfg {
  static constexpr int kAccBufs = NMAT == 2 ? 1 : 2;
  static constexpr uint32_t kAccCols = NMAT == 2 ? 256 : 128;
  static constexpr uint32_t kAStageCols = NMAT * 32;
  // MMA stages: a dequantised weight stage in tensor memory and an activation
  // stage in shared memory, completed together on one barrier (one wait per
  // chunk for the MMA issuer)
  static constexpr int kA = (int)(256 / kAStageCols);  // 4 (gate/up) or 8 (down)
  static constexpr int kB = kA;
  static constexpr int kRaw = NMAT == 2 ? 10 : 8;      // raw Q4_0 stages (bytes in flight from HBM)
  static constexpr int kDqWarps = 8 * DQG;
  static constexpr int kEpiWarp0 = kDqWarps;           // 4 epilogue warps; warp w reads TMEM lanes 32 (w % 4) ..
  static constexpr int kMmaWarp = kDqWarps + 4, kRawWarp = kDqWarps + 5, kBWarp = kDqWarps + 6;
  // one MMA-issuing thread per matrix: issuing a tcgen05.mma costs its thread
  // ~85 cycles whatever N is, so gate and up are issued from two warps
  static constexpr int kIssuers = NMAT;
  static constexpr int kMmaWarp2 = kDqWarps + 7;       // issues the up matrix (gate/up only)
  static constexpr int kThreads = 32 * (kDqWarps + 7 + (NMAT == 2 ? 1 : 0));
  static constexpr size_t kRawStage = raw_stage_bytes<NMAT>();
  static constexpr size_t kSmem = kB * kBTileBytes + kRaw * kRawStage + 1024;
  static_assert(kEpiWarp0 % 4 == 0, "epilogue warps must start at a multiple of 4");
  static_assert(kSmem <= 227 * 1024, "shared memory");
};
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemA0 = 256;  // first column of the weight stages

// Persistent grouped GEMM: one CTA per SM walks the call's tiles (GEMM unit of
// up to kGemmN pairs of one expert) x (128-row tile of the matrix), tile t =
// blockIdx.x + i * gridDim.x, with one pipeline that runs on across tiles:
// the loaders fetch chunk after chunk of tile after tile, the dequantising
// warps and the MMA warp consume them in the same order, and the MMA warp
// accumulates tile i into its TMEM buffer (i % 2 for down, the one buffer for
// gate/up) once the epilogue warps have drained the tile that used it before.
// Every role walks the same tile list; chunk g (counted over the CTA's tiles)
// uses stage g % depth of each ring.
template <int NMAT, int DQG>
__global__ void __launch_bounds__(GemmCfg<NMAT, DQG>::kThreads, 1)
    umma_gemm_kernel(const __grid_constant__ GemmMaps maps, const __grid_constant__ RawMaps raw_maps,
                     const GemmJob j) {
  using C = GemmCfg<NMAT, DQG>;
  int lo, hi;
  if (!gunit_range(j.hdr, j.gunit_begin, j.range_kind, j.stage, lo, hi)) return;
  const int nM = (j.R + kGemmM - 1) / kGemmM;
  const int nT = (hi - lo) * nM;
  if ((int)blockIdx.x >= nT) return;
  const int n_my = (nT - 1 - (int)blockIdx.x) / (int)gridDim.x + 1;  // tiles of this CTA
  const int n_chunks = j.nb / 2;                                      // 64 inputs = 2 blocks per chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char *sm =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *sb_base = sm;
  unsigned char *raw = sb_base + C::kB * kBTileBytes;
  // full[s]: the dequantising warps' arrivals plus the activation copy's bytes;
  // empty[s]: the MMAs that read stage s have completed
  __shared__ __align__(8) uint64_t full[C::kA], empty[C::kA], rfull[C::kRaw], rempty[C::kRaw],
      accfull[C::kAccBufs], accempty[C::kAccBufs], done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_fail;

  if (tid == 0) {
    for (int s = 0; s < C::kA; ++s) {
      g_mbar_init(&full[s], kDqThreads + 1);
      g_mbar_init(&empty[s], C::kIssuers);
    }
    for (int s = 0; s < C::kRaw; ++s) {
      g_mbar_init(&rfull[s], 1);
      g_mbar_init(&rempty[s], kDqThreads);
    }
    for (int b = 0; b < C::kAccBufs; ++b) {
      g_mbar_init(&accfull[b], C::kIssuers);
      g_mbar_init(&accempty[b], 128);
    }
    g_mbar_init(&done, C::kIssuers);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (warp == C::kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(gsa(&tmem_base)),
                 "r"(kTmemCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  // tile i of this CTA: GEMM unit and 128-row tile
  auto tile_unit = [&](int i, int &mt) -> int {
    const int t = (int)blockIdx.x + i * (int)gridDim.x;
    mt = t % nM;
    return lo + t / nM;
  };

  if (warp == C::kRawWarp) {
    // ---- raw Q4_0 loader: per chunk, blocks 2c, 2c+1 of row tiles 4 mt .. 4 mt + 3
    // of each matrix: one tensor copy of the nibbles, one of the scales (tiles
    // past the matrix land as zeros)
    if (lane == 0) {
      const CUtensorMap *mn = NMAT == 2 ? &raw_maps.gu_nib : &raw_maps.dn_nib;
      const CUtensorMap *ms = NMAT == 2 ? &raw_maps.gu_sc : &raw_maps.dn_sc;
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(mn)) : "memory");
      asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(ms)) : "memory");
      int g = 0;
      bool stop = false;
      for (int i = 0; i < n_my && !stop; ++i) {
        int mt;
        const WorkUnit wu = j.gunits[tile_unit(i, mt)];
        const int slot_ix = j.slot0 + j.items[wu.item].slot, rt0 = 4 * mt;
        for (int c = 0; c < n_chunks; ++c, ++g) {
          const int s = g % C::kRaw;
          if (g >= C::kRaw && !g_mbar_wait(&rempty[s], (uint32_t)((g / C::kRaw) - 1) & 1u, &s_fail)) {
            s_fail = 1;
            stop = true;
            break;
          }
          unsigned char *rs = raw + (size_t)s * C::kRawStage;
          expect_tx(&rfull[s], (uint32_t)C::kRawStage);
          if (NMAT == 2) {
            tma_load_5d(rs, mn, 0, 2 * c, rt0, 0, slot_ix, &rfull[s]);
            tma_load_5d(rs + NMAT * 4096, ms, 0, 2 * c, rt0, 0, slot_ix, &rfull[s]);
          } else {
            tma_load_4d(rs, mn, 0, 2 * c, rt0, slot_ix, &rfull[s]);
            tma_load_4d(rs + NMAT * 4096, ms, 0, 2 * c, rt0, slot_ix, &rfull[s]);
          }
        }
      }
      drain_ring(rfull, C::kRaw, g);
    }
  } else if (warp == C::kBWarp) {
    // ---- activation loader: rows [pair_begin, pair_begin + box) of the sorted
    // buffer, columns [64 c, 64 c + 64), one TMA tensor copy per chunk
    if (lane == 0) {
      for (int b = 0; b < 4; ++b)
        asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(&maps.box[b])) : "memory");
      int g = 0;
      bool stop = false;
      for (int i = 0; i < n_my && !stop; ++i) {
        int mt;
        const WorkUnit wu = j.gunits[tile_unit(i, mt)];
        const int nr = (wu.pair_count + 15) & ~15;
        const int bsel = nr <= 16 ? 0 : nr <= 32 ? 1 : nr <= 64 ? 2 : 3;
        const uint32_t b_bytes = (uint32_t)(16 << bsel) * 128u;
        for (int c = 0; c < n_chunks; ++c, ++g) {
          const int s = g % C::kB;
          if (g >= C::kB && !g_mbar_wait(&empty[s], (uint32_t)((g / C::kB) - 1) & 1u, &s_fail)) {
            s_fail = 1;
            stop = true;
            break;
          }
          expect_tx(&full[s], b_bytes);
          tma_load_2d(sb_base + (size_t)s * kBTileBytes, &maps.box[bsel], c * kGemmK, wu.pair_begin, &full[s]);
        }
      }
      // no copy may still be landing when the CTA leaves: the last stages'
      // barriers complete once their bytes (and dequantised halves) are in
      drain_ring(full, C::kB, g);
    }
  } else if (warp == C::kMmaWarp || (NMAT == 2 && warp == C::kMmaWarp2)) {
    // ---- MMA issuers (gate/up: one per matrix): tile i into accumulator buffer
    // i % kAccBufs, once the epilogue has drained the tile that used it before
    // (i - kAccBufs); every issuer commits each stage and each tile, so the
    // barriers complete once both matrices' MMAs have
    if (lane == 0) {
      const int m = (NMAT == 2 && warp == C::kMmaWarp2) ? 1 : 0;
      int g = 0;
      bool stop = false;
      for (int i = 0; i < n_my && !stop; ++i) {
        int mt;
        const WorkUnit wu = j.gunits[tile_unit(i, mt)];
        const int nr = (wu.pair_count + 15) & ~15;
        const uint32_t idesc = idesc_bf16(kGemmM, nr);
        const int buf = i % C::kAccBufs, use = i / C::kAccBufs;
        if (use >= 1 && !g_mbar_wait(&accempty[buf], (uint32_t)(use - 1) & 1u, &s_fail)) {
          s_fail = 1;
          break;
        }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t dcol = tmem + (uint32_t)buf * C::kAccCols + (uint32_t)(m * kGemmN);
        for (int c = 0; c < n_chunks; ++c, ++g) {
          const int sa = g % C::kA;
          if (!g_mbar_wait(&full[sa], (uint32_t)(g / C::kA) & 1u, &s_fail)) {
            s_fail = 1;
            stop = true;
            break;
          }
          asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
          const uint64_t bd = sw128_desc(gsa(sb_base + (size_t)sa * kBTileBytes));
          const uint32_t a_col = tmem + kTmemA0 + (uint32_t)sa * C::kAStageCols + (uint32_t)(m * 32);
#pragma unroll
          for (int ks = 0; ks < kGemmK / 16; ++ks)
            umma_ts(dcol, a_col + (uint32_t)(ks * 8), bd + (uint64_t)(ks * 2), idesc, (c > 0 || ks > 0) ? 1u : 0u);
          umma_commit(&empty[sa]);
        }
        if (!stop) umma_commit(&accfull[buf]);
      }
      umma_commit(&done);  // also on failure: `done` then tracks the MMAs in flight
    }
  } else if (warp >= C::kEpiWarp0) {
    // ---- epilogue (4 warps): warp w reads TMEM lanes 32 (w % 4) .. + 31 (rows of
    // the tile): gate/up -> h = silu(g) * u rounded to bf16 (pair-sorted rows);
    // down -> y in fp32 (rows by pair).  The buffer is released once read.
    const int q = warp & 3;
    for (int i = 0; i < n_my; ++i) {
      int mt;
      const WorkUnit wu = j.gunits[tile_unit(i, mt)];
      const int n = wu.pair_count, nr = (n + 15) & ~15, buf = i % C::kAccBufs;
      if (!g_mbar_wait_warp(&accfull[buf], (uint32_t)(i / C::kAccBufs) & 1u, &s_fail)) {
        s_fail = 1;
        break;
      }
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int row = mt * kGemmM + q * 32 + lane;
      const uint32_t lane_addr = tmem + (uint32_t)buf * C::kAccCols + ((uint32_t)(q * 32) << 16);
      // down: the tile's pairs (rows of y), lane l holding pairs l, l + 32, l + 64, l + 96
      static_assert(kGemmN == 128, "four pair registers per lane");
      int p0 = 0, p1 = 0, p2 = 0, p3 = 0;
      if (NMAT == 1) {
        const int32_t *pp = j.perm + wu.pair_begin;
        p0 = lane < n ? pp[lane] : 0;
        p1 = 32 + lane < n ? pp[32 + lane] : 0;
        p2 = 64 + lane < n ? pp[64 + lane] : 0;
        p3 = 96 + lane < n ? pp[96 + lane] : 0;
      }
      for (int c0 = 0; c0 < nr; c0 += 16) {
        __syncwarp();
        if (NMAT == 2) {
          // gate and up columns loaded together; h = silu(g) * u for all 16, then
          // the stores.  __expf and __fdividef err by a few fp32 ulps, far below
          // the rounding of h to bf16 (an exponential that overflows gives h = 0,
          // the value's limit)
          uint32_t gr[16], ur[16];
          tmem_ld16_issue(lane_addr + c0, gr);
          tmem_ld16_issue(lane_addr + kGemmN + c0, ur);
          tmem_ld_wait();
          __nv_bfloat16 hb[16];
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const float gv = __uint_as_float(gr[i2]), uv = __uint_as_float(ur[i2]);
            hb[i2] = __float2bfloat16_rn(__fdividef(gv, 1.f + __expf(-gv)) * uv);
          }
          if (row < j.R) {
            __nv_bfloat16 *dst = j.h16s + (size_t)(wu.pair_begin + c0) * j.R + row;
#pragma unroll
            for (int i2 = 0; i2 < 16; ++i2)
              if (c0 + i2 < n) dst[(size_t)i2 * j.R] = hb[i2];
          }
        } else {
          float g[16];
          tmem_ld16(lane_addr + c0, g);
          const int pr = c0 < 32 ? p0 : c0 < 64 ? p1 : c0 < 96 ? p2 : p3;
#pragma unroll
          for (int i2 = 0; i2 < 16; ++i2) {
            const int col = c0 + i2;
            const int p = __shfl_sync(0xffffffffu, pr, (c0 & 31) + i2);
            if (col < n && row < j.R) j.y[(size_t)p * j.R + row] = g[i2];
          }
        }
      }
      asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
      g_mbar_arrive(&accempty[buf]);
    }
  } else {
    // ---- dequant (DQG groups of 8 warps, chunks in turn) into the tensor-memory
    // weight stage: gate/up: thread = (matrix, row), both blocks (32 columns);
    // down: thread = (block, row) (16 columns).  Warp w writes TMEM lanes
    // 32 (w % 4) .. + 31, the rows its threads dequantise.
    const int grp = warp / 8, lt = tid & (kDqThreads - 1);
    const int r = lt & 127, hi_half = lt >> 7;
    const uint32_t lane_base = (uint32_t)((r & ~31) << 16);
    int g = 0;
    bool stop = false;
    for (int i = 0; i < n_my && !stop; ++i) {
      int mt;
      (void)tile_unit(i, mt);
      const int n_rt = min(4, (j.R >> 5) - 4 * mt);  // valid 32-row tiles
      const bool valid = (r >> 5) < n_rt;
      for (int c = 0; c < n_chunks; ++c, ++g) {
        if (DQG > 1 && g % DQG != grp) continue;
        const int sa = g % C::kA, rsi = g % C::kRaw;
        if (!g_mbar_wait_warp(&rfull[rsi], (uint32_t)(g / C::kRaw) & 1u, &s_fail)) {
          s_fail = 1;
          stop = true;
          break;
        }
        const unsigned char *rs = raw + (size_t)rsi * C::kRawStage;
        uint32_t v0[16], v1[16];
        if (NMAT == 2) {
          const unsigned char *nib = rs + hi_half * 4096, *sc = rs + NMAT * 4096 + hi_half * 512;
          dequant_block(nib, sc, r, 0, valid, v0);
          dequant_block(nib, sc, r, 1, valid, v1);
        } else {
          dequant_block(rs, rs + NMAT * 4096, r, hi_half, valid, v0);
        }
        g_mbar_arrive(&rempty[rsi]);
        // the stage's previous MMAs (chunk g - kA) must have read it
        if (g >= C::kA && !g_mbar_wait_warp(&empty[sa], (uint32_t)((g / C::kA) - 1) & 1u, &s_fail)) {
          s_fail = 1;
          stop = true;
          break;
        }
        __syncwarp();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        const uint32_t a_col = tmem + lane_base + kTmemA0 + (uint32_t)sa * C::kAStageCols;
        if (NMAT == 2) {
          tmem_st16(a_col + (uint32_t)hi_half * 32, v0);
          tmem_st16(a_col + (uint32_t)hi_half * 32 + 16, v1);
        } else {
          tmem_st16(a_col + (uint32_t)hi_half * 16, v0);
        }
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        g_mbar_arrive(&full[sa]);
      }
    }
  }

  // MMAs in flight must finish before TMEM is freed: `done` is committed on
  // every path of the issuer
  if ((warp == C::kMmaWarp || (NMAT == 2 && warp == C::kMmaWarp2)) && lane == 0)
    (void)g_mbar_wait(&done, 0, nullptr);
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (s_fail && tid == 0 && j.err) atomicExch(j.err, 4);
  if (warp == C::kMmaWarp)
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kTmemCols));
}

template <int NMAT, int DQG>
cudaError_t launch_gemm_t(const GemmMaps &maps, const RawMaps &raw, const GemmJob &j, int max_gunits,
                          cudaStream_t st) {
  using C = GemmCfg<NMAT, DQG>;
  if (max_gunits <= 0) return cudaSuccess;
  if (j.nb % 2) return cudaErrorInvalidValue;
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(umma_gemm_kernel<NMAT, DQG>, C::kSmem, cur);
  if (e != cudaSuccess) return e;
  int dev = 0, n_sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&n_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sms <= 0)
    return cudaErrorInvalidValue;
  const long tiles = (long)max_gunits * ((j.R + kGemmM - 1) / kGemmM);
  const int grid = (int)std::min<long>(tiles, n_sms);
  umma_gemm_kernel<NMAT, DQG><<<grid, C::kThreads, C::kSmem, st>>>(maps, raw, j);
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
  return launch_gemm_t<2, kGemmDqg>(xs_maps, raw, j, max_gunits, st);
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
  return launch_gemm_t<1, kGemmDqg>(h16s_maps, raw, j, max_gunits, st);
}

}  // namespace moe
