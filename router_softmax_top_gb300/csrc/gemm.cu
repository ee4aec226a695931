// Prefill path: token-sorted grouped GEMM of the expert FFN on the 5th-gen
// tensor cores (tcgen05.mma, kind::f16, bf16 operands, fp32 accumulators in
// TMEM), where one call routes many tokens to each expert and the FFN is a
// dense contraction (2 * 3 * H * F flops per routed pair, "Multi-GPU LLM
// Calculator: VRAM Split and RAM Offload", "Decode and prefill").
//
// One CTA computes one output tile: 128 output features (rows of W) x up to
// kGemmN routed pairs of one expert, looping over the input dimension in
// chunks of 64.  Roles (8 warps):
//   warp 7     brings the chunk's Q4_0 tile into shared memory with bulk
//              copies (4 contiguous runs of nibbles and of scales per matrix);
//   warps 0-3  dequantise it to bf16, w = (q - 8) * bf16(d) rounded to bf16,
//              built with bf16x2 operations from the nibble bits, into shared
//              memory in the 128-byte-swizzled K-major layout the MMA reads;
//   warps 4-5  gather the pairs' input rows (bf16) with cp.async into the same
//              layout;
//   warp 6     one thread issues the MMAs (gate and up share the inputs and
//              accumulate into two TMEM regions) and commits each stage back to
//              the producers;
//   warps 0-3  finally read the accumulators from TMEM: gate/up -> h =
//              silu(g) * u rounded to bf16; down -> y in fp32.
// Stages are guarded by mbarriers; every wait is bounded and, on timeout, sets
// the handle's error word, frees TMEM and returns.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kGemmM = 128;   // output features per tile
constexpr int kGemmK = 64;    // input features per pipeline stage (128 bytes of bf16)
constexpr int kStages = 3;
constexpr int kGemmThreads = 256;
constexpr uint32_t kGemmSpin = 1u << 26;

__device__ __forceinline__ uint32_t gsa(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ void g_mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(gsa(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void g_mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(gsa(bar)) : "memory");
}
__device__ __forceinline__ bool g_mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kGemmSpin; ++i) {
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
        : "=r"(ok)
        : "r"(gsa(bar)), "r"(parity)
        : "memory");
    if (ok) return true;
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

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  const __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<const uint32_t *>(&v);
}

struct GemmJob {
  const uint8_t *slots;
  uint64_t slot_stride;
  MatLayout m0, m1;  // gate, up (NMAT 2) or down (NMAT 1)
  int R, nb;         // output rows, input 32-blocks
  const __nv_bfloat16 *x;  // input rows [*, 32 nb] bf16
  int x_div;               // input row of pair p is p / x_div
  const int32_t *perm;
  const WorkItem *items;
  const WorkUnit *gunits;
  const int32_t *gunit_begin;
  const PlanHdr *hdr;
  int range_kind, stage;
  __nv_bfloat16 *h16;  // gate/up output [pairs, R]
  float *y;            // down output [pairs, R]
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

constexpr int kRawStages = 4;  // raw Q4_0 chunks in flight (bulk copies)

template <int NMAT>
constexpr size_t gemm_stage_bytes() {  // bf16 A (per matrix) + B tiles of one K chunk
  return (size_t)NMAT * kGemmM * 128 + (size_t)kGemmN * 128;
}
template <int NMAT>
constexpr size_t raw_stage_bytes() {   // Q4_0 of one chunk: 4 row tiles x 2 blocks, per matrix
  return (size_t)NMAT * (4 * 1024 + 4 * 128);
}
template <int NMAT>
constexpr size_t gemm_smem_bytes() {
  return kStages * gemm_stage_bytes<NMAT>() + kRawStages * raw_stage_bytes<NMAT>() + 1024;
}

template <int NMAT>
__global__ void __launch_bounds__(kGemmThreads, 1) umma_gemm_kernel(GemmJob j) {
  int lo, hi;
  if (!gunit_range(j.hdr, j.gunit_begin, j.range_kind, j.stage, lo, hi)) return;
  const int gu = lo + (int)blockIdx.y;
  if (gu >= hi) return;
  const WorkUnit wu = j.gunits[gu];
  const WorkItem it = j.items[wu.item];
  const int n = wu.pair_count;                       // 1..kGemmN
  const int nr = (n + 15) & ~15;                     // MMA N: pairs rounded up to 16
  const int m0 = blockIdx.x * kGemmM;
  const int rt0 = m0 >> 5, n_rt = min(4, (j.R >> 5) - rt0);  // valid 32-row tiles
  const int nb = j.nb, n_chunks = nb / 2;            // 64 inputs = 2 blocks per chunk
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  extern __shared__ __align__(1024) unsigned char sm_raw[];
  unsigned char *sm =
      reinterpret_cast<unsigned char *>((reinterpret_cast<uintptr_t>(sm_raw) + 1023) & ~(uintptr_t)1023);
  unsigned char *raw = sm + kStages * gemm_stage_bytes<NMAT>();
  __shared__ __align__(8) uint64_t full[kStages], empty[kStages], rfull[kRawStages], rempty[kRawStages], done;
  __shared__ uint32_t tmem_base;
  __shared__ int s_rows[kGemmN];
  __shared__ int s_fail;

  constexpr uint32_t kCols = NMAT == 2 ? 2 * kGemmN : kGemmN;  // TMEM columns (power of 2)
  constexpr int kProducers = 128 + 64;                       // dequant + gather threads
  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      g_mbar_init(&full[s], kProducers);
      g_mbar_init(&empty[s], 1);
    }
    for (int s = 0; s < kRawStages; ++s) {
      g_mbar_init(&rfull[s], 1);
      g_mbar_init(&rempty[s], 128);
    }
    g_mbar_init(&done, 1);
    s_fail = 0;
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
  }
  if (tid < kGemmN) s_rows[tid] = tid < n ? j.perm[wu.pair_begin + tid] : -1;
  if (warp == 7) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(gsa(&tmem_base)),
                 "r"(kCols));
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
  const uint32_t tmem = tmem_base;
  const uint8_t *slot = j.slots + (uint64_t)it.slot * j.slot_stride;

  if (warp == 7) {
    // ---- raw Q4_0 loader: per chunk and matrix, 4 contiguous 1 KB nibble runs
    // (32 rows x blocks 2c, 2c+1 of one row tile) and 4 runs of 128 B scales
    if (lane == 0) {
      for (int c = 0; c < n_chunks; ++c) {
        const int s = c % kRawStages;
        if (c >= kRawStages && !g_mbar_wait(&rempty[s], (uint32_t)((c / kRawStages) - 1) & 1u)) {
          s_fail = 1;
          break;
        }
        unsigned char *rs = raw + (size_t)s * raw_stage_bytes<NMAT>();
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(gsa(&rfull[s])),
                     "r"((uint32_t)(NMAT * n_rt * (1024 + 128)))
                     : "memory");
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const MatLayout &L = m == 0 ? j.m0 : j.m1;
          for (int q = 0; q < n_rt; ++q) {
            const uint64_t e = ((uint64_t)(rt0 + q) * nb + 2 * c) * 32;
            unsigned char *dn = rs + m * (4 * 1024 + 4 * 128) + q * 1024;
            unsigned char *ds = rs + m * (4 * 1024 + 4 * 128) + 4 * 1024 + q * 128;
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 1024, [%2];" ::"r"(
                    gsa(dn)),
                "l"(slot + L.nib_off + e * 16), "r"(gsa(&rfull[s]))
                : "memory");
            asm volatile(
                "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], 128, [%2];" ::"r"(
                    gsa(ds)),
                "l"(slot + L.sc_off + e * 2), "r"(gsa(&rfull[s]))
                : "memory");
          }
        }
      }
    }
  } else if (warp < 4) {
    // ---- dequant: row r of the tile, both matrices, raw smem -> swizzled bf16
    const int r = tid;
    const bool valid = (r >> 5) < n_rt;
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % kStages, rsi = c % kRawStages;
      if (c >= kStages && !g_mbar_wait(&empty[s], (uint32_t)((c / kStages) - 1) & 1u)) { s_fail = 1; break; }
      if (!g_mbar_wait(&rfull[rsi], (uint32_t)(c / kRawStages) & 1u)) { s_fail = 1; break; }
      const unsigned char *rs = raw + (size_t)rsi * raw_stage_bytes<NMAT>();
      unsigned char *st = sm + (size_t)s * gemm_stage_bytes<NMAT>();
#pragma unroll
      for (int m = 0; m < NMAT; ++m) {
        unsigned char *a = st + (size_t)m * kGemmM * 128;
#pragma unroll
        for (int bi = 0; bi < 2; ++bi) {
          uint4 q = make_uint4(0x88888888u, 0x88888888u, 0x88888888u, 0x88888888u);
          float d = 0.f;
          if (valid) {
            const unsigned char *rm = rs + m * (4 * 1024 + 4 * 128);
            q = *reinterpret_cast<const uint4 *>(rm + (r >> 5) * 1024 + bi * 512 + (r & 31) * 16);
            d = __half2float(__ushort_as_half(
                *reinterpret_cast<const unsigned short *>(rm + 4 * 1024 + (r >> 5) * 128 + bi * 64 + (r & 31) * 2)));
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
                                   ((p01 >> 4) & 0x000F000Fu) | 0x43004300u,
                                   ((p23 >> 4) & 0x000F000Fu) | 0x43004300u};
            __nv_bfloat162 o[4];
#pragma unroll
            for (int z = 0; z < 4; ++z)
              o[z] = __hmul2(__hsub2(*reinterpret_cast<const __nv_bfloat162 *>(&v[z]), k136), d2);
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
      }
      g_mbar_arrive(&rempty[rsi]);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      g_mbar_arrive(&full[s]);
    }
  } else if (warp < 6) {
    // ---- gather the pairs' input rows (nr rows, zero padding past n) with
    // cp.async; a chunk is published once it landed
    const int t = tid - 128;  // 0..63
    const int K = 32 * nb;
    for (int c = 0; c < n_chunks; ++c) {
      const int s = c % kStages;
      if (c >= kStages && !g_mbar_wait(&empty[s], (uint32_t)((c / kStages) - 1) & 1u)) { s_fail = 1; break; }
      unsigned char *bsm = sm + (size_t)s * gemm_stage_bytes<NMAT>() + (size_t)NMAT * kGemmM * 128;
      for (int i = t; i < nr * 8; i += 64) {
        const int rr = i >> 3, cc = i & 7;
        unsigned char *dst = bsm + sw128_off(rr, cc);
        const int src_row = s_rows[rr];
        if (src_row >= 0) {
          const __nv_bfloat16 *src = j.x + (size_t)(src_row / j.x_div) * K + c * kGemmK + cc * 8;
          asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(gsa(dst)), "l"(src) : "memory");
        } else {
          *reinterpret_cast<uint4 *>(dst) = make_uint4(0, 0, 0, 0);
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
      // publish the previous chunk: its copies have landed once at most one
      // group (this one) is pending.  Publishing one behind (not kStages - 1)
      // keeps the publication of chunk c independent of the MMA of chunk c - 1.
      if (c >= 1) {
        asm volatile("cp.async.wait_group 1;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        g_mbar_arrive(&full[(c - 1) % kStages]);
      }
    }
    asm volatile("cp.async.wait_all;" ::: "memory");
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    if (n_chunks >= 1) g_mbar_arrive(&full[(n_chunks - 1) % kStages]);
  } else if (warp == 6) {
    // ---- MMA issuer
    if (lane == 0) {
      const uint32_t idesc = idesc_bf16(kGemmM, nr);
      bool ok = true;
      for (int c = 0; c < n_chunks && ok; ++c) {
        const int s = c % kStages;
        if (!g_mbar_wait(&full[s], (uint32_t)(c / kStages) & 1u)) { ok = false; s_fail = 1; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        unsigned char *st = sm + (size_t)s * gemm_stage_bytes<NMAT>();
        const uint32_t b_addr = gsa(st + (size_t)NMAT * kGemmM * 128);
#pragma unroll
        for (int m = 0; m < NMAT; ++m) {
          const uint32_t a_addr = gsa(st + (size_t)m * kGemmM * 128);
#pragma unroll
          for (int ks = 0; ks < kGemmK / 16; ++ks)
            umma(tmem + (uint32_t)(m * kGemmN), sw128_desc(a_addr + ks * 32), sw128_desc(b_addr + ks * 32), idesc,
                 (c > 0 || ks > 0) ? 1u : 0u);
        }
        umma_commit(&empty[s]);
      }
      if (ok) umma_commit(&done);
    }
  }

  // ---- epilogue (warps 0-3 own TMEM lanes 0-127 = the tile's rows)
  if (warp < 4) {
    const bool ok = !s_fail && g_mbar_wait(&done, 0);
    if (!ok) {
      s_fail = 1;
    } else {
      asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
      const int row = m0 + tid;
      const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);
      for (int c0 = 0; c0 < nr; c0 += 16) {
        float g[16], u[16];
        tmem_ld16(lane_addr + c0, g);
        if (NMAT == 2) tmem_ld16(lane_addr + kGemmN + c0, u);
        if (row < j.R) {
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int col = c0 + i;
            if (col < n) {
              const int pair = s_rows[col];
              if (NMAT == 2)
                j.h16[(size_t)pair * j.R + row] = __float2bfloat16_rn(g[i] / (1.f + expf(-g[i])) * u[i]);
              else
                j.y[(size_t)pair * j.R + row] = g[i];
            }
          }
        }
      }
    }
  }
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
  __syncthreads();
  if (s_fail && tid == 0 && j.err) atomicExch(j.err, 4);
  if (warp == 7) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(kCols));
}

template <int NMAT>
cudaError_t launch_gemm_t(const GemmJob &j, int max_gunits, cudaStream_t st) {
  if (max_gunits <= 0) return cudaSuccess;
  if (j.nb % 2) return cudaErrorInvalidValue;
  const size_t smem = gemm_smem_bytes<NMAT>();
  static size_t cur = 0;
  const cudaError_t e = ensure_dyn_smem(umma_gemm_kernel<NMAT>, smem, cur);
  if (e != cudaSuccess) return e;
  dim3 grid((j.R + kGemmM - 1) / kGemmM, max_gunits);
  umma_gemm_kernel<NMAT><<<grid, kGemmThreads, smem, st>>>(j);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_gemm_gateup(const FfnArgs &a, const __nv_bfloat16 *x, const WorkUnit *gunits,
                               const int32_t *gunit_begin, __nv_bfloat16 *h16, int range_kind, int stage,
                               int max_gunits, cudaStream_t st) {
  GemmJob j;
  j.slots = a.slots;
  j.slot_stride = a.slot_stride;
  j.m0 = a.lay.gate;
  j.m1 = a.lay.up;
  j.R = a.F;
  j.nb = a.H / 32;
  j.x = x;
  j.x_div = a.k;
  j.perm = a.perm;
  j.items = a.items;
  j.gunits = gunits;
  j.gunit_begin = gunit_begin;
  j.hdr = a.hdr;
  j.range_kind = range_kind;
  j.stage = stage;
  j.h16 = h16;
  j.y = nullptr;
  j.err = a.err;
  return launch_gemm_t<2>(j, max_gunits, st);
}

cudaError_t launch_gemm_down(const FfnArgs &a, const __nv_bfloat16 *h16, const WorkUnit *gunits,
                             const int32_t *gunit_begin, int range_kind, int stage, int max_gunits,
                             cudaStream_t st) {
  GemmJob j;
  j.slots = a.slots;
  j.slot_stride = a.slot_stride;
  j.m0 = a.lay.down;
  j.m1 = a.lay.down;
  j.R = a.H;
  j.nb = a.F / 32;
  j.x = h16;
  j.x_div = 1;
  j.perm = a.perm;
  j.items = a.items;
  j.gunits = gunits;
  j.gunit_begin = gunit_begin;
  j.hdr = a.hdr;
  j.range_kind = range_kind;
  j.stage = stage;
  j.h16 = nullptr;
  j.y = a.y;
  j.err = a.err;
  return launch_gemm_t<1>(j, max_gunits, st);
}

}  // namespace moe
