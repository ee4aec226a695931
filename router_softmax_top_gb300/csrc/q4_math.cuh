// Q4_0 GEMV building blocks shared by the decode-path kernels (tile GEMV,
// down + combine, fused miss, decode layer kernel): CTA shape, bounded
// mbarrier and copy helpers, the nibble decode and the per-block dot product
// in the one canonical order every kernel of the path uses.
#pragma once

#include "common.cuh"

namespace moe {
namespace q4 {

constexpr int kWarps = 8;
constexpr int kThreads = 32 * kWarps;
constexpr uint32_t kSpinLimit = 1u << 26;  // bounded mbarrier waits

// ------------------------------------------------------------ PTX helpers
__device__ __forceinline__ uint32_t smem_u32(const void *p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void fence_proxy_async() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
// Raises the barrier's expected transaction bytes without an arrival (the
// arrival comes separately, once the rest of the phase's data is written).
__device__ __forceinline__ void mbar_expect_tx_only(uint64_t *bar, uint32_t bytes) {
  asm volatile("mbarrier.expect_tx.relaxed.cta.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
          smem_u32(dst)),
      "l"(src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for phase `parity` of bar; gives up after kSpinLimit polls.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity) {
  for (uint32_t i = 0; i < kSpinLimit; ++i)
    if (mbar_try_wait(bar, parity)) return true;
  return false;
}
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
  asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
__device__ __forceinline__ void cp_async_wait1() { asm volatile("cp.async.wait_group 1;" ::: "memory"); }

// Records a device-side failure (a bulk copy that never completed) in the
// handle's mapped error word.
__device__ __forceinline__ void flag_error(int32_t *err, int code) {
  if (err) atomicExch(err, code);
}

// ----------------------------------------------------------- Q4_0 math
// Four nibbles, one per byte of v (values 0..15), as floats 0.5 + q/256: the
// byte lands in bits 16..19 under exponent 126, so no conversion instruction is
// needed.  sum (0.5 + q/256) x = X/2 + (sum q x)/256, hence
// sum (q - 8) x = 256 s - 136 X with X = sum x.
__device__ __forceinline__ float nib_f(uint32_t v, int byte) {
  return __int_as_float(__byte_perm(v, 0x3F000000u, 0x7054u | ((uint32_t)byte << 8)));
}

__device__ __forceinline__ void decode_block(const uint4 q, float f[32]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0x0F0F0F0Fu;
    const uint32_t hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      f[4 * i + b] = nib_f(lo, b);
      f[16 + 4 * i + b] = nib_f(hi, b);
    }
  }
}

// s = sum_j f_j x_j over one block (x from shared memory, broadcast reads).
__device__ __forceinline__ float dot32(const float f[32], const float *xb) {
  float s0 = 0.f, s1 = 0.f;
#pragma unroll
  for (int i = 0; i < 16; i += 4) {
    const float4 a = *reinterpret_cast<const float4 *>(xb + i);
    const float4 b = *reinterpret_cast<const float4 *>(xb + 16 + i);
    s0 = fmaf(f[i + 0], a.x, s0);
    s0 = fmaf(f[i + 1], a.y, s0);
    s0 = fmaf(f[i + 2], a.z, s0);
    s0 = fmaf(f[i + 3], a.w, s0);
    s1 = fmaf(f[16 + i + 0], b.x, s1);
    s1 = fmaf(f[16 + i + 1], b.y, s1);
    s1 = fmaf(f[16 + i + 2], b.z, s1);
    s1 = fmaf(f[16 + i + 3], b.w, s1);
  }
  return s0 + s1;
}

// acc + d * (sum (q - 8) x) for one block.
__device__ __forceinline__ float block_term(const float f[32], float d, const float *xb,
                                            float xsum, float acc) {
  return fmaf(d, fmaf(256.f, dot32(f, xb), -136.f * xsum), acc);
}

__device__ __forceinline__ float half_bits(unsigned short v) {
  return __half2float(__ushort_as_half(v));
}

// Stage n input rows of K values (fp32 or bf16) into shared memory and the
// per-block sums X_b (one warp per block: lane j holds value j, fixed xor tree).
// l2_only: read through L2 only (inputs written by other CTAs of the same kernel).
__device__ __forceinline__ void stage_rows(float *xs, float *xsum, const void *x, int x_bf16,
                                           const int *rows, int n, int K, bool l2_only = false) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nb = K / 32;
  for (int t = 0; t < n; ++t) {
    const int row = rows[t];
    if (x_bf16) {
      const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(x) + (size_t)row * K;
      for (int c = tid; c < K; c += kThreads) xs[t * K + c] = __bfloat162float(src[c]);
    } else {
      const float4 *src =
          reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(x) + (size_t)row * K);
      float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)t * K);
      if (l2_only)
        for (int c = tid; c < K / 4; c += kThreads) dst[c] = __ldcg(src + c);
      else
        for (int c = tid; c < K / 4; c += kThreads) dst[c] = src[c];
    }
  }
  __syncthreads();
  for (int i = warp; i < n * nb; i += kWarps) {
    float v = xs[(size_t)i * 32 + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) xsum[i] = v;
  }
  __syncthreads();
}

__device__ __forceinline__ int ld_acquire(const int32_t *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}

// One block of one row read from the canonical tile in shared memory:
// returns the 16 nibble bytes and writes the scale bits.
__device__ __forceinline__ uint4 canon_block(const unsigned char *canon, int row, int b, int nb,
                                             unsigned short &dbits) {
  const unsigned short *blk = reinterpret_cast<const unsigned short *>(canon + ((size_t)row * nb + b) * 18);
  dbits = blk[0];
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = (uint32_t)blk[1 + 2 * i] | ((uint32_t)blk[2 + 2 * i] << 16);
  return make_uint4(v[0], v[1], v[2], v[3]);
}

}  // namespace q4
}  // namespace moe
