// Expert FFN kernels of the GEMV (decode / small-batch) path and the slot fill.
//
//  * repack_kernel: one missed canonical Q4_0 expert block (from the staging
//    area or straight from the mapped host store) -> repacked slot planes.
//  * q4_gemv_kernel<2>: gate and up rows of one expert for up to 8 of its
//    tokens, then h = silu(g) * u ("llama.cpp + MoE expert cache",
//    "Limitations": merged gate/up, SiLU).
//  * q4_gemv_kernel<1>: down rows, y = W_down h per pair.
//  * combine_kernel: out_t = sum over picks in ascending order of w * y
//    ("The idea: cache the hot experts on the GPU", step 4).
//
// Each output of a pair is computed by the same code in the same order
// whatever the slot, the stage or the other tokens of its work unit, so the
// result does not depend on the slot budget.
#include "common.cuh"

namespace moe {
namespace {

constexpr int kGemvThreads = 256;
constexpr int kGemvWarps = kGemvThreads / 32;

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

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

__device__ __forceinline__ unsigned short ld_stream_u16(const void *p) {
  unsigned short r;
  asm volatile("ld.global.nc.L1::no_allocate.u16 %0, [%1];" : "=h"(r) : "l"(p));
  return r;
}

struct GemvJob {
  const uint8_t *slots;
  uint64_t slot_stride;
  MatLayout m0, m1;  // m1 used when two matrices share the input (gate, up)
  int R, nb;         // rows and 32-blocks per row
  const void *x;     // rows of K = 32 nb values
  int x_bf16;
  int x_div;         // input row of pair p is p / x_div
  const int32_t *perm;
  const WorkItem *items;
  const WorkUnit *units;
  const int32_t *unit_begin;
  const PlanHdr *hdr;
  int range_kind, stage;
  float *out;        // out[pair * R + r]
  int max_tok;       // tokens per unit the shared memory was sized for
};

__device__ __forceinline__ bool unit_range(const PlanHdr *h, const int32_t *ub, int kind, int stage,
                                           int &lo, int &hi) {
  if (h->error || stage >= h->n_stages) return false;
  if (kind == 0) { lo = 0; hi = h->hit_units; }
  else if (kind == 1) { lo = stage == 0 ? h->hit_units : ub[stage]; hi = ub[stage + 1]; }
  else { lo = ub[stage]; hi = ub[stage + 1]; }
  return true;
}

template <int NMAT>
__global__ void __launch_bounds__(kGemvThreads) q4_gemv_kernel(GemvJob j) {
  int lo, hi;
  if (!unit_range(j.hdr, j.unit_begin, j.range_kind, j.stage, lo, hi)) return;
  const int u = lo + (int)blockIdx.y;
  if (u >= hi) return;
  const WorkUnit wu = j.units[u];
  const WorkItem it = j.items[wu.item];
  const int n = wu.pair_count;
  const int K = 32 * j.nb, nb = j.nb, R = j.R;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(16) float sm[];
  float *xs = sm;                                  // [max_tok][K]
  float *xsum = xs + (size_t)j.max_tok * K;        // [max_tok][nb]
  float *red = xsum + (size_t)j.max_tok * nb;      // [warps][NMAT][max_tok][32]

  for (int t = 0; t < n; ++t) {
    const int pair = j.perm[wu.pair_begin + t];
    const int row = pair / j.x_div;
    if (j.x_bf16) {
      const __nv_bfloat16 *src = reinterpret_cast<const __nv_bfloat16 *>(j.x) + (size_t)row * K;
      for (int c = tid; c < K; c += kGemvThreads) xs[t * K + c] = __bfloat162float(src[c]);
    } else {
      const float4 *src = reinterpret_cast<const float4 *>(reinterpret_cast<const float *>(j.x) +
                                                           (size_t)row * K);
      float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)t * K);
      for (int c = tid; c < K / 4; c += kGemvThreads) dst[c] = src[c];
    }
  }
  __syncthreads();
  for (int i = tid; i < n * nb; i += kGemvThreads) {
    const int t = i / nb, b = i - t * nb;
    const float *xb = xs + (size_t)t * K + 32 * b;
    float s = 0.f;
#pragma unroll
    for (int q = 0; q < 32; ++q) s += xb[q];
    xsum[t * nb + b] = s;
  }
  __syncthreads();

  const int r = blockIdx.x * 32 + lane;
  const uint8_t *slot = j.slots + (uint64_t)it.slot * j.slot_stride;
  const uint4 *nib0 = reinterpret_cast<const uint4 *>(slot + j.m0.nib_off);
  const unsigned short *sc0 = reinterpret_cast<const unsigned short *>(slot + j.m0.sc_off);
  const uint4 *nib1 = reinterpret_cast<const uint4 *>(slot + j.m1.nib_off);
  const unsigned short *sc1 = reinterpret_cast<const unsigned short *>(slot + j.m1.sc_off);

  const int bpw = (nb + kGemvWarps - 1) / kGemvWarps;
  const int b0 = warp * bpw, b1 = min(nb, b0 + bpw);
  float acc0[kTokPerUnit], acc1[kTokPerUnit];
#pragma unroll
  for (int t = 0; t < kTokPerUnit; ++t) { acc0[t] = 0.f; acc1[t] = 0.f; }

  for (int b = b0; b < b1; ++b) {
    const size_t e = (size_t)b * R + r;
    const uint4 q0 = ld_stream(nib0 + e);
    const float d0 = __half2float(__ushort_as_half(ld_stream_u16(sc0 + e)));
    float f0[32];
    decode_block(q0, f0);
    float f1[32];
    float d1 = 0.f;
    if (NMAT == 2) {
      const uint4 q1 = ld_stream(nib1 + e);
      d1 = __half2float(__ushort_as_half(ld_stream_u16(sc1 + e)));
      decode_block(q1, f1);
    }
#pragma unroll
    for (int t = 0; t < kTokPerUnit; ++t) {
      if (t < n) {
        const float *xb = xs + (size_t)t * K + 32 * b;
        const float cx = -136.f * xsum[t * nb + b];
        const float s0 = dot32(f0, xb);
        acc0[t] = fmaf(d0, fmaf(256.f, s0, cx), acc0[t]);
        if (NMAT == 2) {
          const float s1 = dot32(f1, xb);
          acc1[t] = fmaf(d1, fmaf(256.f, s1, cx), acc1[t]);
        }
      }
    }
  }
#pragma unroll
  for (int t = 0; t < kTokPerUnit; ++t) {
    if (t < n) {
      red[((warp * NMAT + 0) * j.max_tok + t) * 32 + lane] = acc0[t];
      if (NMAT == 2) red[((warp * NMAT + 1) * j.max_tok + t) * 32 + lane] = acc1[t];
    }
  }
  __syncthreads();
  // warp t finishes token t (fixed summation order over the K-split warps)
  for (int t = warp; t < n; t += kGemvWarps) {
    float g = 0.f, v = 0.f;
    for (int w = 0; w < kGemvWarps; ++w) {
      g += red[((w * NMAT + 0) * j.max_tok + t) * 32 + lane];
      if (NMAT == 2) v += red[((w * NMAT + 1) * j.max_tok + t) * 32 + lane];
    }
    const int pair = j.perm[wu.pair_begin + t];
    float o;
    if (NMAT == 2) o = g / (1.f + expf(-g)) * v;
    else o = g;
    j.out[(size_t)pair * R + r] = o;
  }
}

size_t gemv_smem(int NMAT, int max_tok, int nb) {
  return sizeof(float) * ((size_t)max_tok * 32 * nb + (size_t)max_tok * nb +
                          (size_t)kGemvWarps * NMAT * max_tok * 32);
}

template <int NMAT>
cudaError_t launch_gemv(GemvJob j, int max_units, cudaStream_t st) {
  if (max_units <= 0) return cudaSuccess;
  const size_t smem = gemv_smem(NMAT, j.max_tok, j.nb);
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(q4_gemv_kernel<NMAT>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  dim3 grid(j.R / 32, max_units);
  q4_gemv_kernel<NMAT><<<grid, kGemvThreads, smem, st>>>(j);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- repack
struct RepackJob {
  RepackArgs a;
  int S;
};

__global__ void __launch_bounds__(256) repack_kernel(RepackJob jb) {
  const RepackArgs &a = jb.a;
  const PlanHdr *h = a.hdr;
  if (h->error || a.stage >= h->n_stages) return;
  const int n0 = h->n_stage0_miss, nM = h->n_miss, S = jb.S;
  int m_lo, m_hi;
  if (a.stage == 0) { m_lo = 0; m_hi = n0; }
  else { m_lo = n0 + (a.stage - 1) * S; m_hi = min(nM, n0 + a.stage * S); }
  const int mi = m_lo + (int)blockIdx.y;
  if (mi >= m_hi) return;
  const MissItem m = a.miss[mi];
  const uint8_t *src = a.by_expert
                           ? a.src_base + a.src_layer_off + (uint64_t)m.expert * a.src_expert_stride
                           : a.src_base + (uint64_t)(mi - m_lo) * a.src_slot_stride;
  uint8_t *dst = a.slots + (uint64_t)m.slot * a.slot_stride;

  const int tg = a.lay.gate.rows / 32, td = a.lay.down.rows / 32;
  int tile = blockIdx.x;
  const MatLayout *L;
  if (tile < tg) L = &a.lay.gate;
  else if (tile < 2 * tg) { L = &a.lay.up; tile -= tg; }
  else { L = &a.lay.down; tile -= 2 * tg; }
  (void)td;
  const int R = L->rows, nb = L->nb, r0 = tile * 32;
  // the canonical matrix starts where its nibble plane starts (same byte count)
  const uint4 *csrc = reinterpret_cast<const uint4 *>(src + L->nib_off + (uint64_t)r0 * nb * 18);
  const int n16 = 32 * nb * 18 / 16;

  extern __shared__ __align__(16) unsigned char rs[];
  uint4 *s4 = reinterpret_cast<uint4 *>(rs);
  // plain loads: the source may be mapped host memory
  for (int i = threadIdx.x; i < n16; i += blockDim.x) s4[i] = csrc[i];
  __syncthreads();

  uint4 *nib = reinterpret_cast<uint4 *>(dst + L->nib_off);
  unsigned short *sc = reinterpret_cast<unsigned short *>(dst + L->sc_off);
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nw = blockDim.x >> 5;
  for (int b = warp; b < nb; b += nw) {
    const unsigned short *blk = reinterpret_cast<const unsigned short *>(rs + ((size_t)lane * nb + b) * 18);
    uint32_t v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) v[i] = (uint32_t)blk[1 + 2 * i] | ((uint32_t)blk[2 + 2 * i] << 16);
    const size_t e = (size_t)b * R + r0 + lane;
    nib[e] = make_uint4(v[0], v[1], v[2], v[3]);
    sc[e] = blk[0];
  }
}

// ---------------------------------------------------------------- combine
__global__ void combine_kernel(const float *y, const float *w, const PlanHdr *hdr, int T, int k,
                               int H, float *out) {
  if (hdr->error) return;
  const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  if (i >= (size_t)T * H) return;
  const int t = (int)(i / H), c = (int)(i - (size_t)t * H);
  float acc = 0.f;
  for (int q = 0; q < k; ++q) acc = fmaf(w[t * k + q], y[((size_t)t * k + q) * H + c], acc);
  out[i] = acc;
}

}  // namespace

static int max_tok_for(const FfnArgs &) { return kTokPerUnit; }

cudaError_t launch_gateup(const FfnArgs &a, int range_kind, int stage, int max_units,
                          cudaStream_t st) {
  GemvJob j;
  j.slots = a.slots;
  j.slot_stride = a.slot_stride;
  j.m0 = a.lay.gate;
  j.m1 = a.lay.up;
  j.R = a.F;
  j.nb = a.H / 32;
  j.x = a.x;
  j.x_bf16 = a.x_bf16;
  j.x_div = a.k;
  j.perm = a.perm;
  j.items = a.items;
  j.units = a.units;
  j.unit_begin = a.unit_begin;
  j.hdr = a.hdr;
  j.range_kind = range_kind;
  j.stage = stage;
  j.out = a.h;
  j.max_tok = a.max_tok > 0 ? a.max_tok : max_tok_for(a);
  return launch_gemv<2>(j, max_units, st);
}

cudaError_t launch_down(const FfnArgs &a, int range_kind, int stage, int max_units,
                        cudaStream_t st) {
  GemvJob j;
  j.slots = a.slots;
  j.slot_stride = a.slot_stride;
  j.m0 = a.lay.down;
  j.m1 = a.lay.down;
  j.R = a.H;
  j.nb = a.F / 32;
  j.x = a.h;
  j.x_bf16 = 0;
  j.x_div = 1;
  j.perm = a.perm;
  j.items = a.items;
  j.units = a.units;
  j.unit_begin = a.unit_begin;
  j.hdr = a.hdr;
  j.range_kind = range_kind;
  j.stage = stage;
  j.out = a.y;
  j.max_tok = a.max_tok > 0 ? a.max_tok : max_tok_for(a);
  return launch_gemv<1>(j, max_units, st);
}

cudaError_t launch_combine(const float *y, const float *w, const PlanHdr *hdr, int T, int k, int H,
                           float *out, cudaStream_t st) {
  const size_t n = (size_t)T * H;
  combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, w, hdr, T, k, H, out);
  return cudaGetLastError();
}

size_t repack_smem(const SlotLayout &lay) {
  const int nbmax = lay.gate.nb > lay.down.nb ? lay.gate.nb : lay.down.nb;
  return (size_t)32 * nbmax * 18;
}

cudaError_t launch_repack(const RepackArgs &a, int S, int max_miss, cudaStream_t st) {
  if (max_miss <= 0) return cudaSuccess;
  static bool attr_done = false;
  if (!attr_done) {
    cudaError_t e = cudaFuncSetAttribute(repack_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         227 * 1024);
    if (e != cudaSuccess) return e;
    attr_done = true;
  }
  const size_t smem = repack_smem(a.lay);
  if (smem > 227 * 1024) return cudaErrorInvalidValue;
  RepackJob jb{a, S};
  dim3 grid(2 * a.lay.gate.rows / 32 + a.lay.down.rows / 32, max_miss);
  repack_kernel<<<grid, 256, smem, st>>>(jb);
  return cudaGetLastError();
}

}  // namespace moe
