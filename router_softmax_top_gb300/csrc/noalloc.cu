// moe_expert_ffn_static: one expert's Q4_0 SwiGLU FFN applied to a few tokens,
// with no memory allocation at all.
//
// Who needs it: code that runs where cudaMalloc is not an option -- inside a
// CUDA graph being captured (allocation calls are not capturable), in a real-
// time or signal-handling context that must not block on the allocator, under
// a memory budget that forbids growing the pool, or from a host thread that
// does not own the CUDA context's allocator (plugins living inside another
// framework's process).  Such callers still own their inputs and outputs; the
// only intermediate this computation needs (the SwiGLU activations h of the
// tokens, plus two work counters) lives in a fixed array compiled into the
// library instead of a per-call or per-handle allocation.
//
// The scratch array is file-scope __device__ memory: every GPU that loads this
// library holds it (kScratchBytes) until the process exits, and all calls on a
// device share it.  Calls that overlap on the GPU (two streams at once, or two
// host threads) race on it; serialise them.  Its contents persist between calls;
// the counters that must start at zero are cleared (cudaMemsetAsync, not an
// allocation) at the start of every call.  Host code must not use the array's
// name as a device address: the first call on each device looks up its device
// address with cudaGetSymbolAddress (with that device current) and caches it,
// so that first call should come before any stream capture.
//
// Failure reporting without allocation: a down tile waits (bounded, 2 s) for
// the gate/up tiles of the call.  If that wait gives up, the tile writes NaN
// into its 32 output rows of every token (so a failed call never leaves stale
// values that look valid) and records the failure in a status word of a
// 64 KiB page compiled into the library, which the first call in the process
// page-locks and maps (cudaHostRegister of static memory; nothing is
// allocated).  The first call issued after the failed kernel has finished
// reads the record, clears it, launches nothing and returns MOE_ERR_TIMEOUT.
//
// Cost note: a down tile reads h of every token, but the shared memory holds
// the inputs of at most G tokens at a time (G < T for large hidden or FFN
// widths, e.g. hidden 4096 / FFN 1536 at 8 tokens); each group of G tokens
// then decodes the tile's weights again, once per group.
//
// The arithmetic is that of the library's fused miss kernel: per 32-row tile,
// lane = row, warp w of 8 sums the 32-blocks w, w+8, ... in ascending order,
// the warp partial sums are added in warp order.
#include <cstdlib>
#include <mutex>

#include "common.cuh"
#include "moe_cache.h"

#define MOE_API extern "C" __attribute__((visibility("default")))

namespace moe {
namespace {

constexpr int kNaMaxTok = 8;          // tokens per call
constexpr int kNaMaxDim = 4096;       // hidden and FFN width
constexpr size_t kNaCounterBytes = 256;
constexpr size_t kScratchBytes = kNaCounterBytes + sizeof(float) * kNaMaxTok * kNaMaxDim;  // 128.25 KiB
constexpr int kNaWarps = 8, kNaThreads = 256;
constexpr uint32_t kNaSpin = 1u << 26;
constexpr uint64_t kNaWaitNs = 2000000000ull;       // limit of a down tile's wait
constexpr uint64_t kNaInjectWaitNs = 20000000ull;   // ... under the test injection
constexpr int kNaMaxDevices = 64;
constexpr size_t kNaStatusPage = 65536;  // a whole page also where pages are 64 KiB

// [0, 256): counters (queue head, finished gate/up tiles); then h [T][F] fp32.
static __device__ __align__(256) unsigned char g_noalloc_scratch[kScratchBytes];

// Failure records, one int32 per device 64 bytes apart, in a static page that
// is page-locked and mapped at set-up: the kernel sets its device's word when
// a wait gives up; the host reads and clears it.
alignas(kNaStatusPage) static int32_t g_na_status[kNaStatusPage / sizeof(int32_t)];

__device__ __forceinline__ uint32_t na_smem(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ float na_nib(uint32_t v, int byte) {
  return __int_as_float(__byte_perm(v, 0x3F000000u, 0x7054u | ((uint32_t)byte << 8)));
}

__device__ __forceinline__ void na_decode(const uint4 q, float f[32]) {
  const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const uint32_t lo = w[i] & 0x0F0F0F0Fu, hi = (w[i] >> 4) & 0x0F0F0F0Fu;
#pragma unroll
    for (int b = 0; b < 4; ++b) {
      f[4 * i + b] = na_nib(lo, b);
      f[16 + 4 * i + b] = na_nib(hi, b);
    }
  }
}

// acc + d * sum_j (q_j - 8) x_j, with f_j = 0.5 + q_j/256 (see the fused miss kernel).
__device__ __forceinline__ float na_term(const float f[32], float d, const float *xb, float xsum,
                                         float acc) {
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
  return fmaf(d, fmaf(256.f, s0 + s1, -136.f * xsum), acc);
}

__device__ __forceinline__ uint4 na_block(const unsigned char *canon, int row, int b, int nb,
                                          unsigned short &dbits) {
  const unsigned short *blk = reinterpret_cast<const unsigned short *>(canon + ((size_t)row * nb + b) * 18);
  dbits = blk[0];
  uint32_t v[4];
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = (uint32_t)blk[1 + 2 * i] | ((uint32_t)blk[2 + 2 * i] << 16);
  return make_uint4(v[0], v[1], v[2], v[3]);
}

__device__ __forceinline__ void na_stage(float *xs, float *xsum, const float *x, int n, int K,
                                         bool l2_only) {
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nb = K / 32;
  for (int t = 0; t < n; ++t) {
    const float4 *src = reinterpret_cast<const float4 *>(x + (size_t)t * K);
    float4 *dst = reinterpret_cast<float4 *>(xs + (size_t)t * K);
    if (l2_only)
      for (int c = tid; c < K / 4; c += kNaThreads) dst[c] = __ldcg(src + c);
    else
      for (int c = tid; c < K / 4; c += kNaThreads) dst[c] = src[c];
  }
  __syncthreads();
  for (int i = warp; i < n * nb; i += kNaWarps) {
    float v = xs[(size_t)i * 32 + lane];
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    if (lane == 0) xsum[i] = v;
  }
  __syncthreads();
}

struct NaJob {
  const uint8_t *blk;  // canonical expert block [gate | up | down]
  int H, F, T;
  int G;               // tokens per shared-memory input group
  const float *x;      // [T, H]
  float *y;            // [T, H]
  unsigned char *scratch;
  int32_t *status;     // device alias of this device's failure record (mapped host word)
  int inject;          // test hook: down tiles wait for a count that is never reached
  uint64_t wait_ns;    // limit of a down tile's wait
};

__device__ __forceinline__ uint64_t na_now_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

size_t na_smem(int nbH, int nbF, int G) {
  const size_t canon = (size_t)32 * 18 * (2 * nbH > nbF ? 2 * nbH : nbF);
  const int kmax = 32 * (nbH > nbF ? nbH : nbF), nbmax = nbH > nbF ? nbH : nbF;
  return canon + sizeof(float) * ((size_t)G * kmax + (size_t)G * nbmax + (size_t)kNaWarps * 2 * G * 32);
}

// Work queue: F/32 gate/up tiles (32 rows of gate and of up), then H/32 down
// tiles; a down tile waits (bounded) until every gate/up tile has written h.
__global__ void __launch_bounds__(kNaThreads) expert_ffn_static_kernel(NaJob j) {
  const int nbH = j.H / 32, nbF = j.F / 32, tF = j.F / 32, tH = j.H / 32, T = j.T, G = j.G;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  int *counters = reinterpret_cast<int *>(j.scratch);
  float *h = reinterpret_cast<float *>(j.scratch + kNaCounterBytes);
  extern __shared__ __align__(128) unsigned char sm[];
  const size_t canon_bytes = (size_t)32 * 18 * (2 * nbH > nbF ? 2 * nbH : nbF);
  unsigned char *canon = sm;
  float *xs = reinterpret_cast<float *>(sm + canon_bytes);
  const int kmax = 32 * (nbH > nbF ? nbH : nbF), nbmax = nbH > nbF ? nbH : nbF;
  float *xsum = xs + (size_t)G * kmax;
  float *red = xsum + (size_t)G * nbmax;  // [warps][2][G][32]
  __shared__ int s_wk, s_ok;
  const uint64_t gate_off = 0, mat_gu = (uint64_t)j.F * nbH * 18;
  const uint64_t up_off = mat_gu, down_off = 2 * mat_gu;

  for (;;) {
    if (tid == 0) s_wk = atomicAdd(&counters[0], 1);
    __syncthreads();
    const int wk = s_wk;
    if (wk >= tF + tH) break;
    const bool gu = wk < tF;
    const int t = gu ? wk : wk - tF;
    const int nb = gu ? nbH : nbF, K = 32 * nb;
    const size_t tile_bytes = (size_t)32 * nb * 18;
    const int nmat = gu ? 2 : 1;
    for (int mm = 0; mm < nmat; ++mm) {
      const uint8_t *src = j.blk + (gu ? (mm == 0 ? gate_off : up_off) : down_off) + (uint64_t)t * tile_bytes;
      for (int i = tid; i < (int)(tile_bytes / 16); i += kNaThreads) {
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(na_smem(canon + mm * tile_bytes + 16 * i)),
                     "l"(src + 16 * i)
                     : "memory");
      }
    }
    asm volatile("cp.async.commit_group;" ::: "memory");
    if (!gu) {
      if (tid == 0) {
        // every gate/up tile has written h once counters[1] reaches tF (the
        // injected fault waits for one more, which never comes)
        const int need = j.inject ? tF + 1 : tF;
        int ok = 0;
        uint64_t t0 = 0;
        for (uint32_t i = 0; i < kNaSpin; ++i) {
          int v;
          asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(&counters[1]) : "memory");
          if (v >= need) { ok = 1; break; }
          if ((i & 63u) == 63u) {
            const uint64_t now = na_now_ns();
            if (t0 == 0) t0 = now;
            else if (now - t0 > j.wait_ns) break;
          }
          __nanosleep(64);
        }
        s_ok = ok;
      }
      __syncthreads();
      if (!s_ok) {
        // gave up: this tile's rows of y become NaN for every token and the
        // failure is recorded for the host; no copy may still be landing
        asm volatile("cp.async.wait_all;" ::: "memory");
        for (int i = tid; i < T * 32; i += kNaThreads)
          j.y[(size_t)(i >> 5) * j.H + t * 32 + (i & 31)] = __int_as_float(0x7fc00000);
        if (tid == 0) {
          asm volatile("st.relaxed.sys.global.b32 [%0], %1;" ::"l"(j.status), "r"(1) : "memory");
          __threadfence_system();
        }
        continue;
      }
    }
    for (int g0 = 0; g0 < T; g0 += G) {
      const int gn = min(G, T - g0);
      na_stage(xs, xsum, (gu ? j.x : h) + (size_t)g0 * K, gn, K, !gu);
      if (g0 == 0) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
      }
      float acc0[kNaMaxTok], acc1[kNaMaxTok];
#pragma unroll
      for (int q = 0; q < kNaMaxTok; ++q) { acc0[q] = 0.f; acc1[q] = 0.f; }
#pragma unroll 1
      for (int b = warp; b < nb; b += kNaWarps) {
        float f0[32], f1[32];
        unsigned short d0b, d1b = 0;
        na_decode(na_block(canon, lane, b, nb, d0b), f0);
        if (gu) na_decode(na_block(canon + tile_bytes, lane, b, nb, d1b), f1);
        const float d0 = __half2float(__ushort_as_half(d0b)), d1 = __half2float(__ushort_as_half(d1b));
#pragma unroll
        for (int q = 0; q < kNaMaxTok; ++q) {
          if (q < gn) {
            const float *xb = xs + (size_t)q * K + 32 * b;
            acc0[q] = na_term(f0, d0, xb, xsum[q * nb + b], acc0[q]);
            if (gu) acc1[q] = na_term(f1, d1, xb, xsum[q * nb + b], acc1[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kNaMaxTok; ++q) {
        if (q < gn) {
          red[((warp * 2 + 0) * G + q) * 32 + lane] = acc0[q];
          red[((warp * 2 + 1) * G + q) * 32 + lane] = acc1[q];
        }
      }
      __syncthreads();
      for (int q = warp; q < gn; q += kNaWarps) {
        float g = 0.f, v = 0.f;
        for (int w = 0; w < kNaWarps; ++w) {
          g += red[((w * 2 + 0) * G + q) * 32 + lane];
          if (gu) v += red[((w * 2 + 1) * G + q) * 32 + lane];
        }
        if (gu) h[(size_t)(g0 + q) * j.F + t * 32 + lane] = g / (1.f + expf(-g)) * v;
        else j.y[(size_t)(g0 + q) * j.H + t * 32 + lane] = g;
      }
      __syncthreads();
    }
    if (gu && tid == 0) {
      __threadfence();
      atomicAdd(&counters[1], 1);
    }
  }
}

std::mutex g_na_mu;
void *g_na_ptr[kNaMaxDevices] = {};       // device address of g_noalloc_scratch, per device
int32_t *g_na_dstatus[kNaMaxDevices] = {};  // device alias of the device's failure record
bool g_na_status_mapped = false;          // the status page is page-locked and mapped
size_t g_na_smem_set[kNaMaxDevices] = {};

// Test hook: MOE_STATIC_INJECT_WAIT=1 in the environment makes the down tiles
// of a call wait for a gate/up count that is never reached, so that their
// bounded wait gives up (after kNaInjectWaitNs) and the failure path runs.
bool na_inject() {
  const char *v = getenv("MOE_STATIC_INJECT_WAIT");
  return v && v[0] == '1';
}

}  // namespace
}  // namespace moe

using namespace moe;

MOE_API int moe_expert_ffn_static(const void *d_expert_block, int32_t hidden, int32_t ffn,
                                  const float *d_x, int32_t n_tokens, float *d_y, void *cuda_stream) {
  if (n_tokens == 0) return MOE_OK;
  if (!d_expert_block || !d_x || !d_y || n_tokens < 0) return MOE_ERR_INVALID_ARG;
  if (n_tokens > kNaMaxTok || hidden < 64 || ffn < 64 || hidden % 64 || ffn % 64 ||
      hidden > kNaMaxDim || ffn > kNaMaxDim)
    return MOE_ERR_UNSUPPORTED;
  if ((uintptr_t)d_expert_block % 16 || (uintptr_t)d_x % 16 || (uintptr_t)d_y % 16)
    return MOE_ERR_INVALID_ARG;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kNaMaxDevices) return MOE_ERR_CUDA;
  int G = n_tokens;
  while (G > 1 && na_smem(hidden / 32, ffn / 32, G) > 200 * 1024) --G;
  const size_t smem = na_smem(hidden / 32, ffn / 32, G);
  if (smem > 200 * 1024) return MOE_ERR_UNSUPPORTED;
  void *scratch = nullptr;
  int32_t *dstatus = nullptr;
  {
    // set-up, once per device (the status page once per process), and the
    // kernel's shared-memory limit, which only ever grows
    std::lock_guard<std::mutex> lock(g_na_mu);
    if (!g_na_status_mapped) {
      if (cudaHostRegister(g_na_status, sizeof(g_na_status), cudaHostRegisterMapped | cudaHostRegisterPortable) !=
          cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      g_na_status_mapped = true;
    }
    if (!g_na_ptr[dev]) {
      void *p = nullptr, *ps = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || !p ||
          cudaHostGetDevicePointer(&ps, &g_na_status[dev * 16], 0) != cudaSuccess || !ps) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      g_na_dstatus[dev] = static_cast<int32_t *>(ps);
      g_na_ptr[dev] = p;
    }
    if (smem > g_na_smem_set[dev] && smem > 48 * 1024) {
      if (cudaFuncSetAttribute(expert_ffn_static_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               (int)smem) != cudaSuccess) {
        cudaGetLastError();
        return MOE_ERR_CUDA;
      }
      g_na_smem_set[dev] = smem;
    }
    scratch = g_na_ptr[dev];
    dstatus = g_na_dstatus[dev];
  }
  // a failure recorded by an earlier call that has finished on the GPU
  if (__atomic_exchange_n(&g_na_status[dev * 16], 0, __ATOMIC_ACQ_REL) != 0) return MOE_ERR_TIMEOUT;
  cudaStream_t st = (cudaStream_t)cuda_stream;
  if (cudaMemsetAsync(scratch, 0, kNaCounterBytes, st) != cudaSuccess) return MOE_ERR_CUDA;
  NaJob j;
  j.blk = static_cast<const uint8_t *>(d_expert_block);
  j.H = hidden;
  j.F = ffn;
  j.T = n_tokens;
  j.G = G;
  j.x = d_x;
  j.y = d_y;
  j.scratch = static_cast<unsigned char *>(scratch);
  j.status = dstatus;
  j.inject = na_inject() ? 1 : 0;
  j.wait_ns = j.inject ? kNaInjectWaitNs : kNaWaitNs;
  const int items = ffn / 32 + hidden / 32;
  expert_ffn_static_kernel<<<items < 128 ? items : 128, kNaThreads, smem, st>>>(j);
  if (cudaGetLastError() != cudaSuccess) return MOE_ERR_CUDA;
  return MOE_OK;
}
