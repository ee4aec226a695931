// Expert FFN kernels of the GEMV (decode / small-batch) path and the slot fill.
//
//  * fill_kernel: missed canonical Q4_0 expert blocks (from the staging area or
//    straight from the mapped host store) -> repacked slot planes.  A bounded
//    grid loops over (miss, 32-row tile) pairs with cp.async double buffering,
//    so many host reads are in flight while SMs stay free for the hit compute.
//  * q4_tile_gemv_kernel<2>: gate and up rows (one 32-row tile) of one expert
//    for up to 8 of its tokens, then h = silu(g) * u ("llama.cpp + MoE expert
//    cache", "Limitations": merged gate/up, SiLU).
//  * q4_tile_gemv_kernel<1>: down rows, y = W_down h per pair (staged calls).
//  * down_combine_kernel: down rows of all k picks of one token and the
//    weighted sum over picks in ascending order ("The idea: cache the hot
//    experts on the GPU", step 4), for single-stage calls.
//  * combine_kernel: the weighted sum from stored y (staged calls).
//
// Weight tiles reach shared memory by bulk copies (cp.async.bulk, completion on
// an mbarrier): a 32-row tile of one matrix is two contiguous regions in the
// slot.  Compute reads them back lane-per-row (conflict-free 16-byte loads).
//
// Budget invariance: every output of a pair is reduced in one canonical order
// whatever kernel, slot, stage or work unit computes it: warp w of 8 sums the
// 32-blocks b = w, w+8, w+16, ... in ascending order, the 8 partial sums are
// added in warp order, and the weighted sum runs over picks in ascending order.
#include "q4_math.cuh"

namespace moe {
namespace {

using namespace q4;
constexpr int kFillCtas = 48;

__device__ __forceinline__ bool unit_range(const PlanHdr *h, const int32_t *ub, int kind, int stage,
                                           int &lo, int &hi) {
  if (h->error || stage >= h->n_stages) return false;
  if (kind == 0) { lo = 0; hi = h->hit_units; }
  else if (kind == 1) { lo = stage == 0 ? h->hit_units : ub[stage]; hi = ub[stage + 1]; }
  else { lo = ub[stage]; hi = ub[stage + 1]; }
  return true;
}

// ------------------------------------------------------ tile GEMV (units)
struct TileJob {
  const uint8_t *slots;
  uint64_t slot_stride;
  MatLayout m0, m1;  // m1 used when two matrices share the input (gate, up)
  int R, nb;         // rows and 32-blocks per row
  const void *x;     // input rows of K = 32 nb values
  int x_bf16;
  int x_div;         // input row of pair p is p / x_div
  const int32_t *perm;
  const WorkItem *items;
  const WorkUnit *units;
  const int32_t *unit_begin;
  const PlanHdr *hdr;
  int range_kind, stage;
  float *out;        // out[pair * R + r]
  int G;             // tokens per shared-memory group of inputs (<= kTokPerUnit)
  int32_t *err;
};

size_t tile_smem(int NMAT, int nb, int G) {
  return 128 + (size_t)NMAT * nb * (512 + 64) + sizeof(float) * ((size_t)G * 32 * nb + (size_t)G * nb +
                                                                  (size_t)kWarps * NMAT * G * 32);
}

template <int NMAT>
__global__ void __launch_bounds__(kThreads) q4_tile_gemv_kernel(TileJob j) {
  int lo, hi;
  if (!unit_range(j.hdr, j.unit_begin, j.range_kind, j.stage, lo, hi)) return;
  const int u = lo + (int)blockIdx.y;
  if (u >= hi) return;
  const WorkUnit wu = j.units[u];
  const WorkItem it = j.items[wu.item];
  const int n = wu.pair_count, G = j.G, nb = j.nb, K = 32 * nb;
  const int tile = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm);
  unsigned char *p = sm + 128;
  uint4 *wn[2];
  unsigned short *ws[2];
#pragma unroll
  for (int m = 0; m < NMAT; ++m) {
    wn[m] = reinterpret_cast<uint4 *>(p);
    p += (size_t)nb * 512;
    ws[m] = reinterpret_cast<unsigned short *>(p);
    p += (size_t)nb * 64;
  }
  float *xs = reinterpret_cast<float *>(p);
  float *xsum = xs + (size_t)G * K;
  float *red = xsum + (size_t)G * nb;  // [warps][NMAT][G][32]
  __shared__ int rows[kTokPerUnit];

  if (tid == 0) {
    mbar_init(bar, 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0) {
    const uint8_t *slot = j.slots + (uint64_t)it.slot * j.slot_stride;
    const uint32_t bn = (uint32_t)nb * 512, bs = (uint32_t)nb * 64;
    mbar_expect_tx(bar, NMAT * (bn + bs));
    const MatLayout *mats[2] = {&j.m0, &j.m1};
#pragma unroll
    for (int m = 0; m < NMAT; ++m) {
      bulk_g2s(wn[m], slot + mats[m]->nib_off + (uint64_t)tile * bn, bn, bar);
      bulk_g2s(ws[m], slot + mats[m]->sc_off + (uint64_t)tile * bs, bs, bar);
    }
  }
  if (tid < n) rows[tid] = j.perm[wu.pair_begin + tid] / j.x_div;
  __syncthreads();

  for (int g0 = 0; g0 < n; g0 += G) {
    const int gn = min(G, n - g0);
    stage_rows(xs, xsum, j.x, j.x_bf16, rows + g0, gn, K);
    if (g0 == 0 && !mbar_wait(bar, 0)) {
      flag_error(j.err, 2);
      mbar_wait(bar, 0);
      return;
    }
    float acc0[kTokPerUnit], acc1[kTokPerUnit];
#pragma unroll
    for (int t = 0; t < kTokPerUnit; ++t) { acc0[t] = 0.f; acc1[t] = 0.f; }
#pragma unroll 1
    for (int b = warp; b < nb; b += kWarps) {
      float f0[32], f1[32];
      const float d0 = half_bits(ws[0][b * 32 + lane]);
      decode_block(wn[0][b * 32 + lane], f0);
      float d1 = 0.f;
      if (NMAT == 2) {
        d1 = half_bits(ws[1][b * 32 + lane]);
        decode_block(wn[1][b * 32 + lane], f1);
      }
#pragma unroll
      for (int t = 0; t < kTokPerUnit; ++t) {
        if (t < gn) {
          const float *xb = xs + (size_t)t * K + 32 * b;
          const float xsb = xsum[t * nb + b];
          acc0[t] = block_term(f0, d0, xb, xsb, acc0[t]);
          if (NMAT == 2) acc1[t] = block_term(f1, d1, xb, xsb, acc1[t]);
        }
      }
    }
#pragma unroll
    for (int t = 0; t < kTokPerUnit; ++t) {
      if (t < gn) {
        red[((warp * NMAT + 0) * G + t) * 32 + lane] = acc0[t];
        if (NMAT == 2) red[((warp * NMAT + 1) * G + t) * 32 + lane] = acc1[t];
      }
    }
    __syncthreads();
    for (int t = warp; t < gn; t += kWarps) {
      float g = 0.f, v = 0.f;
      for (int w = 0; w < kWarps; ++w) {
        g += red[((w * NMAT + 0) * G + t) * 32 + lane];
        if (NMAT == 2) v += red[((w * NMAT + 1) * G + t) * 32 + lane];
      }
      const int pair = j.perm[wu.pair_begin + g0 + t];
      const float o = (NMAT == 2) ? g / (1.f + expf(-g)) * v : g;
      j.out[(size_t)pair * j.R + tile * 32 + lane] = o;
    }
    __syncthreads();
  }
}

template <int NMAT>
cudaError_t launch_tile(TileJob j, int max_units, cudaStream_t st) {
  if (max_units <= 0) return cudaSuccess;
  if (j.R % 32) return cudaErrorInvalidValue;
  const size_t budget = 200 * 1024;
  int G = j.G;
  while (G > 1 && tile_smem(NMAT, j.nb, G) > budget) --G;
  j.G = G;
  const size_t smem = tile_smem(NMAT, j.nb, G);
  if (smem > budget) return cudaErrorInvalidValue;
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(q4_tile_gemv_kernel<NMAT>, smem, cur);
  if (e != cudaSuccess) return e;
  dim3 grid(j.R / 32, max_units);
  q4_tile_gemv_kernel<NMAT><<<grid, kThreads, smem, st>>>(j);
  return cudaGetLastError();
}

// ------------------------------------------------------ down + combine
struct DownCombineJob {
  const uint8_t *slots;
  uint64_t slot_stride;
  MatLayout down;
  int H, F, k;
  const float *h;  // [T*k, F]
  const float *w;  // [T*k]
  const int32_t *gpu_slot;
  const PlanHdr *hdr;
  float *out;      // [T, H]
  int NS;          // tile stages in shared memory
  int32_t *err;
};

size_t dc_smem(int nb, int k, int NS) {
  return 128 + (size_t)NS * nb * 576 + sizeof(float) * ((size_t)k * 32 * nb + (size_t)k * nb +
                                                         (size_t)k * kWarps * 32);
}

__global__ void __launch_bounds__(kThreads) down_combine_kernel(DownCombineJob j) {
  if (j.hdr->error) return;
  const int t = blockIdx.y, tile = blockIdx.x, k = j.k, nb = j.F / 32, F = j.F, NS = j.NS;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t bn = (uint32_t)nb * 512, bs = (uint32_t)nb * 64;

  extern __shared__ __align__(128) unsigned char sm[];
  uint64_t *bar = reinterpret_cast<uint64_t *>(sm);  // [NS] (NS <= 8)
  unsigned char *stages = sm + 128;
  float *xs = reinterpret_cast<float *>(stages + (size_t)NS * nb * 576);
  float *xsum = xs + (size_t)k * F;
  float *red = xsum + (size_t)k * nb;  // [k][warps][32]
  __shared__ int rows[kMaxTopK];

  auto issue = [&](int q) {
    const int s = q % NS;
    unsigned char *dst = stages + (size_t)s * nb * 576;
    const uint8_t *slot = j.slots + (uint64_t)j.gpu_slot[t * k + q] * j.slot_stride;
    mbar_expect_tx(&bar[s], bn + bs);
    bulk_g2s(dst, slot + j.down.nib_off + (uint64_t)tile * bn, bn, &bar[s]);
    bulk_g2s(dst + bn, slot + j.down.sc_off + (uint64_t)tile * bs, bs, &bar[s]);
  };
  if (tid == 0) {
    for (int s = 0; s < NS; ++s) mbar_init(&bar[s], 1);
    fence_mbar_init();
  }
  __syncthreads();
  if (tid == 0)
    for (int q = 0; q < NS && q < k; ++q) issue(q);
  if (tid < k) rows[tid] = t * k + tid;
  __syncthreads();
  stage_rows(xs, xsum, j.h, 0, rows, k, F);

  for (int q = 0; q < k; ++q) {
    const int s = q % NS;
    if (!mbar_wait(&bar[s], (uint32_t)(q / NS) & 1u)) {
      flag_error(j.err, 2);
      return;
    }
    const uint4 *wn = reinterpret_cast<const uint4 *>(stages + (size_t)s * nb * 576);
    const unsigned short *wsc = reinterpret_cast<const unsigned short *>(stages + (size_t)s * nb * 576 + bn);
    float acc = 0.f;
#pragma unroll 1
    for (int b = warp; b < nb; b += kWarps) {
      float f[32];
      decode_block(wn[b * 32 + lane], f);
      acc = block_term(f, half_bits(wsc[b * 32 + lane]), xs + (size_t)q * F + 32 * b,
                       xsum[q * nb + b], acc);
    }
    red[(q * kWarps + warp) * 32 + lane] = acc;
    __syncthreads();  // stage s is free again
    if (tid == 0 && q + NS < k) {
      fence_proxy_async();
      issue(q + NS);
    }
  }
  if (warp == 0) {
    float o = 0.f;
    for (int q = 0; q < k; ++q) {
      float y = 0.f;
      for (int w = 0; w < kWarps; ++w) y += red[(q * kWarps + w) * 32 + lane];
      o = fmaf(j.w[t * k + q], y, o);
    }
    j.out[(size_t)t * j.H + tile * 32 + lane] = o;
  }
}

// ---------------------------------------------------------------- fill
struct FillJob {
  RepackArgs a;
  int S;
  int nb_max;
};

__global__ void __launch_bounds__(kThreads) fill_kernel(FillJob jb) {
  const RepackArgs &a = jb.a;
  const PlanHdr *h = a.hdr;
  if (h->error || a.stage >= h->n_stages) return;
  // stage 0 holds n0 misses, every later stage stage_cap (<= S; the last may hold fewer)
  const int n0 = h->n_stage0_miss, nM = h->n_miss, C = h->stage_cap;
  int m_lo, m_hi;
  if (a.stage == 0) { m_lo = 0; m_hi = n0; }
  else {
    if (C < 1 || C > jb.S) return;
    m_lo = n0 + (a.stage - 1) * C;
    m_hi = min(nM, n0 + a.stage * C);
  }
  const int tg = a.lay.gate.rows / 32, td = a.lay.down.rows / 32;
  const int tiles = 2 * tg + td;
  const int n_work = (m_hi - m_lo) * tiles;
  const size_t buf_bytes = (size_t)32 * jb.nb_max * 18;
  extern __shared__ __align__(128) unsigned char rs[];

  // work item -> (source tile, destination slot, matrix, tile index)
  auto locate = [&](int wk, const uint8_t *&src, uint8_t *&dst, const MatLayout *&L, int &tl) {
    const int mi = m_lo + wk / tiles;
    tl = wk % tiles;
    const MissItem m = a.miss[mi];
    const uint8_t *blk = a.by_expert
                             ? a.src_base + a.src_layer_off + (uint64_t)m.expert * a.src_expert_stride
                             : a.src_base + (uint64_t)(mi - m_lo) * a.src_slot_stride;
    dst = a.slots + (uint64_t)m.slot * a.slot_stride;
    if (tl < tg) L = &a.lay.gate;
    else if (tl < 2 * tg) { L = &a.lay.up; tl -= tg; }
    else { L = &a.lay.down; tl -= 2 * tg; }
    // the canonical matrix starts where its nibble plane starts (same byte count)
    src = blk + L->nib_off + (uint64_t)tl * 32 * L->nb * 18;
  };
  auto issue = [&](int wk, int buf) {
    const uint8_t *src;
    uint8_t *dst;
    const MatLayout *L;
    int tl;
    locate(wk, src, dst, L, tl);
    const int n16 = 36 * L->nb;  // 32 rows x nb blocks x 18 bytes / 16
    unsigned char *b = rs + (size_t)buf * buf_bytes;
    for (int i = threadIdx.x; i < n16; i += kThreads) cp_async16(b + 16 * i, src + 16 * i);
  };

  int wk = blockIdx.x;
  if (wk < n_work) issue(wk, 0);
  cp_async_commit();
  for (int it = 0; wk < n_work; ++it, wk += gridDim.x) {
    const int nxt = wk + gridDim.x;
    if (nxt < n_work) issue(nxt, (it + 1) & 1);
    cp_async_commit();
    cp_async_wait1();
    __syncthreads();
    const uint8_t *src;
    uint8_t *dst;
    const MatLayout *L;
    int tl;
    locate(wk, src, dst, L, tl);
    const int nb = L->nb;
    const unsigned char *b0 = rs + (size_t)(it & 1) * buf_bytes;
    uint4 *nib = reinterpret_cast<uint4 *>(dst + L->nib_off);
    unsigned short *sc = reinterpret_cast<unsigned short *>(dst + L->sc_off);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    for (int b = warp; b < nb; b += kWarps) {
      const unsigned short *blk =
          reinterpret_cast<const unsigned short *>(b0 + ((size_t)lane * nb + b) * 18);
      uint32_t v[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) v[i] = (uint32_t)blk[1 + 2 * i] | ((uint32_t)blk[2 + 2 * i] << 16);
      const uint64_t e = tile_elem(tl * 32 + lane, b, nb);
      nib[e] = make_uint4(v[0], v[1], v[2], v[3]);
      sc[e] = blk[0];
    }
    __syncthreads();
  }
}

// ------------------------------------------------------ fused miss path
// For single-stage calls of at most 8 tokens: every missed expert is read once
// from its source (mapped host store or staging), written into its slot in the
// tiled layout, and used for compute on the way, so the misses' FFN hides
// under the transfer.  Work items come from a queue in order: all gate/up
// tiles (32 rows of gate and of up), then all down tiles; a down tile waits for
// the gate/up tiles of its expert (a per-miss counter; bounded wait).  Since
// items are claimed in order by running CTAs, the tiles a down tile waits for
// are already being processed.  The per-pair arithmetic and its order are
// those of q4_tile_gemv_kernel and down_combine_kernel.
struct FusedMissJob {
  const uint8_t *src_base;
  uint64_t src_layer_off, src_expert_stride, src_slot_stride;
  int by_expert;
  uint8_t *slots;
  uint64_t slot_stride;
  SlotLayout lay;
  const MissItem *miss;
  const PlanHdr *hdr;
  const WorkItem *items;
  const int32_t *perm;
  const void *x;
  int x_bf16;
  int k, H, F;
  float *h;        // [T*k, F]
  float *y;        // [T*k, H]
  int32_t *sync;   // [0] queue head, [1 + m] finished gate/up tiles of miss m
  int32_t *err;
  int G;           // tokens per shared-memory input group
};


size_t fused_smem(int nbH, int nbF, int G) {
  const size_t canon = (size_t)32 * 18 * (2 * nbH > nbF ? 2 * nbH : nbF);
  const int kmax = 32 * (nbH > nbF ? nbH : nbF), nbmax = nbH > nbF ? nbH : nbF;
  return canon + sizeof(float) * ((size_t)G * kmax + (size_t)G * nbmax + (size_t)kWarps * 2 * G * 32);
}


__global__ void __launch_bounds__(kThreads) fused_miss_kernel(FusedMissJob j) {
  const PlanHdr *hd = j.hdr;
  if (hd->error) return;
  const int nM = hd->n_stage0_miss, nH = hd->n_hits;
  const int nbH = j.H / 32, nbF = j.F / 32, tF = j.F / 32, tH = j.H / 32;
  const int n_a = nM * tF, n_total = n_a + nM * tH;
  if (n_total == 0) return;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, G = j.G;

  extern __shared__ __align__(128) unsigned char sm[];
  const size_t canon_bytes = (size_t)32 * 18 * (2 * nbH > nbF ? 2 * nbH : nbF);
  unsigned char *canon = sm;
  float *xs = reinterpret_cast<float *>(sm + canon_bytes);
  const int kmax = 32 * (nbH > nbF ? nbH : nbF), nbmax = nbH > nbF ? nbH : nbF;
  float *xsum = xs + (size_t)G * kmax;
  float *red = xsum + (size_t)G * nbmax;  // [warps][2][G][32]
  __shared__ int s_wk, s_ok;
  __shared__ int rows[kTokPerUnit];

  for (;;) {
    if (tid == 0) s_wk = atomicAdd(&j.sync[0], 1);
    __syncthreads();
    const int wk = s_wk;
    if (wk >= n_total) break;
    const bool is_gu = wk < n_a;
    const int m = is_gu ? wk / tF : (wk - n_a) / tH;
    const int t = is_gu ? wk % tF : (wk - n_a) % tH;
    const MissItem mi = j.miss[m];
    const WorkItem it = j.items[nH + m];
    const int n = it.pair_count;
    const uint8_t *blk = j.by_expert
                             ? j.src_base + j.src_layer_off + (uint64_t)mi.expert * j.src_expert_stride
                             : j.src_base + (uint64_t)m * j.src_slot_stride;
    uint8_t *dst = j.slots + (uint64_t)mi.slot * j.slot_stride;
    const int nb = is_gu ? nbH : nbF;
    const int nmat = is_gu ? 2 : 1;
    // canonical rows [32t, 32t+32) of each matrix of this item
    const MatLayout *L0 = is_gu ? &j.lay.gate : &j.lay.down;
    const MatLayout *L1 = &j.lay.up;
    const size_t tile_bytes = (size_t)32 * nb * 18;
    for (int mm = 0; mm < nmat; ++mm) {
      const MatLayout *L = mm == 0 ? L0 : L1;
      const uint8_t *src = blk + L->nib_off + (uint64_t)t * tile_bytes;
      for (int i = tid; i < (int)(tile_bytes / 16); i += kThreads)
        cp_async16(canon + mm * tile_bytes + 16 * i, src + 16 * i);
    }
    cp_async_commit();
    if (!is_gu) {
      // the tile is on its way; h of this expert needs all its gate/up tiles
      if (tid == 0) {
        int ok = 0;
        for (uint32_t i = 0; i < kSpinLimit; ++i) {
          if (ld_acquire(&j.sync[1 + m]) >= tF) { ok = 1; break; }
          __nanosleep(64);
        }
        s_ok = ok;
      }
      __syncthreads();
      if (!s_ok) {
        flag_error(j.err, 3);
        asm volatile("cp.async.wait_all;" ::: "memory");
        return;
      }
    }
    if (tid < n) rows[tid] = is_gu ? j.perm[it.pair_begin + tid] / j.k : j.perm[it.pair_begin + tid];
    __syncthreads();
    const int K = 32 * nb;
    for (int g0 = 0; g0 < n; g0 += G) {
      const int gn = min(G, n - g0);
      if (is_gu) stage_rows(xs, xsum, j.x, j.x_bf16, rows + g0, gn, K);
      else stage_rows(xs, xsum, j.h, 0, rows + g0, gn, K, true);
      if (g0 == 0) {
        asm volatile("cp.async.wait_all;" ::: "memory");
        __syncthreads();
      }
      float acc0[kTokPerUnit], acc1[kTokPerUnit];
#pragma unroll
      for (int q = 0; q < kTokPerUnit; ++q) { acc0[q] = 0.f; acc1[q] = 0.f; }
#pragma unroll 1
      for (int b = warp; b < nb; b += kWarps) {
        float f0[32], f1[32];
        unsigned short d0b, d1b = 0;
        const uint4 q0 = canon_block(canon, lane, b, nb, d0b);
        decode_block(q0, f0);
        uint4 q1 = make_uint4(0, 0, 0, 0);
        if (is_gu) {
          q1 = canon_block(canon + tile_bytes, lane, b, nb, d1b);
          decode_block(q1, f1);
        }
        if (g0 == 0) {
          const uint64_t e = tile_elem(t * 32 + lane, b, nb);
          reinterpret_cast<uint4 *>(dst + L0->nib_off)[e] = q0;
          reinterpret_cast<unsigned short *>(dst + L0->sc_off)[e] = d0b;
          if (is_gu) {
            reinterpret_cast<uint4 *>(dst + L1->nib_off)[e] = q1;
            reinterpret_cast<unsigned short *>(dst + L1->sc_off)[e] = d1b;
          }
        }
        const float d0 = half_bits(d0b), d1 = half_bits(d1b);
#pragma unroll
        for (int q = 0; q < kTokPerUnit; ++q) {
          if (q < gn) {
            const float *xb = xs + (size_t)q * K + 32 * b;
            const float xsb = xsum[q * nb + b];
            acc0[q] = block_term(f0, d0, xb, xsb, acc0[q]);
            if (is_gu) acc1[q] = block_term(f1, d1, xb, xsb, acc1[q]);
          }
        }
      }
#pragma unroll
      for (int q = 0; q < kTokPerUnit; ++q) {
        if (q < gn) {
          red[((warp * 2 + 0) * G + q) * 32 + lane] = acc0[q];
          red[((warp * 2 + 1) * G + q) * 32 + lane] = acc1[q];
        }
      }
      __syncthreads();
      for (int q = warp; q < gn; q += kWarps) {
        float g = 0.f, v = 0.f;
        for (int w = 0; w < kWarps; ++w) {
          g += red[((w * 2 + 0) * G + q) * 32 + lane];
          if (is_gu) v += red[((w * 2 + 1) * G + q) * 32 + lane];
        }
        const int pair = j.perm[it.pair_begin + g0 + q];
        if (is_gu) j.h[(size_t)pair * j.F + t * 32 + lane] = g / (1.f + expf(-g)) * v;
        else j.y[(size_t)pair * j.H + t * 32 + lane] = g;
      }
      __syncthreads();
    }
    if (is_gu && tid == 0) {
      __threadfence();
      atomicAdd(&j.sync[1 + m], 1);
    }
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

TileJob base_job(const FfnArgs &a) {
  TileJob j;
  j.slots = a.slots;
  j.slot_stride = a.slot_stride;
  j.perm = a.perm;
  j.items = a.items;
  j.units = a.units;
  j.unit_begin = a.unit_begin;
  j.hdr = a.hdr;
  j.G = a.max_tok;
  j.err = a.err;
  return j;
}

}  // namespace

cudaError_t launch_gateup(const FfnArgs &a, int range_kind, int stage, int max_units,
                          cudaStream_t st) {
  TileJob j = base_job(a);
  j.m0 = a.lay.gate;
  j.m1 = a.lay.up;
  j.R = a.F;
  j.nb = a.H / 32;
  j.x = a.x;
  j.x_bf16 = a.x_bf16;
  j.x_div = a.k;
  j.range_kind = range_kind;
  j.stage = stage;
  j.out = a.h;
  return launch_tile<2>(j, max_units, st);
}

cudaError_t launch_down(const FfnArgs &a, int range_kind, int stage, int max_units,
                        cudaStream_t st) {
  TileJob j = base_job(a);
  j.m0 = a.lay.down;
  j.m1 = a.lay.down;
  j.R = a.H;
  j.nb = a.F / 32;
  j.x = a.h;
  j.x_bf16 = 0;
  j.x_div = 1;
  j.range_kind = range_kind;
  j.stage = stage;
  j.out = a.y;
  return launch_tile<1>(j, max_units, st);
}

static int dc_stages(int F, int k) {
  const int nb = F / 32;
  int NS = k < 8 ? k : 8;
  while (NS > 1 && dc_smem(nb, k, NS) > 200 * 1024) --NS;
  return NS;
}

bool down_combine_supported(int F, int k) {
  return dc_smem(F / 32, k, dc_stages(F, k)) <= 200 * 1024;
}

cudaError_t launch_down_combine(const FfnArgs &a, const float *w, const int32_t *gpu_slot, int T,
                                float *out, cudaStream_t st) {
  DownCombineJob j;
  j.slots = a.slots;
  j.slot_stride = a.slot_stride;
  j.down = a.lay.down;
  j.H = a.H;
  j.F = a.F;
  j.k = a.k;
  j.h = a.h;
  j.w = w;
  j.gpu_slot = gpu_slot;
  j.hdr = a.hdr;
  j.out = out;
  j.NS = dc_stages(a.F, a.k);
  j.err = a.err;
  const size_t smem = dc_smem(a.F / 32, a.k, j.NS);
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(down_combine_kernel, smem, cur);
  if (e != cudaSuccess) return e;
  dim3 grid(a.H / 32, T);
  down_combine_kernel<<<grid, kThreads, smem, st>>>(j);
  return cudaGetLastError();
}

cudaError_t launch_combine(const float *y, const float *w, const PlanHdr *hdr, int T, int k, int H,
                           float *out, cudaStream_t st) {
  const size_t n = (size_t)T * H;
  combine_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(y, w, hdr, T, k, H, out);
  return cudaGetLastError();
}

cudaError_t launch_fused_miss(const FfnArgs &a, const RepackArgs &r, int32_t *sync, int grid,
                              cudaStream_t st) {
  FusedMissJob j;
  j.src_base = r.src_base;
  j.src_layer_off = r.src_layer_off;
  j.src_expert_stride = r.src_expert_stride;
  j.src_slot_stride = r.src_slot_stride;
  j.by_expert = r.by_expert;
  j.slots = r.slots;
  j.slot_stride = r.slot_stride;
  j.lay = r.lay;
  j.miss = r.miss;
  j.hdr = r.hdr;
  j.items = a.items;
  j.perm = a.perm;
  j.x = a.x;
  j.x_bf16 = a.x_bf16;
  j.k = a.k;
  j.H = a.H;
  j.F = a.F;
  j.h = a.h;
  j.y = a.y;
  j.sync = sync;
  j.err = a.err;
  int G = a.max_tok;
  while (G > 1 && fused_smem(a.H / 32, a.F / 32, G) > 200 * 1024) --G;
  j.G = G;
  const size_t smem = fused_smem(a.H / 32, a.F / 32, G);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(fused_miss_kernel, smem, cur);
  if (e != cudaSuccess) return e;
  fused_miss_kernel<<<grid, kThreads, smem, st>>>(j);
  return cudaGetLastError();
}

bool fused_miss_supported(int H, int F) { return fused_smem(H / 32, F / 32, 1) <= 200 * 1024; }

cudaError_t launch_repack(const RepackArgs &a, int S, int max_miss, cudaStream_t st) {
  if (max_miss <= 0) return cudaSuccess;
  FillJob jb{a, S, a.lay.gate.nb > a.lay.down.nb ? a.lay.gate.nb : a.lay.down.nb};
  const size_t smem = 2 * (size_t)32 * jb.nb_max * 18;
  static DynSmemLimit cur;
  const cudaError_t e = ensure_dyn_smem(fill_kernel, smem, cur);
  if (e != cudaSuccess) return e;
  const int tiles = 2 * a.lay.gate.rows / 32 + a.lay.down.rows / 32;
  const int grid = tiles * max_miss < kFillCtas ? tiles * max_miss : kFillCtas;
  fill_kernel<<<grid, kThreads, smem, st>>>(jb);
  return cudaGetLastError();
}

}  // namespace moe
