/*
 * Seeded synthetic inputs for the routed-MoE expert-slot cache.
 *
 * This module only draws random numbers and lays them out as inputs: the Q4_0
 * expert store (random nibbles, random fp16 scales), router logits built from a
 * Zipf-skewed, temporally sticky routing trace, and N(0,1) activations.  It
 * holds none of the method's arithmetic (no dequantisation, no softmax, no
 * top-k, no slot map, no FFN).  Both the CPU oracle and the CUDA path read the
 * inputs it writes; neither is imported here.
 *
 * Generators (published methods, written from their definitions):
 *   - SplitMix64 (Steele, Lea & Flood, "Fast splittable pseudorandom number
 *     generators", OOPSLA 2014): used to derive one independent seed per
 *     (seed, purpose, a, b) key.
 *   - PCG32 XSH-RR 64/32 (O'Neill, "PCG: A Family of Simple Fast
 *     Space-Efficient Statistically Good Algorithms for Random Number
 *     Generation", 2014): one stream per key.
 *   - Box-Muller transform for N(0,1).
 *   - Zipf(s) over ranks 1..E by inverse CDF on the normalised r^-s weights.
 *
 * Expert block layout written here (one contiguous block per (layer, expert)):
 *   [gate: F rows x H/32 blocks][up: F rows x H/32 blocks][down: H rows x F/32 blocks]
 * every block 18 bytes: fp16 scale d (little-endian) then 16 bytes of nibbles.
 * The scale is U(0.01, 0.05) rounded to nearest-even binary16; nibbles are
 * uniform on 0..15 (uniform random bytes).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ---- SplitMix64 ---------------------------------------------------------- */
static uint64_t sm64_next(uint64_t *s) {
    uint64_t z = (*s += 0x9E3779B97F4A7C15ULL);
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ULL;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBULL;
    return z ^ (z >> 31);
}

/* ---- PCG32 (XSH-RR, 64-bit state, 32-bit output) ------------------------- */
typedef struct { uint64_t state, inc; } pcg32_t;

static uint32_t pcg32_next(pcg32_t *r) {
    uint64_t old = r->state;
    r->state = old * 6364136223846793005ULL + r->inc;
    uint32_t xorshifted = (uint32_t)(((old >> 18u) ^ old) >> 27u);
    uint32_t rot = (uint32_t)(old >> 59u);
    return (xorshifted >> rot) | (xorshifted << ((32u - rot) & 31u));
}

static void pcg32_seed(pcg32_t *r, uint64_t initstate, uint64_t initseq) {
    r->state = 0u;
    r->inc = (initseq << 1u) | 1u;
    pcg32_next(r);
    r->state += initstate;
    pcg32_next(r);
}

/* One independent stream per key (seed, purpose, a, b). */
static pcg32_t stream_for(uint64_t seed, uint64_t purpose, uint64_t a, uint64_t b) {
    uint64_t s = seed;
    uint64_t h = sm64_next(&s);
    s = h ^ purpose;  h = sm64_next(&s);
    s = h ^ a;        h = sm64_next(&s);
    s = h ^ b;        h = sm64_next(&s);
    uint64_t seq = sm64_next(&s);
    pcg32_t r;
    pcg32_seed(&r, h, seq);
    return r;
}

/* Uniform double in [0,1) with 53 random bits. */
static double unif53(pcg32_t *r) {
    uint32_t a = pcg32_next(r) >> 5, b = pcg32_next(r) >> 6;
    return (a * 67108864.0 + b) * (1.0 / 9007199254740992.0);
}

/* Standard normal by Box-Muller (one value per call; u1 in (0,1]). */
static double normal01(pcg32_t *r) {
    double u1 = 1.0 - unif53(r);
    double u2 = unif53(r);
    return sqrt(-2.0 * log(u1)) * cos(6.283185307179586476925286766559 * u2);
}

/* Round a finite double to IEEE binary16, ties to even (normal and subnormal
 * range; values here are far from overflow). */
static uint16_t double_to_fp16_rne(double v) {
    uint16_t sign = 0;
    if (v < 0) { sign = 0x8000; v = -v; }
    if (v == 0.0) return sign;
    int e;
    double m = frexp(v, &e);          /* v = m * 2^e, m in [0.5, 1) */
    int exp16 = e - 1 + 15;           /* biased exponent for 1.f form */
    if (exp16 >= 1) {
        /* normal: 11 significant bits */
        double scaled = ldexp(m, 11);  /* in [1024, 2048) */
        double fl = floor(scaled);
        double rem = scaled - fl;
        uint32_t q = (uint32_t)fl;
        if (rem > 0.5 || (rem == 0.5 && (q & 1u))) q++;
        if (q == 2048u) { q = 1024u; exp16++; }
        if (exp16 >= 31) return (uint16_t)(sign | 0x7C00); /* overflow -> inf */
        return (uint16_t)(sign | (uint16_t)(exp16 << 10) | (uint16_t)(q - 1024u));
    }
    /* subnormal: units of 2^-24 */
    double scaled = ldexp(v, 24);
    double fl = floor(scaled);
    double rem = scaled - fl;
    uint32_t q = (uint32_t)fl;
    if (rem > 0.5 || (rem == 0.5 && (q & 1u))) q++;
    return (uint16_t)(sign | (uint16_t)q);  /* q == 1024 becomes the smallest normal */
}

/* Round fp32 to bfloat16, ties to even (finite inputs). */
static uint16_t float_to_bf16_rne(float f) {
    uint32_t u;
    memcpy(&u, &f, 4);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

enum {
    PURPOSE_WEIGHTS = 1,
    PURPOSE_PERM = 2,
    PURPOSE_TRACE = 3,
    PURPOSE_LOGITS = 4,
    PURPOSE_X = 5,
    PURPOSE_IID_LOGITS = 6,
};

/* Bytes of one expert block: 3 matrices of F*H values at 18 bytes per 32. */
uint64_t synth_expert_bytes(int H, int F) {
    return 3ull * (uint64_t)F * (uint64_t)H / 32ull * 18ull;
}

static void fill_matrix(pcg32_t *r, uint8_t *dst, int rows, int cols) {
    int nb = cols / 32;
    for (int i = 0; i < rows; ++i) {
        for (int b = 0; b < nb; ++b) {
            uint8_t *blk = dst + ((uint64_t)i * nb + b) * 18u;
            uint16_t d = double_to_fp16_rne(0.01 + 0.04 * unif53(r));
            blk[0] = (uint8_t)(d & 0xFF);
            blk[1] = (uint8_t)(d >> 8);
            for (int w = 0; w < 4; ++w) {
                uint32_t v = pcg32_next(r);
                blk[2 + 4 * w + 0] = (uint8_t)(v);
                blk[2 + 4 * w + 1] = (uint8_t)(v >> 8);
                blk[2 + 4 * w + 2] = (uint8_t)(v >> 16);
                blk[2 + 4 * w + 3] = (uint8_t)(v >> 24);
            }
        }
    }
}

/* Write one (layer, expert) block. */
void synth_fill_expert(uint8_t *dst, int layer, int expert, int H, int F, uint64_t seed) {
    pcg32_t r = stream_for(seed, PURPOSE_WEIGHTS, (uint64_t)layer, (uint64_t)expert);
    uint64_t mat = (uint64_t)F * H / 32u * 18u;
    fill_matrix(&r, dst, F, H);            /* gate */
    fill_matrix(&r, dst + mat, F, H);      /* up   */
    fill_matrix(&r, dst + 2 * mat, H, F);  /* down */
}

/* Whole store: dst[layer][expert] blocks, contiguous, expert stride = block bytes,
 * layer stride = E * block bytes.  Parallel over (layer, expert); the bytes do
 * not depend on the thread count. */
void synth_fill_store(uint8_t *dst, int L, int E, int H, int F, uint64_t seed, int n_threads) {
    uint64_t eb = synth_expert_bytes(H, F);
    long n = (long)L * E;
#ifdef _OPENMP
    if (n_threads > 0) omp_set_num_threads(n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (long i = 0; i < n; ++i) {
        int layer = (int)(i / E), expert = (int)(i % E);
        synth_fill_expert(dst + (uint64_t)i * eb, layer, expert, H, F, seed);
    }
    (void)n_threads;
}

/* Seeded random permutation of 0..E-1 (Fisher-Yates). */
void synth_permutation(int32_t *perm, int E, uint64_t seed, int layer) {
    pcg32_t r = stream_for(seed, PURPOSE_PERM, (uint64_t)layer, 0);
    for (int i = 0; i < E; ++i) perm[i] = i;
    for (int i = E - 1; i > 0; --i) {
        int j = (int)(unif53(&r) * (i + 1));
        int32_t t = perm[i]; perm[i] = perm[j]; perm[j] = t;
    }
}

/*
 * Routing trace for one (layer, stream): picks[t*k + i], t in [0, n_tok).
 * Rank r in 1..E is drawn with probability proportional to r^-s (s = 0 gives
 * uniform) and mapped to an expert by a per-layer random permutation.  For
 * t > 0 each pick is, with probability p_sticky, copied from a pick of token
 * t-1 that this token has not used yet (chosen uniformly among those);
 * otherwise it is drawn from the Zipf law, rejecting experts already picked.
 * `stream` separates independent sequences (e.g. batch-8 decode streams or
 * prefill batches).
 */
void synth_trace(int32_t *picks, int n_tok, int E, int k, double zipf_s, double p_sticky,
                 uint64_t seed, int layer, int stream) {
    int32_t *perm = (int32_t *)malloc(sizeof(int32_t) * E);
    double *cdf = (double *)malloc(sizeof(double) * E);
    synth_permutation(perm, E, seed, layer);
    double acc = 0.0;
    for (int r = 0; r < E; ++r) { acc += pow((double)(r + 1), -zipf_s); cdf[r] = acc; }
    for (int r = 0; r < E; ++r) cdf[r] /= acc;
    pcg32_t g = stream_for(seed, PURPOSE_TRACE, (uint64_t)layer, (uint64_t)stream);
    for (int t = 0; t < n_tok; ++t) {
        int32_t *cur = picks + (long)t * k;
        const int32_t *prev = t > 0 ? picks + (long)(t - 1) * k : NULL;
        for (int i = 0; i < k; ++i) {
            int chosen = -1;
            double u = unif53(&g);
            if (prev && u < p_sticky) {
                int cand[1024], nc = 0;
                for (int j = 0; j < k; ++j) {
                    int used = 0;
                    for (int q = 0; q < i; ++q) used |= (cur[q] == prev[j]);
                    if (!used && nc < 1024) cand[nc++] = prev[j];
                }
                if (nc > 0) chosen = cand[(int)(unif53(&g) * nc)];
            }
            while (chosen < 0) {
                double v = unif53(&g);
                int lo = 0, hi = E - 1;
                while (lo < hi) { int mid = (lo + hi) / 2; if (cdf[mid] > v) hi = mid; else lo = mid + 1; }
                int e = perm[lo];
                int used = 0;
                for (int q = 0; q < i; ++q) used |= (cur[q] == e);
                if (!used) chosen = e;
            }
            cur[i] = chosen;
        }
    }
    free(perm);
    free(cdf);
}

/*
 * Router logits whose top-k is exactly the picked set of each token: picked
 * experts get 3 + 2*U(0,1) (redrawn on an exact tie with another picked value),
 * the others N(0,1) redrawn until below 2.5.  `key` separates call sites
 * (e.g. step index); `layer` and `stream` as in synth_trace.
 */
void synth_logits_from_picks(float *logits, const int32_t *picks, int n_tok, int E, int k,
                             uint64_t seed, int layer, int stream, uint64_t key) {
    pcg32_t g = stream_for(seed, PURPOSE_LOGITS, ((uint64_t)layer << 32) | (uint32_t)stream, key);
    for (int t = 0; t < n_tok; ++t) {
        float *row = logits + (long)t * E;
        for (int e = 0; e < E; ++e) {
            float v;
            do { v = (float)normal01(&g); } while (!(v < 2.5f));
            row[e] = v;
        }
        for (int i = 0; i < k; ++i) {
            int e = picks[(long)t * k + i];
            for (;;) {
                float v = (float)(3.0 + 2.0 * unif53(&g));
                int tie = 0;
                for (int q = 0; q < i; ++q) tie |= (row[picks[(long)t * k + q]] == v);
                if (!tie) { row[e] = v; break; }
            }
        }
    }
}

/* i.i.d. N(0,1) fp32 values. */
void synth_normal_f32(float *out, uint64_t n, uint64_t seed, uint64_t purpose, uint64_t a, uint64_t b) {
    pcg32_t g = stream_for(seed, purpose, a, b);
    for (uint64_t i = 0; i < n; ++i) out[i] = (float)normal01(&g);
}

/* i.i.d. N(0,1) drawn in fp32 then rounded to bf16 (returned as raw bits). */
void synth_normal_bf16(uint16_t *out, uint64_t n, uint64_t seed, uint64_t purpose, uint64_t a, uint64_t b) {
    pcg32_t g = stream_for(seed, purpose, a, b);
    for (uint64_t i = 0; i < n; ++i) out[i] = float_to_bf16_rne((float)normal01(&g));
}

/* Raw PCG32 output of one keyed stream (used by tests to pin the generator). */
void synth_pcg32_raw(uint32_t *out, int n, uint64_t initstate, uint64_t initseq) {
    pcg32_t r;
    pcg32_seed(&r, initstate, initseq);
    for (int i = 0; i < n; ++i) out[i] = pcg32_next(&r);
}

void synth_splitmix64_raw(uint64_t *out, int n, uint64_t seed) {
    uint64_t s = seed;
    for (int i = 0; i < n; ++i) out[i] = sm64_next(&s);
}

uint16_t synth_fp16_rne(double v) { return double_to_fp16_rne(v); }
uint16_t synth_bf16_rne(float v) { return float_to_bf16_rne(v); }
