/*
 * CPU ORACLE for the routed-MoE layer over a GPU-resident expert-slot cache.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the bench's
 * CPU-baseline / reference legs may load this library.  The product path (the
 * CUDA library and its Python binding) never calls it, and it shares no code,
 * header, table or helper with that path.
 *
 * Plain, slow and written to be checked by eye: every floating-point step is in
 * double, loops are in the order the method states them, no blocking, fusion or
 * reordering.  What each function follows (page title, section):
 *
 *  - Q4_0 block: "Multi-GPU LLM Calculator: VRAM Split and RAM Offload",
 *    section "Memory placement": Q4_0 packs 32 values in 18 bytes (the GGML
 *    block definition).  Layout read as: fp16 scale d (little-endian), then 16
 *    bytes; byte j holds value j in its low nibble and value j+16 in its high
 *    nibble; w = (q - 8) * d.
 *  - Router: the router picks the top-k experts of each token ("llama.cpp +
 *    MoE expert cache", "The idea: cache the hot experts on the GPU", step 1);
 *    weights are the softmax probabilities of the chosen experts (or, in
 *    weight mode 1, renormalised over the chosen k).
 *  - Slot table, -1 = not cached: same section, step 2.
 *  - LRU per layer with a fixed budget: "Longhaul MoE loading" (docs/longhaul.md),
 *    opening paragraph.  Batch planning, protection of the batch's experts from
 *    eviction, duplicates loaded once: same page, the paragraph on expert IDs
 *    planned as a batch at each synchronisation point.  More experts than slots:
 *    split into stages whose partial results are summed (same page, the
 *    paragraph on --ubatch-size and stages).
 *  - Expert FFN with merged gate/up and SiLU: "llama.cpp + MoE expert cache",
 *    "Limitations" (merged gate/up expert tensors, SiLU activation): SwiGLU
 *    h = silu(W_gate x) * (W_up x), y = W_down h.
 *  - Combine: "The idea: cache the hot experts on the GPU", step 4: partial
 *    results added, expert weights applied (weighted sum), here in ascending
 *    pick order.
 *  - Replacement policies beside LRU: the decayed usage score with admission
 *    ("llama.cpp + MoE expert cache", "Keeping the cache fresh") and its sticky
 *    share; adopt, a staged call ending with its most-used experts ("llama.cpp:
 *    fork with multi gpu acceleration ...", "Prefill preheat"); warm start from
 *    usage counts (same page, "Persistent hot experts"), the lifetime activation
 *    counts such a profile holds, and resuming a saved slot-table state.
 *
 * Parity pins live in tests/test_oracle_*.py (hand-worked Q4_0 blocks, exact
 * integer GEMV cases, brute-force router, independent brute-force simulators of
 * LRU, the score policy and adopt, hand-worked warm starts, exactly-once and
 * budget-invariance checks).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* ------------------------------------------------------------ number formats */

/* IEEE 754 binary16 -> double, exactly: 1 sign bit, 5 exponent bits (bias 15),
 * 10 fraction bits; exponent 0 encodes subnormals (fraction * 2^-24), 31
 * encodes infinities and NaNs. */
double orc_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int expo = (h >> 10) & 0x1F;
    int frac = h & 0x3FF;
    double v;
    if (expo == 0) {
        v = ldexp((double)frac, -24);
    } else if (expo == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + frac), expo - 25);
    }
    return sign ? -v : v;
}

/* bfloat16 -> double, exactly: bfloat16 is the top half of an fp32. */
double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* ------------------------------------------------------------------- Q4_0 */

/* Decode one 18-byte Q4_0 block into 32 doubles. */
void orc_q4_0_decode(const uint8_t *blk, double out[32]) {
    double d = orc_fp16_to_double((uint16_t)(blk[0] | (blk[1] << 8)));
    for (int j = 0; j < 16; ++j) {
        int lo = blk[2 + j] & 0x0F;
        int hi = blk[2 + j] >> 4;
        out[j] = (double)(lo - 8) * d;
        out[j + 16] = (double)(hi - 8) * d;
    }
}

/* Dot product of one quantised row (nb consecutive blocks) with v[32*nb]. */
static double row_dot(const uint8_t *row, int nb, const double *v) {
    double acc = 0.0, w[32];
    for (int b = 0; b < nb; ++b) {
        orc_q4_0_decode(row + (size_t)b * 18, w);
        for (int j = 0; j < 32; ++j) acc += w[j] * v[32 * b + j];
    }
    return acc;
}

/* ----------------------------------------------------------------- router */

/*
 * Router for T tokens over E logits each (row-major [T][E]).
 * Selection: the k largest raw logits, in descending order, ties to the lower
 * expert id.  Probabilities: softmax over all E in double with max subtraction.
 * weight_mode 0: w = p of the chosen expert; weight_mode 1: p renormalised over
 * the chosen k.  Returns -1 (and writes nothing useful) if a logit is not
 * finite.
 */
int orc_router(const float *logits, int T, int E, int k, int weight_mode,
               int32_t *ids, double *w) {
    for (long i = 0; i < (long)T * E; ++i)
        if (!isfinite(logits[i])) return -1;
    unsigned char *taken = (unsigned char *)malloc((size_t)E);
    for (int t = 0; t < T; ++t) {
        const float *row = logits + (long)t * E;
        memset(taken, 0, (size_t)E);
        for (int i = 0; i < k; ++i) {
            int best = -1;
            for (int e = 0; e < E; ++e) {
                if (taken[e]) continue;
                if (best < 0 || row[e] > row[best]) best = e;  /* strict: lower id wins ties */
            }
            taken[best] = 1;
            ids[(long)t * k + i] = best;
        }
        double m = row[0];
        for (int e = 1; e < E; ++e) if (row[e] > m) m = row[e];
        double z = 0.0;
        for (int e = 0; e < E; ++e) z += exp((double)row[e] - m);
        double sel = 0.0;
        for (int i = 0; i < k; ++i) {
            double p = exp((double)row[ids[(long)t * k + i]] - m) / z;
            w[(long)t * k + i] = p;
            sel += p;
        }
        if (weight_mode == 1)
            for (int i = 0; i < k; ++i) w[(long)t * k + i] /= sel;
    }
    free(taken);
    return 0;
}

/* ------------------------------------------------------------ LRU slot map */

typedef struct {
    int S, E;
    int32_t *slot_expert;  /* [S]  expert held by each slot, -1 = empty        */
    int32_t *expert_slot;  /* [E]  slot of each expert, -1 = not cached        */
    uint64_t *slot_stamp;  /* [S]  call counter of the slot's last use         */
    uint64_t clock;        /* number of calls planned so far                   */
    int policy;            /* 0: LRU; 1: decayed usage score with admission;
                              2: LRU, staged calls keep their most-used experts */
    int budget;            /* policy 1: admissions per call, 0 = unlimited     */
    float *score;          /* [E]  policy 1: decayed usage per expert (fp32)   */
    int sticky;            /* policy 1: per mille of the slots, highest scores
                              first, that a call may not evict                */
} orc_lru;

orc_lru *orc_lru_new(int S, int E) {
    orc_lru *st = (orc_lru *)calloc(1, sizeof(orc_lru));
    st->S = S;
    st->E = E;
    st->slot_expert = (int32_t *)malloc(sizeof(int32_t) * S);
    st->expert_slot = (int32_t *)malloc(sizeof(int32_t) * E);
    st->slot_stamp = (uint64_t *)calloc((size_t)S, sizeof(uint64_t));
    for (int s = 0; s < S; ++s) st->slot_expert[s] = -1;
    for (int e = 0; e < E; ++e) st->expert_slot[e] = -1;
    st->clock = 0;
    st->policy = 0;
    st->budget = 0;
    st->score = (float *)calloc((size_t)E, sizeof(float));
    return st;
}

/* Replacement policy of the state: 0 = LRU (default), 1 = decayed score,
 * 2 = LRU with adopt (staged calls end holding their most-used experts). */
void orc_lru_set_policy(orc_lru *st, int policy, int budget) {
    st->policy = policy;
    st->budget = budget;
}

/* Sticky share of policy 1, per mille of the slots (0 = none). */
void orc_lru_set_sticky(orc_lru *st, int permille) { st->sticky = permille; }

/* Copy of the decayed scores [E] (policy 1, fp32). */
void orc_lru_scores(const orc_lru *st, float *out) { memcpy(out, st->score, sizeof(float) * st->E); }

void orc_lru_free(orc_lru *st) {
    if (!st) return;
    free(st->slot_expert);
    free(st->expert_slot);
    free(st->slot_stamp);
    free(st->score);
    free(st);
}

/* Copy of the state for inspection: slot_expert[S], expert_slot[E], slot_stamp[S], clock. */
void orc_lru_get(const orc_lru *st, int32_t *slot_expert, int32_t *expert_slot,
                 uint64_t *slot_stamp, uint64_t *clock) {
    memcpy(slot_expert, st->slot_expert, sizeof(int32_t) * st->S);
    memcpy(expert_slot, st->expert_slot, sizeof(int32_t) * st->E);
    memcpy(slot_stamp, st->slot_stamp, sizeof(uint64_t) * st->S);
    *clock = st->clock;
}

/* Per-call plan summary. */
typedef struct {
    int32_t n_unique, n_hits, n_miss, n_stages, n_evict;
    int32_t pick_hits, pick_misses;
    int32_t n_bypass;      /* policy 1: misses computed without taking a slot */
} orc_plan_info;

/* Order two candidate slots for eviction: empty slots first (by slot index),
 * then occupied slots by (stamp, slot index). */
static int victim_before(const orc_lru *st, int a, int b) {
    int ea = st->slot_expert[a] < 0, eb = st->slot_expert[b] < 0;
    if (ea != eb) return ea;               /* empty before occupied */
    if (ea) return a < b;
    if (st->slot_stamp[a] != st->slot_stamp[b]) return st->slot_stamp[a] < st->slot_stamp[b];
    return a < b;
}

static void sort_victims(const orc_lru *st, int *v, int n) {
    for (int i = 1; i < n; ++i) {          /* insertion sort */
        int x = v[i], j = i - 1;
        while (j >= 0 && victim_before(st, x, v[j])) { v[j + 1] = v[j]; --j; }
        v[j + 1] = x;
    }
}

/*
 * Policy 1: decayed usage score with admission ("Keeping the cache fresh": a
 * usage score per expert decayed by 0.9 per token; a missed expert that scores
 * higher than the weakest slot is promoted, up to a budget of copies).  Every
 * miss is still computed (from the host store); only admitted ones take a slot.
 *   clock += 1.  Token by token: every score *= 0.9, then each picked expert's
 *   score += 1, in fp32 (each operation rounded).  The page gives the factor and
 *   no precision; single precision is the reading taken, pinned by a trace on
 *   which it decides an admission (a tie at exactly 1.0 that double precision
 *   would not have).  U, hits and misses as for LRU; the call must fit one stage
 *   (|U| <= S), else -2.  Hits keep their slots (stamped).  Misses in order of
 *   (score descending, id ascending); each, while the budget lasts (0 =
 *   unlimited), takes the next empty slot (ascending index) if any, else the
 *   weakest slot whose expert the call does not pick, by (score ascending,
 *   index ascending), if its own score is strictly higher; otherwise it is
 *   bypassed (slot -1, nothing evicted).  Every admission counts against the
 *   budget.  Miss list in ascending expert order, all in stage 0.
 *   Sticky share (Fork A's option to never evict the most-used share of each
 *   layer's slots): once the call's scores are updated, the
 *   floor(sticky x S / 1000) occupied slots with the highest scores (ties to
 *   the lower index) are not evictable in this call.
 */
static int slot_map_score(orc_lru *st, const int32_t *ids, int T, int k, int32_t *gpu_slot, int32_t *stage,
                          int32_t *miss_expert, int32_t *miss_slot, int32_t *miss_evicted, int32_t *miss_stage,
                          orc_plan_info *info) {
    const int S = st->S, E = st->E;
    memset(info, 0, sizeof(*info));
    unsigned char *used = (unsigned char *)calloc((size_t)E, 1);
    int32_t *cnt = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (long p = 0; p < (long)T * k; ++p) { used[ids[p]] = 1; cnt[ids[p]] += 1; }
    int nU = 0;
    for (int e = 0; e < E; ++e) nU += used[e];
    if (nU > S) { free(used); free(cnt); return -2; }
    st->clock += 1;
    const uint64_t now = st->clock;
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) st->score[e] = st->score[e] * 0.9f;
        for (int q = 0; q < k; ++q) st->score[ids[(long)t * k + q]] = st->score[ids[(long)t * k + q]] + 1.0f;
    }
    int32_t *M = (int32_t *)malloc(sizeof(int32_t) * E), nM = 0;
    int32_t *e_slot = (int32_t *)malloc(sizeof(int32_t) * E);
    int32_t *d_old = (int32_t *)malloc(sizeof(int32_t) * E);
    unsigned char *was_hit = (unsigned char *)calloc((size_t)E, 1);
    int nH = 0;
    for (int e = 0; e < E; ++e) {
        e_slot[e] = -1;
        d_old[e] = -1;
        if (!used[e]) continue;
        if (st->expert_slot[e] >= 0) {
            was_hit[e] = 1;
            ++nH;
            e_slot[e] = st->expert_slot[e];
            st->slot_stamp[e_slot[e]] = now;
        } else {
            M[nM++] = e;
        }
    }
    info->n_unique = nU;
    info->n_hits = nH;
    info->n_miss = nM;
    info->n_stages = 1;
    for (long p = 0; p < (long)T * k; ++p) {
        if (was_hit[ids[p]]) info->pick_hits++;
        else info->pick_misses++;
    }
    /* sticky: the n_sticky occupied slots of highest score are kept */
    const int n_sticky = (int)((int64_t)st->sticky * S / 1000);
    unsigned char *keep = (unsigned char *)calloc((size_t)S, 1);
    for (int s = 0; s < S; ++s) {
        const int e = st->slot_expert[s];
        if (e < 0) continue;
        int above = 0;
        for (int s2 = 0; s2 < S; ++s2) {
            const int e2 = st->slot_expert[s2];
            if (e2 >= 0 && (st->score[e2] > st->score[e] || (st->score[e2] == st->score[e] && s2 < s))) ++above;
        }
        keep[s] = above < n_sticky;
    }
    /* empty slots ascending; slots of experts not picked and not kept, by (score, index) */
    int *fr = (int *)malloc(sizeof(int) * S), nf = 0;
    int *ev = (int *)malloc(sizeof(int) * S), nv = 0;
    for (int s = 0; s < S; ++s) {
        const int e = st->slot_expert[s];
        if (e < 0) fr[nf++] = s;
        else if (!used[e] && !keep[s]) ev[nv++] = s;
    }
    for (int i = 1; i < nv; ++i) {         /* insertion sort by (score asc, index asc) */
        int x = ev[i], j = i - 1;
        while (j >= 0 && (st->score[st->slot_expert[x]] < st->score[st->slot_expert[ev[j]]] ||
                          (st->score[st->slot_expert[x]] == st->score[st->slot_expert[ev[j]]] && x < ev[j]))) {
            ev[j + 1] = ev[j];
            --j;
        }
        ev[j + 1] = x;
    }
    /* misses by (score desc, id asc) */
    int32_t *order = (int32_t *)malloc(sizeof(int32_t) * (nM > 0 ? nM : 1));
    for (int i = 0; i < nM; ++i) order[i] = M[i];
    for (int i = 1; i < nM; ++i) {
        int32_t x = order[i];
        int j = i - 1;
        while (j >= 0 && (st->score[x] > st->score[order[j]] || (st->score[x] == st->score[order[j]] && x < order[j]))) {
            order[j + 1] = order[j];
            --j;
        }
        order[j + 1] = x;
    }
    int remaining = st->budget > 0 ? st->budget : S + 1;
    int fi = 0, vi = 0;
    for (int i = 0; i < nM; ++i) {
        const int m = order[i];
        int s = -1, old = -1;
        if (remaining > 0) {
            if (fi < nf) s = fr[fi++];
            else if (vi < nv && st->score[m] > st->score[st->slot_expert[ev[vi]]]) { s = ev[vi++]; old = st->slot_expert[s]; }
        }
        if (s >= 0) {
            remaining -= 1;
            if (old >= 0) { st->expert_slot[old] = -1; info->n_evict++; }
            st->slot_expert[s] = m;
            st->expert_slot[m] = s;
            st->slot_stamp[s] = now;
            e_slot[m] = s;
            d_old[m] = old;
        } else {
            info->n_bypass++;
        }
    }
    for (int i = 0; i < nM; ++i) {
        miss_expert[i] = M[i];
        miss_slot[i] = e_slot[M[i]];
        miss_evicted[i] = d_old[M[i]];
        miss_stage[i] = 0;
    }
    for (long p = 0; p < (long)T * k; ++p) {
        gpu_slot[p] = e_slot[ids[p]];
        stage[p] = 0;
    }
    free(used); free(cnt); free(keep); free(M); free(e_slot); free(d_old); free(was_hit); free(fr); free(ev);
    free(order);
    return 0;
}

/*
 * Plan one call of one layer: ids[T*k] (router picks) -> gpu_slot[T*k],
 * stage[T*k], the miss list (expert, slot, evicted expert or -1, stage) in
 * ascending expert order, and the summary.  Updates the state.
 *
 * Rule (plain reading of per-layer LRU + per-batch planning):
 *   clock += 1.  U = distinct picked experts, ascending.  Hits = experts of U
 *   already cached; misses M = the rest, ascending.
 *   If |U| <= S: one stage.  Otherwise stage 0 = hits + the first S-|hits|
 *   misses; every later stage takes the next S misses.
 *   Every hit slot is stamped with the clock.  Stage 0 victims: empty slots
 *   (ascending index), then slots whose expert is not picked in this call, by
 *   ascending (stamp, index); experts needed by the call are never victims.
 *   Later-stage victims: slots holding experts of this call's earlier stages,
 *   by ascending (stamp, index).  The i-th miss of a stage takes its i-th
 *   victim; the victim's old expert is marked not cached; the slot gets the
 *   clock as stamp.
 *
 * Policy 2 (LRU with adopt; the prefill preheat of "llama.cpp: fork with multi
 * gpu acceleration ...", section "Prefill preheat": a long prompt's most-used
 * experts stay in the cache, in place of cached experts it used less).  Calls
 * of one stage are planned exactly as LRU.  A call of more than one stage:
 *   rank = (pick count in this call descending, expert id ascending).
 *   Misses are taken lowest rank first (count ascending, id descending), so
 *   that the most-used misses are streamed last; stage 0 as for LRU.
 *   With m misses left after stage 0, G = ceil(m / S) later stages (as many as
 *   LRU needs) stream them through C = ceil(m / G) slots: the S - C slots whose
 *   stage-0 expert ranks highest keep it to the end; the other C slots, in
 *   ascending index, take the i-th later miss at stage 1 + i / C, slot
 *   number i mod C among them.
 */
/* a ranks above b among the call's experts: more picks, then the lower id */
static int adopt_above(const int32_t *cnt, int a, int b) {
    return cnt[a] > cnt[b] || (cnt[a] == cnt[b] && a < b);
}

int orc_slot_map(orc_lru *st, const int32_t *ids, int T, int k,
                 int32_t *gpu_slot, int32_t *stage,
                 int32_t *miss_expert, int32_t *miss_slot, int32_t *miss_evicted,
                 int32_t *miss_stage, orc_plan_info *info) {
    if (st->policy == 1)
        return slot_map_score(st, ids, T, k, gpu_slot, stage, miss_expert, miss_slot, miss_evicted, miss_stage, info);
    const int S = st->S, E = st->E;
    memset(info, 0, sizeof(*info));
    st->clock += 1;
    const uint64_t now = st->clock;

    unsigned char *used = (unsigned char *)calloc((size_t)E, 1);
    int32_t *cnt = (int32_t *)calloc((size_t)E, sizeof(int32_t));
    for (long p = 0; p < (long)T * k; ++p) { used[ids[p]] = 1; cnt[ids[p]] += 1; }

    int32_t *U = (int32_t *)malloc(sizeof(int32_t) * E), nU = 0;
    int32_t *M = (int32_t *)malloc(sizeof(int32_t) * E), nM = 0;
    int32_t *e_stage = (int32_t *)malloc(sizeof(int32_t) * E);
    int32_t *e_slot = (int32_t *)malloc(sizeof(int32_t) * E);
    unsigned char *was_hit = (unsigned char *)calloc((size_t)E, 1);
    unsigned char *in_call = (unsigned char *)calloc((size_t)S, 1); /* slot holds an expert of this call */
    int nH = 0;
    for (int e = 0; e < E; ++e) {
        e_stage[e] = -1;
        e_slot[e] = -1;
        if (!used[e]) continue;
        U[nU++] = e;
        if (st->expert_slot[e] >= 0) { was_hit[e] = 1; ++nH; }
        else M[nM++] = e;
    }
    info->n_unique = nU;
    info->n_hits = nH;
    info->n_miss = nM;
    for (long p = 0; p < (long)T * k; ++p) {
        if (was_hit[ids[p]]) info->pick_hits++;
        else info->pick_misses++;
    }

    /* hits: stage 0, keep their slot, refresh stamp */
    for (int i = 0; i < nU; ++i) {
        int e = U[i];
        if (!was_hit[e]) continue;
        int s = st->expert_slot[e];
        st->slot_stamp[s] = now;
        e_stage[e] = 0;
        e_slot[e] = s;
        in_call[s] = 1;
    }

    const int adopt = st->policy == 2 && nU > S;
    if (adopt) {
        /* misses lowest rank first (insertion sort) */
        for (int i = 1; i < nM; ++i) {
            const int e = M[i];
            int j = i - 1;
            while (j >= 0 && adopt_above(cnt, M[j], e)) { M[j + 1] = M[j]; --j; }
            M[j + 1] = e;
        }
    }

    int n_stage0_miss = (nU <= S) ? nM : (S - nH);
    int *cand = (int *)malloc(sizeof(int) * S);
    int n_cand = 0;
    for (int s = 0; s < S; ++s) {
        int e = st->slot_expert[s];
        if (e < 0 || !used[e]) cand[n_cand++] = s;
    }
    sort_victims(st, cand, n_cand);

    int mi = 0, n_stages = 1;
    /* stage 0 misses */
    for (int i = 0; i < n_stage0_miss; ++i, ++mi) {
        int e = M[mi], s = cand[i];
        int old = st->slot_expert[s];
        if (old >= 0) { st->expert_slot[old] = -1; info->n_evict++; }
        st->slot_expert[s] = e;
        st->expert_slot[e] = s;
        st->slot_stamp[s] = now;
        in_call[s] = 1;
        e_stage[e] = 0;
        e_slot[e] = s;
        miss_expert[mi] = e; miss_slot[mi] = s; miss_evicted[mi] = old; miss_stage[mi] = 0;
    }
    /* later stages, policy 2: the S - C slots holding the highest-ranked
     * experts keep them; the others stream the misses left */
    if (adopt && mi < nM) {
        const int m = nM - mi;
        const int G = (m + S - 1) / S, C = (m + G - 1) / G;
        int *order = (int *)malloc(sizeof(int) * S); /* slots by their expert's rank */
        for (int s2 = 0; s2 < S; ++s2) order[s2] = s2;
        for (int i = 1; i < S; ++i) {
            const int v = order[i];
            int j = i - 1;
            while (j >= 0 && adopt_above(cnt, st->slot_expert[v], st->slot_expert[order[j]])) {
                order[j + 1] = order[j];
                --j;
            }
            order[j + 1] = v;
        }
        unsigned char *kept = (unsigned char *)calloc((size_t)S, 1);
        for (int i = 0; i < S - C; ++i) kept[order[i]] = 1;
        int nq = 0;
        for (int s2 = 0; s2 < S; ++s2)
            if (!kept[s2]) cand[nq++] = s2;
        for (int i = 0; mi < nM; ++i, ++mi) {
            const int e = M[mi], s2 = cand[i % C], j = 1 + i / C;
            const int old = st->slot_expert[s2];
            if (old >= 0) { st->expert_slot[old] = -1; info->n_evict++; }
            st->slot_expert[s2] = e;
            st->expert_slot[e] = s2;
            st->slot_stamp[s2] = now;
            e_stage[e] = j;
            e_slot[e] = s2;
            miss_expert[mi] = e; miss_slot[mi] = s2; miss_evicted[mi] = old; miss_stage[mi] = j;
            if (j + 1 > n_stages) n_stages = j + 1;
        }
        free(order);
        free(kept);
    }
    /* later stages */
    for (int j = 1; mi < nM; ++j) {
        n_stages = j + 1;
        n_cand = 0;
        for (int s = 0; s < S; ++s)
            if (in_call[s]) cand[n_cand++] = s;
        sort_victims(st, cand, n_cand);
        int take = nM - mi < S ? nM - mi : S;
        if (take > n_cand) take = n_cand;  /* cannot happen: all S slots hold this call's experts */
        for (int i = 0; i < take; ++i, ++mi) {
            int e = M[mi], s = cand[i];
            int old = st->slot_expert[s];
            if (old >= 0) { st->expert_slot[old] = -1; info->n_evict++; }
            st->slot_expert[s] = e;
            st->expert_slot[e] = s;
            st->slot_stamp[s] = now;
            e_stage[e] = j;
            e_slot[e] = s;
            miss_expert[mi] = e; miss_slot[mi] = s; miss_evicted[mi] = old; miss_stage[mi] = j;
        }
    }
    info->n_stages = n_stages;

    for (long p = 0; p < (long)T * k; ++p) {
        gpu_slot[p] = e_slot[ids[p]];
        stage[p] = e_stage[ids[p]];
    }
    free(used); free(cnt); free(U); free(M); free(e_stage); free(e_slot); free(was_hit); free(in_call); free(cand);
    return 0;
}

/* ------------------------------------------------------------- expert FFN */

/*
 * One expert on one token.  blk = [gate F x H][up F x H][down H x F] in Q4_0
 * rows.  g = W_gate x, u = W_up x, h = g / (1 + exp(-g)) * u, y = W_down h.
 * Optional outputs g, u, h (length F) for inspection; y has length H.
 */
void orc_expert_ffn_parts(const uint8_t *blk, int H, int F, const double *x,
                          double *g_out, double *u_out, double *h_out, double *y) {
    const int nbH = H / 32, nbF = F / 32;
    const uint8_t *gate = blk;
    const uint8_t *up = blk + (size_t)F * nbH * 18;
    const uint8_t *down = up + (size_t)F * nbH * 18;
    double *h = (double *)malloc(sizeof(double) * F);
    for (int r = 0; r < F; ++r) {
        double g = row_dot(gate + (size_t)r * nbH * 18, nbH, x);
        double u = row_dot(up + (size_t)r * nbH * 18, nbH, x);
        h[r] = g / (1.0 + exp(-g)) * u;
        if (g_out) g_out[r] = g;
        if (u_out) u_out[r] = u;
        if (h_out) h_out[r] = h[r];
    }
    for (int i = 0; i < H; ++i) y[i] = row_dot(down + (size_t)i * nbF * 18, nbF, h);
    free(h);
}

void orc_expert_ffn(const uint8_t *blk, int H, int F, const double *x, double *y) {
    orc_expert_ffn_parts(blk, H, F, x, NULL, NULL, NULL, y);
}

/* ------------------------------------------------------- the whole layer */

enum {
    ORC_STAT_CALLS = 0,
    ORC_STAT_PICK_HITS,
    ORC_STAT_PICK_MISSES,
    ORC_STAT_UNIQUE_HITS,
    ORC_STAT_UNIQUE_MISSES,
    ORC_STAT_EVICTIONS,
    ORC_STAT_BYTES_UPLOADED,
    ORC_STAT_STAGES,
    ORC_STAT_STAGED_CALLS,
    ORC_STAT_BYPASSED,
    ORC_NSTAT
};

typedef struct {
    int L, E, k, H, F, S, weight_mode;
    const uint8_t *store;          /* host store, canonical Q4_0 blocks */
    uint64_t layer_stride, expert_stride, expert_bytes;
    orc_lru **lru;                 /* [L] */
    const uint8_t **slot_src;      /* [L*S] the store block each simulated slot holds */
    uint64_t *stats;               /* [L*ORC_NSTAT] */
    uint32_t *usage;               /* [L*E] lifetime activation counts */
    int n_threads;
} orc_cache;

orc_cache *orc_cache_new(int L, int E, int k, int H, int F, int S, int weight_mode,
                         const uint8_t *store, uint64_t layer_stride, uint64_t expert_stride,
                         int n_threads, int policy, int budget) {
    orc_cache *c = (orc_cache *)calloc(1, sizeof(orc_cache));
    c->L = L; c->E = E; c->k = k; c->H = H; c->F = F; c->S = S; c->weight_mode = weight_mode;
    c->store = store;
    c->layer_stride = layer_stride;
    c->expert_stride = expert_stride;
    c->expert_bytes = 3ull * F * (H / 32) * 18;
    c->lru = (orc_lru **)malloc(sizeof(orc_lru *) * L);
    for (int l = 0; l < L; ++l) {
        c->lru[l] = orc_lru_new(S, E);
        orc_lru_set_policy(c->lru[l], policy, budget);
    }
    c->slot_src = (const uint8_t **)calloc((size_t)L * S, sizeof(uint8_t *));
    c->stats = (uint64_t *)calloc((size_t)L * ORC_NSTAT, sizeof(uint64_t));
    c->usage = (uint32_t *)calloc((size_t)L * E, sizeof(uint32_t));
    c->n_threads = n_threads;
    return c;
}

void orc_cache_free(orc_cache *c) {
    if (!c) return;
    for (int l = 0; l < c->L; ++l) orc_lru_free(c->lru[l]);
    free(c->lru);
    free(c->slot_src);
    free(c->stats);
    free(c->usage);
    free(c);
}

orc_lru *orc_cache_lru(orc_cache *c, int layer) { return c->lru[layer]; }

/*
 * Warm start from a usage profile ("Persistent hot experts": each layer's
 * most-used experts are preloaded before the first request).  counts[L][E]:
 * usage per (layer, expert).  Per layer, the experts with a non-zero count,
 * by (count descending, id ascending), the first S of them in slots 0, 1, ...;
 * every other slot empty; stamps 0; the clock, scores and counters unchanged.
 */
/* Sticky share of policy 1 on every layer, per mille of the slots. */
void orc_cache_set_sticky(orc_cache *c, int permille) {
    for (int l = 0; l < c->L; ++l) orc_lru_set_sticky(c->lru[l], permille);
}

void orc_cache_preload(orc_cache *c, const uint32_t *counts) {
    for (int l = 0; l < c->L; ++l) {
        orc_lru *st = c->lru[l];
        const uint32_t *cnt = counts + (size_t)l * c->E;
        int32_t *order = (int32_t *)malloc(sizeof(int32_t) * c->E);
        int n = 0;
        for (int e = 0; e < c->E; ++e)
            if (cnt[e] > 0) order[n++] = e;
        for (int i = 1; i < n; ++i) {      /* insertion sort by (count desc, id asc) */
            int32_t x = order[i];
            int j = i - 1;
            while (j >= 0 && (cnt[x] > cnt[order[j]] || (cnt[x] == cnt[order[j]] && x < order[j]))) {
                order[j + 1] = order[j];
                --j;
            }
            order[j + 1] = x;
        }
        for (int e = 0; e < c->E; ++e) st->expert_slot[e] = -1;
        for (int sl = 0; sl < c->S; ++sl) {
            st->slot_expert[sl] = -1;
            st->slot_stamp[sl] = 0;
            c->slot_src[(size_t)l * c->S + sl] = NULL;
        }
        for (int i = 0; i < n && i < c->S; ++i) {
            st->slot_expert[i] = order[i];
            st->expert_slot[order[i]] = i;
            c->slot_src[(size_t)l * c->S + i] = c->store + (size_t)l * c->layer_stride + (size_t)order[i] * c->expert_stride;
        }
        free(order);
    }
}

/*
 * Lifetime activation counts ("Persistent hot experts": the cache keeps how
 * often each expert was used, n_layer x n_expert u32, and saves them at
 * shutdown for the next start's preload).  Reading taken: one count per routed
 * (token, pick) pair of every accepted call, whatever its slot outcome (hit,
 * miss, bypass), added when the call is planned; a rejected call (non-finite
 * logit, policy 1 over one stage) counts nothing; u32 arithmetic wraps.
 * out[L][E].
 */
void orc_cache_usage(const orc_cache *c, uint32_t *out) {
    memcpy(out, c->usage, sizeof(uint32_t) * (size_t)c->L * c->E);
}

/*
 * Resume from a saved state (the page saves usage counts only; restoring the
 * slot tables themselves is this library's addition): layer `layer` takes
 * slot_expert[S] (-1 = empty), slot_stamp[S], clock, score[E] (policy 1) and
 * usage[E]; expert_slot is derived and each occupied slot holds its expert's
 * block of the store.  Returns -1, state untouched, when an expert id is out of
 * [-1, E), an expert sits in two slots, an occupied slot's stamp is above the
 * clock, or a score is negative or not finite; else 0.
 */
int orc_cache_set_state(orc_cache *c, int layer, const int32_t *slot_expert, const uint64_t *slot_stamp,
                        uint64_t clock, const float *score, const uint32_t *usage) {
    const int S = c->S, E = c->E;
    orc_lru *st = c->lru[layer];
    for (int sl = 0; sl < S; ++sl) {
        int32_t e = slot_expert[sl];
        if (e < -1 || e >= E) return -1;
        if (e >= 0 && slot_stamp[sl] > clock) return -1;
        for (int s2 = 0; s2 < sl; ++s2)
            if (e >= 0 && slot_expert[s2] == e) return -1;
    }
    for (int e = 0; e < E; ++e)
        if (!(score[e] >= 0.0f) || isinf(score[e])) return -1;
    for (int e = 0; e < E; ++e) st->expert_slot[e] = -1;
    for (int sl = 0; sl < S; ++sl) {
        int32_t e = slot_expert[sl];
        st->slot_expert[sl] = e;
        st->slot_stamp[sl] = slot_stamp[sl];
        if (e >= 0) st->expert_slot[e] = sl;
        c->slot_src[(size_t)layer * S + sl] =
            e >= 0 ? c->store + (size_t)layer * c->layer_stride + (size_t)e * c->expert_stride : NULL;
    }
    st->clock = clock;
    memcpy(st->score, score, sizeof(float) * E);
    memcpy(c->usage + (size_t)layer * E, usage, sizeof(uint32_t) * E);
    return 0;
}

void orc_cache_stats(const orc_cache *c, int layer, uint64_t *out) {
    memcpy(out, c->stats + (size_t)layer * ORC_NSTAT, sizeof(uint64_t) * ORC_NSTAT);
}

/*
 * One routed-MoE layer call.  logits [T][E] fp32; x [T][H] as fp32 (x_bf16 = 0)
 * or raw bf16 bits (x_bf16 = 1).  If `compute` is 0 only the router and the slot
 * map run (the state still advances) and `out` is not written.
 * Optional outputs: ids, w (double), gpu_slot, stage [T*k]; miss list arrays
 * [<= min(E, T*k)]; pair_visits [T*k] (how many times each (token, pick) pair
 * was computed); info.
 * Returns 0, -1 when a logit is not finite, -2 when the layer uses policy 1
 * and the call needs more than one stage (state untouched in both cases).
 */
int orc_layer_forward(orc_cache *c, int layer, const float *logits, const void *x, int x_bf16,
                      int T, int compute, float *out,
                      int32_t *ids_out, double *w_out, int32_t *gpu_slot_out, int32_t *stage_out,
                      int32_t *miss_expert, int32_t *miss_slot, int32_t *miss_evicted,
                      int32_t *miss_stage, int32_t *pair_visits, orc_plan_info *info_out) {
    const int E = c->E, k = c->k, H = c->H, S = c->S;
    const long P = (long)T * k;
    if (T <= 0) return 0;
    int32_t *ids = (int32_t *)malloc(sizeof(int32_t) * P);
    double *w = (double *)malloc(sizeof(double) * P);
    /* step 1: router */
    if (orc_router(logits, T, E, k, c->weight_mode, ids, w) != 0) { free(ids); free(w); return -1; }

    /* step 2: slot table / LRU plan (misses populated per stage below) */
    int32_t *gpu_slot = (int32_t *)malloc(sizeof(int32_t) * P);
    int32_t *stage = (int32_t *)malloc(sizeof(int32_t) * P);
    int maxm = E < P ? E : (int)P;
    int32_t *me = (int32_t *)malloc(sizeof(int32_t) * maxm);
    int32_t *ms = (int32_t *)malloc(sizeof(int32_t) * maxm);
    int32_t *mv = (int32_t *)malloc(sizeof(int32_t) * maxm);
    int32_t *mst = (int32_t *)malloc(sizeof(int32_t) * maxm);
    orc_plan_info info;
    if (orc_slot_map(c->lru[layer], ids, T, k, gpu_slot, stage, me, ms, mv, mst, &info) != 0) {
        free(ids); free(w); free(gpu_slot); free(stage); free(me); free(ms); free(mv); free(mst);
        return -2;  /* policy 1: the call needs more than one stage */
    }

    uint64_t *st = c->stats + (size_t)layer * ORC_NSTAT;
    st[ORC_STAT_CALLS] += 1;
    st[ORC_STAT_PICK_HITS] += (uint64_t)info.pick_hits;
    st[ORC_STAT_PICK_MISSES] += (uint64_t)info.pick_misses;
    st[ORC_STAT_UNIQUE_HITS] += (uint64_t)info.n_hits;
    st[ORC_STAT_UNIQUE_MISSES] += (uint64_t)info.n_miss;
    st[ORC_STAT_EVICTIONS] += (uint64_t)info.n_evict;
    st[ORC_STAT_BYTES_UPLOADED] += (uint64_t)info.n_miss * c->expert_bytes;
    st[ORC_STAT_STAGES] += (uint64_t)info.n_stages;
    st[ORC_STAT_STAGED_CALLS] += info.n_stages > 1 ? 1u : 0u;
    st[ORC_STAT_BYPASSED] += (uint64_t)info.n_bypass;
    for (long p = 0; p < P; ++p) c->usage[(size_t)layer * E + ids[p]] += 1u;

    int32_t *visits = (int32_t *)calloc((size_t)P, sizeof(int32_t));
    const uint8_t **slot_src = c->slot_src + (size_t)layer * S;
    const uint8_t *layer_base = c->store + (size_t)layer * c->layer_stride;
    double *y = NULL, *xd = NULL;
    if (compute) {
        y = (double *)malloc(sizeof(double) * P * H);
        xd = (double *)malloc(sizeof(double) * (size_t)T * H);
        for (long i = 0; i < (long)T * H; ++i)
            xd[i] = x_bf16 ? orc_bf16_to_double(((const uint16_t *)x)[i])
                           : (double)((const float *)x)[i];
    }
    /* step 3, stage by stage: populate the stage's missing slots, then compute
     * every pair of the stage from its slot */
    for (int j = 0; j < info.n_stages; ++j) {
        for (int i = 0; i < info.n_miss; ++i)
            if (mst[i] == j && ms[i] >= 0) slot_src[ms[i]] = layer_base + (size_t)me[i] * c->expert_stride;
        if (!compute) {
            for (long p = 0; p < P; ++p) if (stage[p] == j) visits[p] += 1;
            continue;
        }
#ifdef _OPENMP
        if (c->n_threads > 0) omp_set_num_threads(c->n_threads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
        for (long p = 0; p < P; ++p) {
            if (stage[p] != j) continue;
            /* a bypassed miss (policy 1) is computed from its store block */
            const uint8_t *blk = gpu_slot[p] >= 0 ? slot_src[gpu_slot[p]]
                                                  : layer_base + (size_t)ids[p] * c->expert_stride;
            orc_expert_ffn(blk, H, c->F, xd + (size_t)(p / k) * H, y + (size_t)p * H);
            visits[p] += 1;
        }
    }
    /* step 4: weighted sum over the picks, ascending pick order */
    if (compute) {
        for (int t = 0; t < T; ++t) {
            for (int i = 0; i < H; ++i) {
                double acc = 0.0;
                for (int q = 0; q < k; ++q) acc += w[(long)t * k + q] * y[((size_t)t * k + q) * H + i];
                out[(size_t)t * H + i] = (float)acc;
            }
        }
    }
    if (ids_out) memcpy(ids_out, ids, sizeof(int32_t) * P);
    if (w_out) memcpy(w_out, w, sizeof(double) * P);
    if (gpu_slot_out) memcpy(gpu_slot_out, gpu_slot, sizeof(int32_t) * P);
    if (stage_out) memcpy(stage_out, stage, sizeof(int32_t) * P);
    if (miss_expert) memcpy(miss_expert, me, sizeof(int32_t) * info.n_miss);
    if (miss_slot) memcpy(miss_slot, ms, sizeof(int32_t) * info.n_miss);
    if (miss_evicted) memcpy(miss_evicted, mv, sizeof(int32_t) * info.n_miss);
    if (miss_stage) memcpy(miss_stage, mst, sizeof(int32_t) * info.n_miss);
    if (pair_visits) memcpy(pair_visits, visits, sizeof(int32_t) * P);
    if (info_out) *info_out = info;
    free(ids); free(w); free(gpu_slot); free(stage); free(me); free(ms); free(mv); free(mst);
    free(visits); free(y); free(xd);
    return 0;
}

int orc_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
