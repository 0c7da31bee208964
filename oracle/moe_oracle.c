/*
 * CPU oracle for the routed mixture-of-experts FFN of a decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the plain, slow, obviously correct
 * definition that the CUDA library is checked against.  It shares no code,
 * header, table or helper with the CUDA path, and the product never links,
 * loads or calls it.  Only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg use it.
 *
 * Everything is written out from the definitions, in fp64, one element at a
 * time, with no blocking, fusion or reordering beyond the definition:
 *
 *  - INT4 affine groups of 64 with a 16-bit (scale, bias) per group
 *    (TurboFieldfare, "Vectorization helped when it respected the storage
 *    layout"): weight = scale * q + bias, q in 0..15.
 *  - Router: logits over all experts, pick the top k (the TurboFieldfare
 *    video walkthrough: 8 of 128 experts are named per token and only those
 *    are evaluated), gates = softmax over the k picked logits.
 *  - Each picked expert and the shared expert (evaluated for every token,
 *    same video) compute down( GELU(gate x) * (up x) ).
 *  - Combine: y = y_shared + sum_j gate_j * y_{e_j}.
 *  - Per-layer LRU slot cache (TurboFieldfare, "MoE needed parallel work,
 *    reuse, and coarse overlap": a bounded cache of 16 routed experts per
 *    layer, LRU; goinfer "When the model doesn't fit": plain LRU).
 *
 * Readings where the pages leave a step open:
 *  - router logits are exact fixed point on a 2^-40 grid: every fp16 x bf16
 *    product is rounded half-to-even to a multiple of 2^-40 and summed in
 *    int64, so the sum does not depend on summation order and ties are
 *    well defined (ties go to the lower expert index);
 *  - the gates are renormalised over the k picked experts;
 *  - GELU is the exact erf form (variant 0) or the tanh form (variant 1);
 *  - in a layer stack each layer's FFN input is the RMS-normalised residual
 *    (x = bf16(h / sqrt(mean(h^2) + eps))) and the residual update is
 *    h' = bf16(h + y), both rounded half-to-even;
 *  - LRU: hits refresh their slot; misses, in top-k order, take the slot with
 *    the smallest (last_use, slot index) among slots neither hit nor filled
 *    in this step; empty slots carry last_use = -1.
 *
 * The rows of a matrix-vector product may be spread over host threads
 * (or_set_threads, OpenMP when the compiler has it; one thread by default):
 * each row is still summed by one thread in index order, so no result depends
 * on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define OR_OK 0
#define OR_EDOMAIN 1   /* router product outside |p| < 2^11, or non-finite input */
#define OR_EARG 2

/* ---- 16-bit float decoding, from the IEEE 754 binary16 / bfloat16 definitions ---- */

double or_fp16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 10) & 0x1f;
    int mant = bits & 0x3ff;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -24);                 /* subnormal: mant * 2^-24 */
    else if (expo == 31)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + mant), expo - 25);  /* (1 + mant/1024) * 2^(e-15) */
    return sign ? -v : v;
}

double or_bf16_to_double(uint16_t bits)
{
    int sign = (bits >> 15) & 1;
    int expo = (bits >> 7) & 0xff;
    int mant = bits & 0x7f;
    double v;
    if (expo == 0)
        v = ldexp((double)mant, -133);                /* subnormal: mant * 2^-133 */
    else if (expo == 255)
        v = mant ? NAN : INFINITY;
    else
        v = ldexp((double)(128 + mant), expo - 134);  /* (1 + mant/128) * 2^(e-127) */
    return sign ? -v : v;
}

/* Round a double to the nearest bfloat16 (ties to even), returning its bits. */
uint16_t or_double_to_bf16(double v)
{
    if (isnan(v))
        return 0x7fc0;
    uint16_t sign = signbit(v) ? 0x8000 : 0;
    double a = fabs(v);
    if (a == 0.0)
        return sign;
    int e;
    frexp(a, &e);                   /* a = m * 2^e, m in [0.5, 1) */
    int q_exp = e - 8;              /* 8 significant bits */
    if (q_exp < -133)
        q_exp = -133;               /* subnormal quantum */
    double quantum = ldexp(1.0, q_exp);
    double r = nearbyint(a / quantum) * quantum;   /* default mode: ties to even */
    if (r == 0.0)
        return sign;
    /* largest finite bfloat16 is (2 - 2^-7) * 2^127; beyond the midpoint to 2^128 -> inf */
    if (r >= ldexp(1.0, 128))
        return sign | 0x7f80;
    /* r is now exactly a bfloat16 value: encode it */
    int re;
    double m = frexp(r, &re);       /* r = m * 2^re */
    int biased = re - 1 + 127;      /* r = (2m) * 2^(re-1) */
    uint16_t bits;
    if (biased >= 1) {
        int mant = (int)ldexp(2.0 * m - 1.0, 7);
        bits = (uint16_t)((biased << 7) | mant);
    } else {
        int mant = (int)ldexp(r, 133);
        bits = (uint16_t)mant;      /* subnormal, or the smallest normal if mant == 128 */
    }
    return sign | bits;
}

/* ---- int4 affine weights ---- */

/* W[r][c] of a [rows][cols] projection in canonical layout. */
double or_weight(const uint8_t *q, const uint16_t *sb, int cols, int group, int r, int c)
{
    uint8_t byte = q[(size_t)r * (cols / 2) + c / 2];
    int nib = (c & 1) ? (byte >> 4) : (byte & 0xf);
    const uint16_t *p = sb + ((size_t)r * (cols / group) + c / group) * 2;
    double s = or_fp16_to_double(p[0]);
    double b = or_fp16_to_double(p[1]);
    return s * (double)nib + b;
}

static int or_threads = 1;

/* Host threads for the rows of or_matvec; returns the count in effect (1
 * without OpenMP). */
int or_set_threads(int n)
{
    or_threads = n < 1 ? 1 : n;
#ifdef _OPENMP
    return or_threads;
#else
    return 1;
#endif
}

/* y[rows] = W x, fp64 accumulation in index order. */
void or_matvec(const uint8_t *q, const uint16_t *sb, int rows, int cols, int group,
               const double *x, double *y)
{
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(or_threads) if (or_threads > 1)
#endif
    for (int r = 0; r < rows; ++r) {
        double acc = 0.0;
        for (int c = 0; c < cols; ++c)
            acc += or_weight(q, sb, cols, group, r, c) * x[c];
        y[r] = acc;
    }
}

double or_gelu(double x, int variant)
{
    if (variant == 1) {
        const double k0 = sqrt(2.0 / M_PI);
        return 0.5 * x * (1.0 + tanh(k0 * (x + 0.044715 * x * x * x)));
    }
    return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
}

/* One expert: y[d] = W_down ( GELU(W_gate x) * (W_up x) ), intermediate size f. */
void or_expert_ffn(const uint8_t *gq, const uint16_t *gsb, const uint8_t *uq, const uint16_t *usb,
                   const uint8_t *dq, const uint16_t *dsb, int d, int f, int group, int variant,
                   const double *x, double *y)
{
    double *g = (double *)malloc(sizeof(double) * (size_t)f);
    double *u = (double *)malloc(sizeof(double) * (size_t)f);
    double *a = (double *)malloc(sizeof(double) * (size_t)f);
    or_matvec(gq, gsb, f, d, group, x, g);
    or_matvec(uq, usb, f, d, group, x, u);
    for (int i = 0; i < f; ++i)
        a[i] = or_gelu(g[i], variant) * u[i];
    or_matvec(dq, dsb, d, f, group, a, y);
    free(g);
    free(u);
    free(a);
}

/* ---- router ---- */

/* l_e = sum_i RNE(2^40 * W[e][i] * x[i]) + RNE(2^40 * bias[e]), int64.
 * W fp16 bits [E][d], x bf16 bits [d], bias float [E] or NULL. */
int or_router_logits(const uint16_t *w, const uint16_t *x, const float *bias, int E, int d,
                     int64_t *logits)
{
    const double scale = ldexp(1.0, 40);
    const double lim = ldexp(1.0, 11);
    int status = OR_OK;
    for (int e = 0; e < E; ++e) {
        int64_t acc = 0;
        for (int i = 0; i < d; ++i) {
            double p = or_fp16_to_double(w[(size_t)e * d + i]) * or_bf16_to_double(x[i]);
            if (!(fabs(p) < lim)) {
                status = OR_EDOMAIN;
                continue;
            }
            acc += (int64_t)nearbyint(p * scale);
        }
        if (bias) {
            double b = (double)bias[e];
            if (!(fabs(b) < ldexp(1.0, 20)))
                status = OR_EDOMAIN;
            else
                acc += (int64_t)nearbyint(b * scale);
        }
        logits[e] = acc;
    }
    return status;
}

/* ids[0..k) = experts ranked by (logit descending, index ascending). */
void or_topk(const int64_t *logits, int E, int k, int32_t *ids)
{
    char *taken = (char *)calloc((size_t)E, 1);
    for (int j = 0; j < k; ++j) {
        int best = -1;
        for (int e = 0; e < E; ++e) {
            if (taken[e])
                continue;
            if (best < 0 || logits[e] > logits[best])
                best = e;   /* strict '>' keeps the lower index on ties */
        }
        taken[best] = 1;
        ids[j] = best;
    }
    free(taken);
}

/* gates_j = exp(2^-40 (l_j - l_0)) / sum over the k picked, l_0 the top logit. */
void or_gates(const int64_t *logits, const int32_t *ids, int k, double *gates)
{
    double sum = 0.0;
    int64_t top = logits[ids[0]];
    for (int j = 0; j < k; ++j) {
        gates[j] = exp(ldexp((double)(logits[ids[j]] - top), -40));
        sum += gates[j];
    }
    for (int j = 0; j < k; ++j)
        gates[j] /= sum;
}

/* ---- one layer, one token ---- */

typedef struct {
    int d, f, f_shared, n_experts, top_k, group, gelu_variant;
    const uint16_t *router_w;                       /* fp16 [E][d] */
    const uint8_t *gate_q, *up_q, *down_q;          /* [E][f][d/2], [E][f][d/2], [E][d][f/2] */
    const uint16_t *gate_sb, *up_sb, *down_sb;      /* [E][f][d/g][2], ..., [E][d][f/g][2] */
    const uint8_t *s_gate_q, *s_up_q, *s_down_q;    /* shared: [fs][d/2], [fs][d/2], [d][fs/2] */
    const uint16_t *s_gate_sb, *s_up_sb, *s_down_sb;
} or_layer;

/* x: bf16 bits [d] (the FFN input), bias: float [E] or NULL.
 * Outputs ids[k], gates[k], logits[E] (may be NULL), y[d]. */
int or_moe_layer(const or_layer *L, const uint16_t *x, const float *bias, int32_t *ids,
                 double *gates, int64_t *logits_out, double *y)
{
    const int d = L->d, f = L->f, fs = L->f_shared, E = L->n_experts, k = L->top_k, grp = L->group;
    if (k < 1 || k > E || d % grp || f % grp || fs % grp)
        return OR_EARG;
    int64_t *logits = (int64_t *)malloc(sizeof(int64_t) * (size_t)E);
    double *xd = (double *)malloc(sizeof(double) * (size_t)d);
    double *ye = (double *)malloc(sizeof(double) * (size_t)d);
    int st = or_router_logits(L->router_w, x, bias, E, d, logits);
    or_topk(logits, E, k, ids);
    or_gates(logits, ids, k, gates);
    for (int i = 0; i < d; ++i)
        xd[i] = or_bf16_to_double(x[i]);
    or_expert_ffn(L->s_gate_q, L->s_gate_sb, L->s_up_q, L->s_up_sb, L->s_down_q, L->s_down_sb,
                  d, fs, grp, L->gelu_variant, xd, y);
    const size_t gu_q = (size_t)f * d / 2, gu_sb = (size_t)f * (d / grp) * 2;
    const size_t dn_q = (size_t)d * f / 2, dn_sb = (size_t)d * (f / grp) * 2;
    for (int j = 0; j < k; ++j) {
        size_t e = (size_t)ids[j];
        or_expert_ffn(L->gate_q + e * gu_q, L->gate_sb + e * gu_sb, L->up_q + e * gu_q,
                      L->up_sb + e * gu_sb, L->down_q + e * dn_q, L->down_sb + e * dn_sb, d, f, grp,
                      L->gelu_variant, xd, ye);
        for (int i = 0; i < d; ++i)
            y[i] += gates[j] * ye[i];
    }
    if (logits_out)
        memcpy(logits_out, logits, sizeof(int64_t) * (size_t)E);
    free(logits);
    free(xd);
    free(ye);
    return st;
}

/* ---- residual stream between layers ---- */

void or_rmsnorm_bf16(const uint16_t *h, int d, double eps, uint16_t *x)
{
    double ss = 0.0;
    for (int i = 0; i < d; ++i) {
        double v = or_bf16_to_double(h[i]);
        ss += v * v;
    }
    double r = 1.0 / sqrt(ss / (double)d + eps);
    for (int i = 0; i < d; ++i)
        x[i] = or_double_to_bf16(or_bf16_to_double(h[i]) * r);
}

void or_residual_bf16(const uint16_t *h, const double *y, int d, uint16_t *out)
{
    for (int i = 0; i < d; ++i)
        out[i] = or_double_to_bf16(or_bf16_to_double(h[i]) + y[i]);
}

/* ---- per-layer LRU expert-slot cache ---- */

/* One step of one layer.  expert_of_slot[N] (-1 = empty), last_use[N] (-1 = empty)
 * are updated in place.  For each top-k position j: hit[j] (1/0), slot[j],
 * evicted[j] (expert that was in the slot before a miss, or -1).  Returns the
 * number of misses, or -1 if N < k. */
int or_lru_step(int n_slots, int32_t *expert_of_slot, int64_t *last_use, const int32_t *ids, int k,
                int64_t t, int32_t *hit, int32_t *slot, int32_t *evicted)
{
    if (n_slots < k)
        return -1;
    char *used = (char *)calloc((size_t)n_slots, 1);
    /* hits first */
    for (int j = 0; j < k; ++j) {
        hit[j] = 0;
        slot[j] = -1;
        evicted[j] = -1;
        for (int s = 0; s < n_slots; ++s) {
            if (expert_of_slot[s] == ids[j]) {
                hit[j] = 1;
                slot[j] = s;
                used[s] = 1;
                last_use[s] = t;
                break;
            }
        }
    }
    /* then misses, in top-k order */
    int misses = 0;
    for (int j = 0; j < k; ++j) {
        if (hit[j])
            continue;
        int victim = -1;
        for (int s = 0; s < n_slots; ++s) {
            if (used[s])
                continue;
            if (victim < 0 || last_use[s] < last_use[victim])
                victim = s;   /* strict '<' keeps the lower slot index on ties */
        }
        evicted[j] = expert_of_slot[victim];
        expert_of_slot[victim] = ids[j];
        last_use[victim] = t;
        used[victim] = 1;
        slot[j] = victim;
        ++misses;
    }
    free(used);
    return misses;
}

/* ---- per-layer LFU expert-slot cache ---- */

/* One step of one layer with least-frequently-used eviction.  use_count[E]
 * counts, over the whole run, how often each expert was picked (hit or miss);
 * it is incremented for every top-k position of this step.  Hits refresh
 * their slot's last_use; misses, in top-k order, take the slot that has the
 * smallest (use count of its expert, last_use, slot index) among slots
 * neither hit nor filled in this step, an empty slot counting -1 for both.
 * Outputs and return value as or_lru_step. */
int or_lfu_step(int n_slots, int32_t *expert_of_slot, int64_t *last_use, int64_t *use_count,
                const int32_t *ids, int k, int64_t t, int32_t *hit, int32_t *slot, int32_t *evicted)
{
    if (n_slots < k)
        return -1;
    char *used = (char *)calloc((size_t)n_slots, 1);
    for (int j = 0; j < k; ++j) {
        hit[j] = 0;
        slot[j] = -1;
        evicted[j] = -1;
        for (int s = 0; s < n_slots; ++s) {
            if (expert_of_slot[s] == ids[j]) {
                hit[j] = 1;
                slot[j] = s;
                used[s] = 1;
                last_use[s] = t;
                break;
            }
        }
    }
    int misses = 0;
    for (int j = 0; j < k; ++j) {
        if (hit[j])
            continue;
        int victim = -1;
        int64_t vc = 0;
        for (int s = 0; s < n_slots; ++s) {
            if (used[s])
                continue;
            const int64_t c = expert_of_slot[s] < 0 ? -1 : use_count[expert_of_slot[s]];
            if (victim < 0 || c < vc || (c == vc && last_use[s] < last_use[victim])) {
                victim = s;     /* strict comparisons keep the lower slot index on full ties */
                vc = c;
            }
        }
        evicted[j] = expert_of_slot[victim];
        expert_of_slot[victim] = ids[j];
        last_use[victim] = t;
        used[victim] = 1;
        slot[j] = victim;
        ++misses;
    }
    for (int j = 0; j < k; ++j)
        use_count[ids[j]] += 1;
    free(used);
    return misses;
}
