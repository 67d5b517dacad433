/*
 * moe_oracle.c -- reference oracle for the routed mixture-of-experts FFN layer.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously-correct CPU
 * definition that the CUDA library is checked against.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load it; the
 * library itself never calls it and shares no code, header, table or helper
 * with it.  Single-threaded, fp64 arithmetic throughout, no blocking, no
 * fusion, no reordering beyond what the definitions below state.
 *
 * What is computed (per token t, with E experts, top-k routing, hidden H,
 * expert intermediate I):
 *
 *   1. Routing.  The layer has E routed experts and each token is sent to k
 *      of them ("384 routed experts x 40 MoE layers"; dsv41-flash-offload
 *      wiki, overview).  The pages never write the router function down; the
 *      reading adopted here is: select the k largest fp32 logits, ties to the
 *      lower expert index, outputs in that order; gates are the softmax over
 *      the selected logits only, g_j = exp(l_j - m) / sum_i exp(l_i - m) with
 *      m the largest selected logit (equal, in exact arithmetic, to a full
 *      softmax renormalised over the selection).
 *   2. Route lists.  Per-expert token counts and per-expert lists of token
 *      slots ("route lists ... positive counts", dsv41-flash-offload wiki,
 *      file map).  Slot s = t*k + j; the list of expert e holds its slots in
 *      ascending s (textbook stable counting sort).
 *   3. Expert FFN.  SwiGLU expert, no bias, no scale, no shared expert:
 *      h = silu(Wg_e x) * (Wu_e x), y = Wd_e h, silu(z) = z / (1 + exp(-z)).
 *      Weights follow the [out, in] convention: Wg_e, Wu_e are [I, H],
 *      Wd_e is [H, I], row-major.  Which experts are "busy" (fat threshold 32,
 *      model page launch flags) changes where an expert runs, never what it
 *      computes, so the oracle has no such split.
 *   4. Combine.  out_t = sum_j g_j * y_j, in fixed j order, fp64; the
 *      deliverable is that value rounded to bf16 (round to nearest even)
 *      ("split/combine on GPU", dsv41-flash-offload wiki, file map).
 *
 * bf16 inputs arrive as their raw 16-bit patterns (uint16_t).
 * Preconditions checked here (return value -1 on violation): logits are
 * finite or -inf (no NaN, no +inf), each token's largest selected logit is
 * finite, 1 <= k <= E, every routed index lies in [0, E).
 */
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <math.h>

/* ------------------------------------------------------------------ */
/* bf16 <-> fp64                                                       */
/* ------------------------------------------------------------------ */

/* A bf16 value is the upper 16 bits of an IEEE binary32 value. */
static double bf16_bits_to_double(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 value (8 significant bits, binary32
 * exponent range, ties to even) and return its bit pattern.  Done in one
 * rounding step from fp64, not via fp32, so there is no double rounding. */
uint16_t oracle_double_to_bf16(double v)
{
    if (isnan(v))
        return (uint16_t)0x7FC0u;
    if (v == 0.0)
        return signbit(v) ? (uint16_t)0x8000u : (uint16_t)0x0000u;
    if (isinf(v))
        return v > 0 ? (uint16_t)0x7F80u : (uint16_t)0xFF80u;
    int e;
    (void)frexp(v, &e);            /* |v| = m * 2^e, 0.5 <= m < 1 */
    if (e < -125)
        e = -125;                  /* below the normal range the quantum is fixed */
    double quantum = ldexp(1.0, e - 8);
    double r = nearbyint(v / quantum) * quantum;   /* default mode: ties to even */
    const double bf16_max = ldexp(255.0, 127 - 7); /* 0x7F7F = 1.9921875 * 2^127 */
    if (r > bf16_max)
        return (uint16_t)0x7F80u;
    if (r < -bf16_max)
        return (uint16_t)0xFF80u;
    float f = (float)r;            /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

void oracle_array_to_bf16(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; ++i)
        out[i] = oracle_double_to_bf16(v[i]);
}

/* ------------------------------------------------------------------ */
/* 1. Routing                                                          */
/* ------------------------------------------------------------------ */

typedef struct {
    float value;
    int32_t index;
} scored_expert;

/* Total order: larger logit first; equal logits -> smaller index first.
 * (-0.0 and +0.0 compare equal here, as floats do.) */
static int by_logit_desc_index_asc(const void* pa, const void* pb)
{
    const scored_expert* a = (const scored_expert*)pa;
    const scored_expert* b = (const scored_expert*)pb;
    if (a->value > b->value) return -1;
    if (a->value < b->value) return 1;
    if (a->index < b->index) return -1;
    if (a->index > b->index) return 1;
    return 0;
}

/* logits: fp32 [T, E] row-major.  idx: int32 [T, k].  gates: fp64 [T, k].
 * Returns 0, or -1 on a precondition violation. */
int oracle_route(const float* logits, int64_t T, int E, int k,
                 int32_t* idx, double* gates)
{
    if (E < 1 || k < 1 || k > E || T < 0)
        return -1;
    scored_expert* row = (scored_expert*)malloc(sizeof(scored_expert) * (size_t)E);
    if (!row)
        return -1;
    for (int64_t t = 0; t < T; ++t) {
        const float* l = logits + t * (int64_t)E;
        for (int e = 0; e < E; ++e) {
            if (isnan(l[e]) || (isinf(l[e]) && l[e] > 0)) {
                free(row);
                return -1;
            }
            row[e].value = l[e];
            row[e].index = e;
        }
        /* The comparator is a total order, so any correct sort yields the
         * same sequence. */
        qsort(row, (size_t)E, sizeof(scored_expert), by_logit_desc_index_asc);
        double m = (double)row[0].value;
        if (!isfinite(m)) {
            free(row);
            return -1;
        }
        double denom = 0.0;
        for (int j = 0; j < k; ++j)
            denom += exp((double)row[j].value - m);
        for (int j = 0; j < k; ++j) {
            idx[t * k + j] = row[j].index;
            gates[t * k + j] = exp((double)row[j].value - m) / denom;
        }
    }
    free(row);
    return 0;
}

/* ------------------------------------------------------------------ */
/* 2. Route lists: stable counting sort of the slots by expert          */
/* ------------------------------------------------------------------ */

/* idx: int32 [T*k] (slot s = t*k + j).  counts: [E].  offsets: [E+1]
 * (exclusive prefix sum, offsets[E] = T*k).  perm[p] = slot at sorted
 * position p; inv_perm[s] = sorted position of slot s. */
int oracle_permute(const int32_t* idx, int64_t T, int E, int k,
                   int32_t* counts, int32_t* offsets,
                   int32_t* perm, int32_t* inv_perm)
{
    int64_t P = T * (int64_t)k;
    if (E < 1 || k < 1 || T < 0)
        return -1;
    for (int e = 0; e < E; ++e)
        counts[e] = 0;
    for (int64_t s = 0; s < P; ++s) {
        if (idx[s] < 0 || idx[s] >= E)
            return -1;
        counts[idx[s]] += 1;
    }
    offsets[0] = 0;
    for (int e = 0; e < E; ++e)
        offsets[e + 1] = offsets[e] + counts[e];
    int32_t* cursor = (int32_t*)malloc(sizeof(int32_t) * (size_t)E);
    if (!cursor)
        return -1;
    for (int e = 0; e < E; ++e)
        cursor[e] = offsets[e];
    for (int64_t s = 0; s < P; ++s) {
        int32_t p = cursor[idx[s]]++;
        perm[p] = (int32_t)s;
        inv_perm[s] = p;
    }
    free(cursor);
    return 0;
}

/* ------------------------------------------------------------------ */
/* 3. One expert applied to one token                                  */
/* ------------------------------------------------------------------ */

static double silu(double z)
{
    return z / (1.0 + exp(-z));
}

/* x: bf16 [H].  Wg, Wu: bf16 [I, H].  Wd: bf16 [H, I].  y: fp64 [H].
 * h: caller scratch fp64 [I] (returned, so tests can inspect it). */
void oracle_expert_ffn(const uint16_t* x, const uint16_t* Wg, const uint16_t* Wu,
                       const uint16_t* Wd, int H, int I, double* h, double* y)
{
    for (int i = 0; i < I; ++i) {
        double a = 0.0, b = 0.0;
        for (int c = 0; c < H; ++c) {
            double xc = bf16_bits_to_double(x[c]);
            a += bf16_bits_to_double(Wg[(int64_t)i * H + c]) * xc;
            b += bf16_bits_to_double(Wu[(int64_t)i * H + c]) * xc;
        }
        h[i] = silu(a) * b;
    }
    for (int r = 0; r < H; ++r) {
        double acc = 0.0;
        for (int i = 0; i < I; ++i)
            acc += bf16_bits_to_double(Wd[(int64_t)r * I + i]) * h[i];
        y[r] = acc;
    }
}

/* ------------------------------------------------------------------ */
/* 1+3+4. Whole layer for a list of tokens                             */
/* ------------------------------------------------------------------ */

/* Runs routing, the selected experts and the combine for n tokens.
 *   x:      bf16 [n, H]  (the tokens' activations)
 *   logits: fp32 [n, E]
 *   Wg, Wu, Wd: per-expert pointer tables of length E; entry e points at
 *           that expert's [I, H] / [I, H] / [H, I] bf16 matrix.  Entries of
 *           experts that no listed token selects may be NULL.
 *   out:    fp64 [n, H] combined output (not rounded).
 *   idx, gates: optional [n, k] routing results (may be NULL).
 * Returns 0, -1 on a precondition violation, -2 if a selected expert's
 * weights were not supplied. */
int oracle_moe_tokens(int64_t n, const uint16_t* x, const float* logits,
                      int E, int k, int H, int I,
                      const uint16_t* const* Wg, const uint16_t* const* Wu,
                      const uint16_t* const* Wd,
                      double* out, int32_t* idx, double* gates)
{
    int rc = 0;
    int32_t* sel = (int32_t*)malloc(sizeof(int32_t) * (size_t)k);
    double* g = (double*)malloc(sizeof(double) * (size_t)k);
    double* h = (double*)malloc(sizeof(double) * (size_t)I);
    double* y = (double*)malloc(sizeof(double) * (size_t)H);
    if (!sel || !g || !h || !y) {
        rc = -1;
        goto done;
    }
    for (int64_t t = 0; t < n; ++t) {
        if (oracle_route(logits + t * (int64_t)E, 1, E, k, sel, g) != 0) {
            rc = -1;
            goto done;
        }
        double* o = out + t * (int64_t)H;
        for (int c = 0; c < H; ++c)
            o[c] = 0.0;
        for (int j = 0; j < k; ++j) {
            int e = sel[j];
            if (!Wg[e] || !Wu[e] || !Wd[e]) {
                rc = -2;
                goto done;
            }
            oracle_expert_ffn(x + t * (int64_t)H, Wg[e], Wu[e], Wd[e], H, I, h, y);
            for (int c = 0; c < H; ++c)
                o[c] += g[j] * y[c];
        }
        if (idx)
            for (int j = 0; j < k; ++j)
                idx[t * k + j] = sel[j];
        if (gates)
            for (int j = 0; j < k; ++j)
                gates[t * k + j] = g[j];
    }
done:
    free(sel);
    free(g);
    free(h);
    free(y);
    return rc;
}

/* ------------------------------------------------------------------ */
/* 4. Combine on its own                                               */
/* ------------------------------------------------------------------ */

/* out[t] = sum_j gates[t*k+j] * y_sorted[inv_perm[t*k+j]], fp64, j ascending.
 *   y_sorted: fp64 [T*k, H]; inv_perm: int32 [T*k]; gates: fp64 [T*k];
 *   out: fp64 [T, H]. */
int oracle_combine(const double* y_sorted, const int32_t* inv_perm, const double* gates,
                   int64_t T, int k, int H, double* out)
{
    int64_t P = T * (int64_t)k;
    for (int64_t t = 0; t < T; ++t) {
        double* o = out + t * (int64_t)H;
        for (int c = 0; c < H; ++c)
            o[c] = 0.0;
        for (int j = 0; j < k; ++j) {
            int64_t p = inv_perm[t * k + j];
            if (p < 0 || p >= P)
                return -1;
            const double* y = y_sorted + p * (int64_t)H;
            for (int c = 0; c < H; ++c)
                o[c] += gates[t * k + j] * y[c];
        }
    }
    return 0;
}
