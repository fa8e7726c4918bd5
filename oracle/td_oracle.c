/*
 * td_oracle.c -- plain, slow CPU oracle for the TidalDecode decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may call, link or
 * load this file: only the tests, the package's smoke check and the bench's
 * CPU-baseline / reference arm use it.  It shares no code, header, table or
 * helper with the CUDA library; the two meet only through seeded inputs.
 *
 * What it computes, and from where (TidalDecode: Fast and Accurate LLM
 * Decoding with Position Persistent Sparse Attention -- paper review page):
 *
 *   - attention of one query head over a set of cached tokens,
 *     A = q K^T / sqrt(d), H = softmax(A) V          (review §三, "Position
 *     Persistent Sparse Attention (PPSA)", standard attention formula);
 *   - token selection: keep the k positions with the highest attention
 *     score (review §二, "core insight"; §三 Figure 2, "Full Attention +
 *     Token Selection -> top-k tokens");
 *   - position persistence: every later layer attends only to the positions
 *     chosen at the most recent selection layer (review §三, PPSA "reuse the
 *     token set of the previous selection layer"; Figure 2 rows "PPSA (reuse
 *     selected tokens)");
 *   - the per-step layer schedule [full | full+select | sparse]
 *     (review §三 Figure 2);
 *   - the overlap of two token sets (review §三, token-selection
 *     sensitivity, Figure 4(a));
 *   - a coverage budget for the selection (Token Sparse Attention page, §2
 *     "Dynamic Token Coverage").
 *
 * Readings where the page is silent:
 *   - "attention score" for selection is the scaled pre-softmax logit a;
 *   - with grouped-query attention the score of a KV head is the sum of the
 *     scaled logits of the query heads in its group;
 *   - ties at the k-th score go to the lower position; -0.0 equals +0.0;
 *   - the selected positions are stored in ascending order, padded with -1
 *     when the context is shorter than k;
 *   - softmax over an empty set gives an all-zero output;
 *   - scale is the fp32 value 1/sqrt(d), widened to double by the caller.
 *
 * Arithmetic: every input is a bf16 bit pattern widened exactly to double;
 * all sums, the exponential and the division are in double precision.
 * There is no blocking, fusion or reordering beyond the definition.
 *
 * Optional OpenMP: oracle_decode_step runs its independent (batch, KV head)
 * groups in parallel when compiled with -fopenmp; each group's arithmetic is
 * unchanged by this.
 *
 * ORACLE_MUTANT (compile-time, tests only): plants one deliberate mistake so
 * that the pin tests can show they catch it.  0 (the default) is the oracle.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifndef ORACLE_MUTANT
#define ORACLE_MUTANT 0
#endif

enum { MODE_FULL = 0, MODE_FULL_SELECT = 1, MODE_SPARSE = 2 };

enum {
    ORACLE_OK = 0,
    ORACLE_ERR_ARG = 1,
    ORACLE_ERR_NO_SELECTION = 2,
    ORACLE_ERR_NOMEM = 3
};

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
double oracle_bf16_to_double(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Scaled logit of one query head against one key row:
 *   a = scale * sum_i q[i] * k[i]                       (A = QK / sqrt(d)) */
double oracle_logit(const uint16_t *q, const uint16_t *krow, int d, double scale)
{
    double dot = 0.0;
    for (int i = 0; i < d; ++i) {
#if ORACLE_MUTANT == 12
        /* mutant: reads the key with a shifted feature index */
        dot += oracle_bf16_to_double(q[i]) * oracle_bf16_to_double(krow[(i + 1) % d]);
#else
        dot += oracle_bf16_to_double(q[i]) * oracle_bf16_to_double(krow[i]);
#endif
    }
#if ORACLE_MUTANT == 1
    (void)scale;
    return dot; /* mutant: the 1/sqrt(d) scale is dropped */
#else
    return scale * dot;
#endif
}

/* p = softmax(a) over n entries, p[j] = exp(a[j] - max a) / sum exp(a - max a).
 * n == 0 leaves p untouched. */
void oracle_softmax(const double *a, int n, double *p)
{
    if (n <= 0)
        return;
    double m = a[0];
    for (int j = 1; j < n; ++j)
        if (a[j] > m)
            m = a[j];
    double sum = 0.0;
    for (int j = 0; j < n; ++j) {
#if ORACLE_MUTANT == 3
        p[j] = exp(m - a[j]); /* mutant: sign of the exponent flipped */
#else
        p[j] = exp(a[j] - m);
#endif
        sum += p[j];
    }
#if ORACLE_MUTANT == 10
    (void)sum; /* mutant: the normaliser is missing */
#else
    for (int j = 0; j < n; ++j)
        p[j] /= sum;
#endif
}

/*
 * Attention of one query head over the rows `rows[0..n_rows)` of one KV head
 * (rows == NULL means rows 0..n_rows-1):
 *     a_j = scale * q . K[rows[j]],  p = softmax(a),  out = sum_j p_j V[rows[j]].
 * An empty row set gives out = 0.  `p_out` (optional, n_rows doubles)
 * receives the weights.  Returns ORACLE_OK or ORACLE_ERR_NOMEM.
 */
int oracle_attend(const uint16_t *q, const uint16_t *K, const uint16_t *V, int d,
                  const int32_t *rows, int n_rows, double scale,
                  double *out, double *p_out)
{
    for (int i = 0; i < d; ++i)
        out[i] = 0.0;
    if (n_rows <= 0)
        return ORACLE_OK;
    double *a = (double *)malloc(sizeof(double) * (size_t)n_rows);
    double *p = (double *)malloc(sizeof(double) * (size_t)n_rows);
    if (!a || !p) {
        free(a);
        free(p);
        return ORACLE_ERR_NOMEM;
    }
    for (int j = 0; j < n_rows; ++j) {
        int64_t r = rows ? rows[j] : j;
        a[j] = oracle_logit(q, K + r * (int64_t)d, d, scale);
    }
    oracle_softmax(a, n_rows, p);
    for (int j = 0; j < n_rows; ++j) {
#if ORACLE_MUTANT == 4
        int jv = (j + 1) % n_rows; /* mutant: value row paired with the next key */
        int64_t r = rows ? rows[jv] : jv;
#else
        int64_t r = rows ? rows[j] : j;
#endif
        const uint16_t *vrow = V + r * (int64_t)d;
        for (int i = 0; i < d; ++i)
            out[i] += p[j] * oracle_bf16_to_double(vrow[i]);
    }
    if (p_out)
        memcpy(p_out, p, sizeof(double) * (size_t)n_rows);
    free(a);
    free(p);
    return ORACLE_OK;
}

/*
 * Selection score of one KV head for the first n tokens: the sum over the G
 * query heads of its group of their scaled logits,
 *     s[t] = sum_h scale * q_h . K[t]          (q_group is [G][d]).
 */
void oracle_group_scores(const uint16_t *q_group, int G, const uint16_t *K, int d, int n,
                         double scale, double *s)
{
    for (int t = 0; t < n; ++t) {
        double acc = 0.0;
#if ORACLE_MUTANT == 7
        G = 1; /* mutant: only the first head of the group is scored */
#endif
        for (int h = 0; h < G; ++h)
            acc += oracle_logit(q_group + (int64_t)h * d, K + (int64_t)t * d, d, scale);
        s[t] = acc;
    }
}

typedef struct {
    double s;
    int32_t pos;
} scored_pos;

/* Order for selection: higher score first; equal scores, lower position first.
 * -0.0 and +0.0 compare equal under C's == and <, so they tie. */
static int by_score_desc_pos_asc(const void *x, const void *y)
{
    const scored_pos *a = (const scored_pos *)x, *b = (const scored_pos *)y;
#if ORACLE_MUTANT == 6
    if (a->s < b->s) return -1; /* mutant: keeps the lowest scores */
    if (a->s > b->s) return 1;
#else
    if (a->s > b->s) return -1;
    if (a->s < b->s) return 1;
#endif
#if ORACLE_MUTANT == 5
    return (a->pos < b->pos) ? 1 : (a->pos > b->pos) ? -1 : 0; /* mutant: ties to the higher index */
#else
    return (a->pos < b->pos) ? -1 : (a->pos > b->pos) ? 1 : 0;
#endif
}

static int by_int_asc(const void *x, const void *y)
{
    int32_t a = *(const int32_t *)x, b = *(const int32_t *)y;
    return (a < b) ? -1 : (a > b) ? 1 : 0;
}

/*
 * Top-k token selection over scores s[0..n): the first min(k, n) positions
 * of the order (score descending, position ascending), written to idx[0..k)
 * in ascending position order and padded with -1.  Returns the number kept.
 */
int oracle_topk(const double *s, int n, int k, int32_t *idx)
{
    if (k <= 0)
        return 0;
    int keep = n < k ? n : k;
#if ORACLE_MUTANT == 11
    if (keep > 0)
        keep -= 1; /* mutant: one position short */
#endif
    if (n > 0) {
        scored_pos *v = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)n);
        if (!v)
            return -1;
        for (int t = 0; t < n; ++t) {
            v[t].s = s[t];
            v[t].pos = t;
        }
        qsort(v, (size_t)n, sizeof(scored_pos), by_score_desc_pos_asc);
        for (int j = 0; j < keep; ++j)
            idx[j] = v[j].pos;
        free(v);
        qsort(idx, (size_t)keep, sizeof(int32_t), by_int_asc);
    }
    for (int j = keep; j < k; ++j)
        idx[j] = -1;
    return keep;
}

/* The entries of a persisted index set that are real positions (not -1). */
static int live_rows(const int32_t *idx, int k, int32_t *rows)
{
    int n = 0;
    for (int j = 0; j < k; ++j) {
#if ORACLE_MUTANT == 8
        rows[n++] = idx[j] < 0 ? 0 : idx[j]; /* mutant: padding read as position 0 */
#else
        if (idx[j] >= 0)
            rows[n++] = idx[j];
#endif
    }
    return n;
}

/*
 * One (batch row, KV head) group through an L-layer decode step
 * (review §三 Figure 2):
 *   FULL         every query head of the group attends over all n_b tokens;
 *   FULL_SELECT  the same, then the group's top-k positions are selected
 *                and become the persisted index set;
 *   SPARSE       every query head attends only over the persisted positions.
 *
 * Per layer l: q_group[l] is [G][d]; K[l], V[l] are [>= n_b][d] rows of this
 * KV head; out[l] is [G][d] doubles.  `idx_state` ([k]) carries the persisted
 * set between layers and `*idx_valid` says whether it holds one on entry and
 * exit.  `idx_per_layer` (optional, L pointers, each [k] or NULL) receives
 * the set each layer used (SPARSE) or produced (FULL_SELECT).
 * Returns ORACLE_ERR_NO_SELECTION for a sparse layer with no set.
 */
int oracle_decode_group(int L, const int32_t *modes, int G, int d, int n_b, int k, double scale,
                        const uint16_t *const *q_group, const uint16_t *const *K,
                        const uint16_t *const *V, int32_t *idx_state, int *idx_valid,
                        double *const *out, int32_t *const *idx_per_layer)
{
    if (L < 0 || G <= 0 || d <= 0 || n_b < 0 || k < 0 || !modes || !idx_valid)
        return ORACLE_ERR_ARG;
    int32_t *first_set = NULL; /* used only by mutant 9 */
    int rc = ORACLE_OK;
    int32_t *rows = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
    double *s = (double *)malloc(sizeof(double) * (size_t)(n_b > 0 ? n_b : 1));
    if (!rows || !s) {
        rc = ORACLE_ERR_NOMEM;
        goto done;
    }
    for (int l = 0; l < L; ++l) {
        int mode = modes[l];
        if (mode == MODE_FULL || mode == MODE_FULL_SELECT) {
            for (int h = 0; h < G; ++h) {
                rc = oracle_attend(q_group[l] + (int64_t)h * d, K[l], V[l], d, NULL, n_b, scale,
                                   out[l] + (int64_t)h * d, NULL);
                if (rc)
                    goto done;
            }
            if (mode == MODE_FULL_SELECT) {
                if (k <= 0 || !idx_state) {
                    rc = ORACLE_ERR_ARG;
                    goto done;
                }
                oracle_group_scores(q_group[l], G, K[l], d, n_b, scale, s);
                if (oracle_topk(s, n_b, k, idx_state) < 0) {
                    rc = ORACLE_ERR_NOMEM;
                    goto done;
                }
                *idx_valid = 1;
#if ORACLE_MUTANT == 9
                if (!first_set) { /* mutant: later layers keep the first selection */
                    first_set = (int32_t *)malloc(sizeof(int32_t) * (size_t)k);
                    memcpy(first_set, idx_state, sizeof(int32_t) * (size_t)k);
                } else {
                    memcpy(idx_state, first_set, sizeof(int32_t) * (size_t)k);
                }
#endif
                if (idx_per_layer && idx_per_layer[l])
                    memcpy(idx_per_layer[l], idx_state, sizeof(int32_t) * (size_t)k);
            }
        } else if (mode == MODE_SPARSE) {
            if (!*idx_valid || !idx_state) {
                rc = ORACLE_ERR_NO_SELECTION;
                goto done;
            }
            int n_live = live_rows(idx_state, k, rows);
            for (int h = 0; h < G; ++h) {
                rc = oracle_attend(q_group[l] + (int64_t)h * d, K[l], V[l], d, rows, n_live, scale,
                                   out[l] + (int64_t)h * d, NULL);
                if (rc)
                    goto done;
            }
            if (idx_per_layer && idx_per_layer[l])
                memcpy(idx_per_layer[l], idx_state, sizeof(int32_t) * (size_t)k);
        } else {
            rc = ORACLE_ERR_ARG;
            goto done;
        }
    }
done:
    free(first_set);
    free(rows);
    free(s);
    return rc;
}

/*
 * A whole decode step over batched tensors (one layer's tensors per pointer):
 *   q[l]   [B][Hq][d]          bf16 bits
 *   K[l]   [B][Hkv][Nmax][d]   bf16 bits (V[l] likewise)
 *   out[l] [B][Hq][d]          doubles
 *   idx_final [B][Hkv][k]      the persisted set after the last layer
 *                              (-1 everywhere if no layer selected)
 * Query head h belongs to KV head h / (Hq / Hkv).  Each (b, kv head) group is
 * independent, so the groups may run in parallel.
 */
int oracle_decode_step(int B, int Hq, int Hkv, int d, int Nmax, const int32_t *seq_lens,
                       int L, const int32_t *modes, int k, double scale,
                       const uint16_t *const *q, const uint16_t *const *K,
                       const uint16_t *const *V, double *const *out, int32_t *idx_final)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv || d <= 0 || Nmax < 0 || L < 0 || !seq_lens)
        return ORACLE_ERR_ARG;
    for (int b = 0; b < B; ++b)
        if (seq_lens[b] < 0 || seq_lens[b] > Nmax)
            return ORACLE_ERR_ARG;
    const int G = Hq / Hkv;
    int rc_all = ORACLE_OK;
#pragma omp parallel for schedule(dynamic, 1)
    for (int bg = 0; bg < B * Hkv; ++bg) {
        int b = bg / Hkv, g = bg % Hkv;
        const uint16_t **qg = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        const uint16_t **Kg = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        const uint16_t **Vg = (const uint16_t **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        double **og = (double **)malloc(sizeof(void *) * (size_t)(L > 0 ? L : 1));
        int32_t *state = (int32_t *)malloc(sizeof(int32_t) * (size_t)(k > 0 ? k : 1));
        int rc = ORACLE_ERR_NOMEM;
        if (qg && Kg && Vg && og && state) {
            for (int l = 0; l < L; ++l) {
                qg[l] = q[l] + ((int64_t)b * Hq + (int64_t)g * G) * d;
                Kg[l] = K[l] + ((int64_t)b * Hkv + g) * (int64_t)Nmax * d;
                Vg[l] = V[l] + ((int64_t)b * Hkv + g) * (int64_t)Nmax * d;
                og[l] = out[l] + ((int64_t)b * Hq + (int64_t)g * G) * d;
            }
            for (int j = 0; j < k; ++j)
                state[j] = -1;
            int valid = 0;
            rc = oracle_decode_group(L, modes, G, d, seq_lens[b], k, scale, qg, Kg, Vg, state,
                                     &valid, og, NULL);
            if (idx_final && k > 0)
                memcpy(idx_final + (int64_t)bg * k, state, sizeof(int32_t) * (size_t)k);
        }
        free(qg);
        free(Kg);
        free(Vg);
        free(og);
        free(state);
        if (rc) {
#pragma omp critical
            rc_all = rc;
        }
    }
    return rc_all;
}

/*
 * Coverage budget (Token Sparse Attention page, §2 "Dynamic Token Coverage":
 * rank tokens by importance and prune the least important while the pruned
 * attention mass stays within tau): the smallest k such that the k highest
 * scores (ties: lower position first) hold at least 1 - tau of softmax(s)
 * over s[0..n), capped at k_max; n if the sum never reaches it (rounding).
 * Returns k, or -1 if memory runs out.
 */
int oracle_coverage_count(const double *s, int n, double tau, int k_max)
{
    if (n <= 0 || k_max <= 0)
        return 0;
    double *p = (double *)malloc(sizeof(double) * (size_t)n);
    scored_pos *v = (scored_pos *)malloc(sizeof(scored_pos) * (size_t)n);
    if (!p || !v) {
        free(p);
        free(v);
        return -1;
    }
    oracle_softmax(s, n, p);
    for (int t = 0; t < n; ++t) {
        v[t].s = s[t];
        v[t].pos = t;
    }
    qsort(v, (size_t)n, sizeof(scored_pos), by_score_desc_pos_asc);
    double mass = 0.0;
    int k = n;
    for (int j = 0; j < n; ++j) {
        mass += p[v[j].pos];
        if (mass >= 1.0 - tau) {
            k = j + 1;
            break;
        }
    }
#if ORACLE_MUTANT == 14
    if (k > 1)
        k -= 1; /* mutant: stops one token before the coverage is reached */
#endif
    free(p);
    free(v);
    return k < k_max ? k : k_max;
}

/*
 * Overlap of two token sets (review §三 "Token selection layer sensitivity",
 * Figure 4(a): how many of the most attended tokens two layers share):
 * the number of positions that occur in both a[0..k) and b[0..k), entries
 * < 0 (padding) ignored.  Every pair is compared: no order is assumed.
 */
int oracle_index_overlap(const int32_t *a, const int32_t *b, int k)
{
    int count = 0;
    for (int i = 0; i < k; ++i) {
#if ORACLE_MUTANT == 13
        /* mutant: padding entries are not skipped (a -1 matches a -1) */
#else
        if (a[i] < 0)
            continue;
#endif
        for (int j = 0; j < k; ++j)
            if (b[j] == a[i]) {
                ++count;
                break;
            }
    }
    return count;
}

/* Which mutant this build carries (0 = the oracle itself). */
int oracle_mutant_id(void) { return ORACLE_MUTANT; }

/* Number of OpenMP threads a parallel region would use (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int oracle_num_threads(void) { return omp_get_max_threads(); }
/* Threads for later parallel regions (n >= 1). */
void oracle_set_threads(int n) { omp_set_num_threads(n > 0 ? n : 1); }
#else
int oracle_num_threads(void) { return 1; }
void oracle_set_threads(int n) { (void)n; }
#endif
