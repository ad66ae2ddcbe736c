/*
 * Plain CPU oracle for the draft-head argmax path.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the smoke check and the benchmark's CPU
 * baseline do.  It shares no code, header, table or constant with the CUDA
 * library: every format decode below is written out here from the format's
 * own definition.
 *
 * What it computes (the plain definition of the method; the fast path must
 * reach exactly this, up to the order of the fp32 additions):
 *
 *   logit[m][n] = sum_{k=0..K-1} W[n][k] * h[m][k]
 *       fp32 accumulation in ascending k, one rounding per add, no fused
 *       multiply-add (the file is compiled with -ffp-contract=off).  This is
 *       the draft head's vocabulary projection: a hidden state of width K
 *       against every row of the head ("Shortlist MTP", section "What I was
 *       testing": width 2,560 against 248,320 rows, one row per draft step,
 *       three per MTP2 verify step).
 *   full_id(n) = d2t[n] (identity when d2t is NULL): the map from a
 *       shortlist index to a full-vocabulary id ("Masked MTP drafts": the
 *       d2t index mapping of EAGLE-3 reused for a frequency-ranked subset).
 *   argmax / top-k over n by (logit descending, full_id ascending); a NaN
 *       ranks below every number.  The tie rule (lowest full-vocabulary id
 *       wins) is not on the pages; it is the reading this project adopts.
 *   NVFP4 head: w = float(e2m1(q) * e4m3(s)) * g, one fp32 rounding for the
 *       global scale g, then the same dot product ("Masked MTP drafts":
 *       requantizing the trimmed head to NVFP4).  The layout (row-major
 *       codes, low nibble = even k, one e4m3 scale per 16 consecutive k of a
 *       row, one fp32 tensor scale) is the reading this project adopts.
 *   candidate scores: logit[m][j] = the same dot for head row
 *       ids[m][j] - id_base, NaN for an id outside the head's rows ("Masked
 *       MTP drafts", section "Update (November 2026)": a drafter's candidates
 *       scored through the target's own LM head, bf16 or NVFP4).
 *   FP8 head: w = float(e4m3(q)) * g, one fp32 rounding for the tensor
 *       scale g, then the same dot product ("[DGX Spark] Qwen3.8-Flash-Next
 *       on two DGX Sparks", section "The costs: a 69% smaller KV pool and
 *       FP8 GDN weights": weights read as FP8 E4M3 halve the bytes; "Masked
 *       MTP drafts": a drafter shipping an FP8 head).  The layout (row-major
 *       codes, one byte per weight, one fp32 tensor scale) is the reading
 *       this project adopts.
 *   requantization of a bf16 head ("Masked MTP drafts": the trimmed head
 *       requantized to NVFP4 at load, at no measured acceptance cost; the
 *       pages give no recipe, so the one below is the plainest reading, in
 *       fp32 with each operation rounded once, in the order written):
 *       NVFP4: g = amax / (6 * 448); per 16-weight block s = RNE_e4m3(
 *       amax_b / (6 g)); code = RNE_e2m1(w / (s g)), all codes 0 when s is 0.
 *       FP8: g = amax / 448; code = RNE_e4m3(w / g).  RNE: the nearest value
 *       of the format, ties to the code with an even last mantissa bit,
 *       magnitudes above the largest value saturating to it; the sign bit
 *       is the sign of the quotient (so -0 keeps its sign).
 *   trim check: W_trim[i] == W_full[ranks[i]] byte for byte, d2t[i] ==
 *       ranks[i] ("Masked MTP drafts": a ranks list next to the model, the
 *       head weight trimmed at load).
 *   ranks builder: histogram of a token stream, top-N by (count desc, id
 *       asc) after a forced id set, set union ("Shortlist MTP", section
 *       "Building the 16k shortlist"; "[DGX Spark] Qwen3.8-Flash-Next on two
 *       DGX Sparks", section "Build the draft vocabulary from your own
 *       text").
 *
 * Threads split the rows n only; every logit is computed by one thread in
 * the same order, so results do not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#include <unistd.h>

#include "oracle.h"

/* ------------------------------------------------------------------ */
/* Format decodes, from the format definitions.                        */
/* ------------------------------------------------------------------ */

/* bfloat16 is the upper half of an IEEE binary32: the value of the 16 bits b
 * is the binary32 whose bit pattern is b followed by sixteen zero bits. */
float oracle_bf16_to_f32(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* E2M1 (4-bit float): bit 3 sign, bits 2..1 exponent (bias 1), bit 0
 * mantissa.  Exponent field 0 is subnormal: value = m * 2^(1-1) * 0.5.
 * Otherwise value = 2^(e-1) * (1 + m/2).  No infinities or NaNs. */
float oracle_e2m1(uint8_t code)
{
    int s = (code >> 3) & 1;
    int e = (code >> 1) & 3;
    int m = code & 1;
    double v;
    if (e == 0)
        v = 0.5 * m;
    else
        v = ldexp(1.0 + 0.5 * m, e - 1);
    return (float)(s ? -v : v);
}

/* E4M3 (8-bit float, the "fn" variant): bit 7 sign, bits 6..3 exponent
 * (bias 7), bits 2..0 mantissa.  Exponent field 0 is subnormal: value =
 * 2^-6 * m/8.  Exponent 15 with mantissa 7 is NaN; there are no infinities,
 * so the largest finite magnitude is 2^8 * 1.75 = 448. */
float oracle_e4m3(uint8_t byte)
{
    int s = (byte >> 7) & 1;
    int e = (byte >> 3) & 15;
    int m = byte & 7;
    double v;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return (float)(s ? -v : v);
}

/* One dequantized NVFP4 weight: the product of the 4-bit value and its
 * block scale is exact in binary32 (at most 2 x 4 significant bits), then
 * the tensor scale is applied with one binary32 rounding. */
float oracle_nvfp4_weight(const uint8_t *q, const uint8_t *scales, float g,
                          int64_t K, int64_t n, int64_t k)
{
    uint8_t byte = q[n * (K / 2) + k / 2];
    uint8_t code = (k & 1) ? (uint8_t)(byte >> 4) : (uint8_t)(byte & 15);
    float prod = oracle_e2m1(code) * oracle_e4m3(scales[n * (K / 16) + k / 16]);
    return prod * g;
}

/* ------------------------------------------------------------------ */
/* Logits: plain fp32 dot products, rows split over threads.           */
/* ------------------------------------------------------------------ */

typedef struct {
    int kind; /* 0 = bf16, 1 = nvfp4, 2 = fp8 */
    const uint16_t *w_bf16;
    const uint8_t *q;
    const uint8_t *scales;
    float g;
    int64_t N, K, M;
    const uint16_t *h;
    float *logits;
    int64_t n_begin, n_end;
} logit_job;

/* One logit: head row n against hidden row hm, ascending k in fp32. */
static float row_dot(const logit_job *j, int64_t n, const uint16_t *hm)
{
    float acc = 0.0f;
    if (j->kind == 0) {
        const uint16_t *wn = j->w_bf16 + n * j->K;
        for (int64_t k = 0; k < j->K; ++k) {
            float prod = oracle_bf16_to_f32(wn[k]) * oracle_bf16_to_f32(hm[k]);
            acc = acc + prod;
        }
    } else if (j->kind == 1) {
        for (int64_t k = 0; k < j->K; ++k) {
            float w = oracle_nvfp4_weight(j->q, j->scales, j->g, j->K, n, k);
            float prod = w * oracle_bf16_to_f32(hm[k]);
            acc = acc + prod;
        }
    } else {
        const uint8_t *qn = j->q + n * j->K;
        for (int64_t k = 0; k < j->K; ++k) {
            float w = oracle_e4m3(qn[k]) * j->g;
            float prod = w * oracle_bf16_to_f32(hm[k]);
            acc = acc + prod;
        }
    }
    return acc;
}

static void *logit_worker(void *arg)
{
    logit_job *j = (logit_job *)arg;
    for (int64_t m = 0; m < j->M; ++m) {
        const uint16_t *hm = j->h + m * j->K;
        for (int64_t n = j->n_begin; n < j->n_end; ++n)
            j->logits[m * j->N + n] = row_dot(j, n, hm);
    }
    return NULL;
}

int oracle_num_cores(void)
{
    long c = sysconf(_SC_NPROCESSORS_ONLN);
    return c > 0 ? (int)c : 1;
}

static int run_logits(logit_job base, int nthreads)
{
    if (nthreads <= 0)
        nthreads = oracle_num_cores();
    if (nthreads > base.N)
        nthreads = base.N > 0 ? (int)base.N : 1;
    if (nthreads == 1) {
        base.n_begin = 0;
        base.n_end = base.N;
        logit_worker(&base);
        return 1;
    }
    pthread_t *tid = (pthread_t *)malloc(sizeof(pthread_t) * (size_t)nthreads);
    logit_job *jobs = (logit_job *)malloc(sizeof(logit_job) * (size_t)nthreads);
    int started = 0;
    for (int t = 0; t < nthreads; ++t) {
        jobs[t] = base;
        jobs[t].n_begin = base.N * t / nthreads;
        jobs[t].n_end = base.N * (t + 1) / nthreads;
        if (pthread_create(&tid[t], NULL, logit_worker, &jobs[t]) != 0) {
            logit_worker(&jobs[t]); /* run inline if a thread cannot start */
            tid[t] = 0;
        } else {
            started++;
        }
    }
    for (int t = 0; t < nthreads; ++t)
        if (tid[t])
            pthread_join(tid[t], NULL);
    free(tid);
    free(jobs);
    return started > 0 ? nthreads : 1;
}

int oracle_logits_bf16(const uint16_t *w, int64_t N, int64_t K, const uint16_t *h,
                       int64_t M, float *logits, int nthreads)
{
    logit_job j;
    memset(&j, 0, sizeof j);
    j.kind = 0;
    j.w_bf16 = w;
    j.N = N;
    j.K = K;
    j.M = M;
    j.h = h;
    j.logits = logits;
    return run_logits(j, nthreads);
}

int oracle_logits_nvfp4(const uint8_t *q, const uint8_t *scales, float g, int64_t N,
                        int64_t K, const uint16_t *h, int64_t M, float *logits,
                        int nthreads)
{
    logit_job j;
    memset(&j, 0, sizeof j);
    j.kind = 1;
    j.q = q;
    j.scales = scales;
    j.g = g;
    j.N = N;
    j.K = K;
    j.M = M;
    j.h = h;
    j.logits = logits;
    return run_logits(j, nthreads);
}

int oracle_logits_fp8(const uint8_t *q, float g, int64_t N, int64_t K, const uint16_t *h,
                      int64_t M, float *logits, int nthreads)
{
    logit_job j;
    memset(&j, 0, sizeof j);
    j.kind = 2;
    j.q = q;
    j.g = g;
    j.N = N;
    j.K = K;
    j.M = M;
    j.h = h;
    j.logits = logits;
    return run_logits(j, nthreads);
}

/* ------------------------------------------------------------------ */
/* Requantization: the nearest code by search over the format's values. */
/* ------------------------------------------------------------------ */

/* Non-negative x -> the code among 0 .. ncodes - 1 (values increasing with
 * the code; vals[c] its value) whose value is nearest, ties to the even
 * code; above the largest value that value is the nearest, which is the
 * saturation.  Bisection finds the neighbours lo <= x < lo + 1. */
static uint8_t nearest_code(float x, const float *vals, int ncodes)
{
    if (x >= vals[ncodes - 1])
        return (uint8_t)(ncodes - 1);
    int lo = 0, hi = ncodes - 1; /* vals[lo] <= x < vals[hi] */
    while (hi - lo > 1) {
        int mid = (lo + hi) / 2;
        if (vals[mid] <= x)
            lo = mid;
        else
            hi = mid;
    }
    double dlo = (double)x - (double)vals[lo], dhi = (double)vals[hi] - (double)x;
    if (dlo < dhi)
        return (uint8_t)lo;
    if (dhi < dlo)
        return (uint8_t)hi;
    return (uint8_t)((lo & 1) == 0 ? lo : hi); /* tie: the even code */
}

/* The non-negative values of each format, by code, from the decoders above. */
static float g_e2m1_vals[8], g_e4m3_vals[127];
static pthread_once_t g_vals_once = PTHREAD_ONCE_INIT;
static void fill_vals(void)
{
    for (int c = 0; c < 8; ++c)
        g_e2m1_vals[c] = oracle_e2m1((uint8_t)c);
    for (int c = 0; c < 127; ++c)
        g_e4m3_vals[c] = oracle_e4m3((uint8_t)c);
}

static uint8_t rne_e2m1(float x) /* 4-bit code, sign in bit 3 */
{
    pthread_once(&g_vals_once, fill_vals);
    uint8_t c = nearest_code(fabsf(x), g_e2m1_vals, 8);
    return signbit(x) ? (uint8_t)(c | 8) : c;
}

static uint8_t rne_e4m3(float x) /* sign in bit 7; 0x7E = 448 is the largest */
{
    pthread_once(&g_vals_once, fill_vals);
    uint8_t c = nearest_code(fabsf(x), g_e4m3_vals, 127);
    return signbit(x) ? (uint8_t)(c | 0x80) : c;
}

static float abs_max_bf16(const uint16_t *w, int64_t n)
{
    float m = 0.0f;
    for (int64_t i = 0; i < n; ++i) {
        float a = fabsf(oracle_bf16_to_f32(w[i]));
        if (a > m)
            m = a;
    }
    return m;
}

float oracle_quantize_nvfp4(const uint16_t *w, int64_t N, int64_t K, uint8_t *q,
                            uint8_t *scales)
{
    float amax = abs_max_bf16(w, N * K);
    float g = amax > 0.0f ? amax / 2688.0f : 1.0f; /* 2688 = 6 * 448 */
    float six_g = 6.0f * g;
    for (int64_t n = 0; n < N; ++n) {
        for (int64_t b = 0; b < K / 16; ++b) {
            const uint16_t *wb = w + n * K + b * 16;
            float amax_b = abs_max_bf16(wb, 16);
            uint8_t sb = rne_e4m3(amax_b / six_g);
            scales[n * (K / 16) + b] = sb;
            float sg = oracle_e4m3(sb) * g;
            for (int j = 0; j < 16; j += 2) {
                uint8_t lo = 0, hi = 0;
                if (oracle_e4m3(sb) != 0.0f) {
                    lo = rne_e2m1(oracle_bf16_to_f32(wb[j]) / sg);
                    hi = rne_e2m1(oracle_bf16_to_f32(wb[j + 1]) / sg);
                }
                q[n * (K / 2) + (b * 16 + j) / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
    return g;
}

float oracle_quantize_fp8(const uint16_t *w, int64_t N, int64_t K, uint8_t *q)
{
    float amax = abs_max_bf16(w, N * K);
    float g = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int64_t i = 0; i < N * K; ++i)
        q[i] = rne_e4m3(oracle_bf16_to_f32(w[i]) / g);
    return g;
}

/* ------------------------------------------------------------------ */
/* Candidate scores: the dot of the head row each id names.            */
/* ------------------------------------------------------------------ */

static void score_ids(const logit_job *j, int64_t id_base, const int32_t *ids, int64_t c,
                      float *out)
{
    for (int64_t m = 0; m < j->M; ++m) {
        const uint16_t *hm = j->h + m * j->K;
        for (int64_t t = 0; t < c; ++t) {
            int64_t n = (int64_t)ids[m * c + t] - id_base;
            out[m * c + t] = (n >= 0 && n < j->N) ? row_dot(j, n, hm) : NAN;
        }
    }
}

void oracle_score_ids_bf16(const uint16_t *w, int64_t N, int64_t K, int64_t id_base,
                           const uint16_t *h, int64_t M, const int32_t *ids, int64_t c,
                           float *out)
{
    logit_job j;
    memset(&j, 0, sizeof j);
    j.kind = 0;
    j.w_bf16 = w;
    j.N = N;
    j.K = K;
    j.M = M;
    j.h = h;
    score_ids(&j, id_base, ids, c, out);
}

void oracle_score_ids_nvfp4(const uint8_t *q, const uint8_t *scales, float g, int64_t N,
                            int64_t K, int64_t id_base, const uint16_t *h, int64_t M,
                            const int32_t *ids, int64_t c, float *out)
{
    logit_job j;
    memset(&j, 0, sizeof j);
    j.kind = 1;
    j.q = q;
    j.scales = scales;
    j.g = g;
    j.N = N;
    j.K = K;
    j.M = M;
    j.h = h;
    score_ids(&j, id_base, ids, c, out);
}

void oracle_score_ids_fp8(const uint8_t *q, float g, int64_t N, int64_t K, int64_t id_base,
                          const uint16_t *h, int64_t M, const int32_t *ids, int64_t c,
                          float *out)
{
    logit_job j;
    memset(&j, 0, sizeof j);
    j.kind = 2;
    j.q = q;
    j.g = g;
    j.N = N;
    j.K = K;
    j.M = M;
    j.h = h;
    score_ids(&j, id_base, ids, c, out);
}

/* ------------------------------------------------------------------ */
/* Argmax / top-k with the tie rule.                                   */
/* ------------------------------------------------------------------ */

/* Does candidate a (logit la, id ia) rank strictly above b?  A NaN ranks
 * below every number; -0 and +0 compare equal, so they fall to the id. */
static int ranks_above(float la, int64_t ia, float lb, int64_t ib)
{
    int na = isnan(la), nb = isnan(lb);
    if (na != nb)
        return nb; /* the number beats the NaN */
    if (!na && la != lb)
        return la > lb;
    return ia < ib;
}

/* For each m: the k best rows n (distinct n) by (logit desc, full id asc),
 * found by k plain scans over all N rows.  Writes full ids, logits and the
 * row index n of each pick.  k may exceed N only if N >= 1; missing slots
 * get id -1. */
void oracle_topk(const float *logits, int64_t N, int64_t M, const int32_t *d2t,
                 int k, int32_t *ids, float *vals, int64_t *rows)
{
    unsigned char *taken = (unsigned char *)calloc((size_t)(N > 0 ? N : 1), 1);
    for (int64_t m = 0; m < M; ++m) {
        memset(taken, 0, (size_t)(N > 0 ? N : 1));
        const float *lm = logits + m * N;
        for (int j = 0; j < k; ++j) {
            int64_t best = -1;
            for (int64_t n = 0; n < N; ++n) {
                if (taken[n])
                    continue;
                if (best < 0) {
                    best = n;
                    continue;
                }
                int64_t idn = d2t ? d2t[n] : n;
                int64_t idb = d2t ? d2t[best] : best;
                if (ranks_above(lm[n], idn, lm[best], idb))
                    best = n;
            }
            int64_t slot = m * k + j;
            if (best < 0) {
                ids[slot] = -1;
                vals[slot] = NAN;
                if (rows)
                    rows[slot] = -1;
            } else {
                taken[best] = 1;
                ids[slot] = (int32_t)(d2t ? d2t[best] : best);
                vals[slot] = lm[best];
                if (rows)
                    rows[slot] = best;
            }
        }
    }
    free(taken);
}

/* ------------------------------------------------------------------ */
/* Trim check.                                                          */
/* ------------------------------------------------------------------ */

/* Number of positions i where W_trim row i differs from W_full row ranks[i]
 * (byte comparison of row_bytes bytes) or d2t[i] != ranks[i].  Returns -1 if
 * a rank lies outside [0, V). */
int64_t oracle_check_trim(const uint8_t *w_full, int64_t V, int64_t row_bytes,
                          const int32_t *ranks, int64_t n, const uint8_t *w_trim,
                          const int32_t *d2t)
{
    int64_t bad = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (ranks[i] < 0 || ranks[i] >= V)
            return -1;
        if (memcmp(w_trim + i * row_bytes, w_full + (int64_t)ranks[i] * row_bytes,
                   (size_t)row_bytes) != 0 ||
            (d2t && d2t[i] != ranks[i]))
            bad++;
    }
    return bad;
}

/* ------------------------------------------------------------------ */
/* Ranks builder.                                                       */
/* ------------------------------------------------------------------ */

/* counts[t] += 1 for every token t.  Returns 0, or -1 (nothing counted) if
 * any token lies outside [0, V). */
int oracle_histogram(const int32_t *tokens, int64_t n, int64_t V, int64_t *counts)
{
    for (int64_t i = 0; i < n; ++i)
        if (tokens[i] < 0 || tokens[i] >= V)
            return -1;
    for (int64_t i = 0; i < n; ++i)
        counts[tokens[i]] += 1;
    return 0;
}

/* Rank order: higher count first, then lower id. */
static const int64_t *g_counts_for_sort;
static int by_rank(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    int64_t cx = g_counts_for_sort[x], cy = g_counts_for_sort[y];
    if (cx != cy)
        return cx > cy ? -1 : 1;
    return (x > y) - (x < y);
}
static int by_id(const void *a, const void *b)
{
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* The shortlist: the distinct forced ids first, in rank order, then every
 * other id in rank order, cut at N entries; sorted ascending if asked.
 * Returns the number of ids written (min(N, V)), or -1 on a bad argument
 * (forced id outside [0, V), N < 0).  Not thread-safe (qsort comparator
 * state). */
int64_t oracle_build_ranks(const int64_t *counts, int64_t V, const int32_t *forced,
                           int64_t n_forced, int64_t N, int sorted, int32_t *out)
{
    if (N < 0 || V < 0)
        return -1;
    for (int64_t i = 0; i < n_forced; ++i)
        if (forced[i] < 0 || forced[i] >= V)
            return -1;
    unsigned char *is_forced = (unsigned char *)calloc((size_t)(V > 0 ? V : 1), 1);
    int32_t *f = (int32_t *)malloc(sizeof(int32_t) * (size_t)(n_forced > 0 ? n_forced : 1));
    int32_t *rest = (int32_t *)malloc(sizeof(int32_t) * (size_t)(V > 0 ? V : 1));
    int64_t nf = 0, nr = 0;
    for (int64_t i = 0; i < n_forced; ++i)
        if (!is_forced[forced[i]]) {
            is_forced[forced[i]] = 1;
            f[nf++] = forced[i];
        }
    for (int64_t t = 0; t < V; ++t)
        if (!is_forced[t])
            rest[nr++] = (int32_t)t;
    g_counts_for_sort = counts;
    qsort(f, (size_t)nf, sizeof(int32_t), by_rank);
    qsort(rest, (size_t)nr, sizeof(int32_t), by_rank);
    int64_t total = N < V ? N : V, w = 0;
    for (int64_t i = 0; i < nf && w < total; ++i)
        out[w++] = f[i];
    for (int64_t i = 0; i < nr && w < total; ++i)
        out[w++] = rest[i];
    if (sorted)
        qsort(out, (size_t)w, sizeof(int32_t), by_id);
    free(is_forced);
    free(f);
    free(rest);
    return w;
}

/* Sorted set union of two id lists (each taken as a set).  out must hold
 * na + nb entries.  Returns the union's size. */
int64_t oracle_union_sorted(const int32_t *a, int64_t na, const int32_t *b, int64_t nb,
                            int32_t *out)
{
    int64_t n = 0;
    for (int64_t i = 0; i < na; ++i)
        out[n++] = a[i];
    for (int64_t i = 0; i < nb; ++i)
        out[n++] = b[i];
    qsort(out, (size_t)n, sizeof(int32_t), by_id);
    int64_t w = 0;
    for (int64_t i = 0; i < n; ++i)
        if (w == 0 || out[w - 1] != out[i])
            out[w++] = out[i];
    return w;
}
