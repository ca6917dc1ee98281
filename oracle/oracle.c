/*
 * fp64 CPU oracle for the exact attention forward pass.
 *
 * TEST INFRASTRUCTURE. Only the test suite, the package smoke check
 * (__graft_entry__.smoke) and the benchmark's CPU-baseline / reference leg may
 * load this library. It shares no code, header, table or helper with the CUDA
 * path, and nothing in the product path calls it.
 *
 * What it computes is the plain, materialising definition of attention:
 *   - "Warmup Guide — Inference Optimization at Depth", Chapter 1: S = Q K^T
 *     is formed in full, P = softmax(S), O = P V;
 *   - same page, Chapter 2: the safe softmax, m = max_j x_j, then
 *     e^{x_i - m} / sum_j e^{x_j - m} — two reduction passes, then normalise;
 *   - same page, Chapter 4: scores are Q_i K_j^T / sqrt(d); the causal mask
 *     hides keys above the diagonal; the per-row statistics m and l are what
 *     the tiled forward keeps, reported here as lse = m + ln l.
 * FlashAttention reaches exactly this result up to rounding order
 * ("FlashAttention, speculative decoding, quantisation and parallelism",
 * Mechanics: "exact, not approximate"), so the definition is the oracle.
 *
 * Readings taken where the pages are silent:
 *   - scale: a caller argument (page 1's pseudocode omits 1/sqrt(d), page 2's
 *     includes it); passed as fp32 and promoted to double here;
 *   - causal alignment when Sq != Sk: bottom-right, key j visible to query i
 *     iff j <= i + (Sk - Sq) (the verify step appends Sq queries after a KV
 *     cache, so query i sees keys [0, Sk - Sq + i]);
 *   - lse: natural log, in units of the scaled logits, lse = m + ln(l);
 *   - a row with no visible key (causal with Sk < Sq only): o = 0, lse = -inf;
 *   - inputs are bf16 bit patterns, decoded exactly to double; every
 *     operation after that is fp64.
 *
 * Besides the definition, the file holds the two online (one-pass, block-wise)
 * forms the pages print and the split-KV combine, each written from its own
 * passage, so that tests can pin "online == two-pass" and "split == unsplit":
 *   - online form 1: page 1, Mechanics pseudocode (running_max, running_sum,
 *     accumulator; the block's row sum is taken under the new max);
 *   - online form 2: "Warmup Guide", Chapter 3 (combine the block-local max
 *     and exp-sum into the running pair; same correction for O);
 *   - split-KV: "Lecture 06 — Making Decode Fast", section 5, Flash-Decoding
 *     (split keys/values, then a small final combine). The pages give no
 *     combine formula; the reading is the log-sum-exp weighting that follows
 *     from Chapter 3's update applied to whole chunks.
 *
 * All entry points return 0 on success and a negative value on a bad argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Exact bf16 -> double: a bf16 value is the top 16 bits of an fp32 value. */
static double bf16_to_double(uint16_t x)
{
    uint32_t u = ((uint32_t)x) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Number of keys query row i may see. */
static int64_t visible_keys(int64_t i, int64_t Sq, int64_t Sk, int causal)
{
    if (!causal)
        return Sk;
    int64_t n = i + (Sk - Sq) + 1;
    if (n < 0)
        n = 0;
    if (n > Sk)
        n = Sk;
    return n;
}

static int check_args(const void *q, const void *k, const void *v, int64_t B, int64_t H,
                      int64_t Sq, int64_t Sk, int64_t d)
{
    if (!q || !k || !v)
        return -1;
    if (B <= 0 || H <= 0 || Sq <= 0 || Sk <= 0 || d <= 0)
        return -2;
    return 0;
}

/* s[j] = scale * (q_i . k_j) for j < n: one materialised row of S (Chapters 1 and 4). */
static void score_row(const uint16_t *qi, const uint16_t *kbh, int64_t n, int64_t d, double scale,
                      double *s)
{
    for (int64_t j = 0; j < n; ++j) {
        const uint16_t *kj = kbh + j * d;
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t)
            dot += bf16_to_double(qi[t]) * bf16_to_double(kj[t]);
        s[j] = scale * dot;
    }
}

/*
 * The definition for one row over keys [j0, j1): materialise s, two-pass safe
 * softmax (max, then sum), normalise to p, then o = sum_j p_j v_j.
 * Writes o[d] and *lse; an empty range gives o = 0, lse = -inf.
 * s is scratch of at least (j1 - j0) doubles.
 */
static void definition_row(const uint16_t *qi, const uint16_t *kbh, const uint16_t *vbh, int64_t j0,
                           int64_t j1, int64_t d, double scale, double *s, double *o, double *lse)
{
    int64_t n = j1 - j0;
    for (int64_t t = 0; t < d; ++t)
        o[t] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return;
    }
    score_row(qi, kbh + j0 * d, n, d, scale, s);
    /* pass 1: row max */
    double m = -INFINITY;
    for (int64_t j = 0; j < n; ++j)
        if (s[j] > m)
            m = s[j];
    /* pass 2: sum of exponentials under the max */
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j)
        l += exp(s[j] - m);
    /* normalise: p_j = e^{s_j - m} / l (kept in s) */
    for (int64_t j = 0; j < n; ++j)
        s[j] = exp(s[j] - m) / l;
    /* o = P V */
    for (int64_t j = 0; j < n; ++j) {
        const uint16_t *vj = vbh + (j0 + j) * d;
        for (int64_t t = 0; t < d; ++t)
            o[t] += s[j] * bf16_to_double(vj[t]);
    }
    *lse = m + log(l);
}

static int row_in_range(const int64_t *r, int64_t B, int64_t H, int64_t Sq)
{
    return r[0] >= 0 && r[0] < B && r[1] >= 0 && r[1] < H && r[2] >= 0 && r[2] < Sq;
}

static void set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0)
        omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

/* Threads an OpenMP parallel region would use right now (1 without OpenMP). */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Materialising two-pass definition for a list of rows.
 * q: bf16 bits [B,H,Sq,d]; k, v: bf16 bits [B,H,Sk,d]; rows: n triples (b,h,i).
 * o: n*d doubles; lse: n doubles. nthreads <= 0 keeps the OpenMP default.
 */
int oracle_attention_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                          int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal, float scale,
                          const int64_t *rows, int64_t n, double *o, double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (n < 0 || (n > 0 && (!rows || !o || !lse)))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (!row_in_range(rows + 3 * r, B, H, Sq))
            return -3;
    set_threads(nthreads);
    const double sc = (double)scale;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Sk);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            if (!s)
                continue;
            int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            const uint16_t *qi = q + ((b * H + h) * Sq + i) * d;
            const uint16_t *kbh = k + (b * H + h) * Sk * d;
            const uint16_t *vbh = v + (b * H + h) * Sk * d;
            int64_t nv = visible_keys(i, Sq, Sk, causal);
            definition_row(qi, kbh, vbh, 0, nv, d, sc, s, o + r * d, lse + r);
        }
        free(s);
    }
    return failed ? -4 : 0;
}

/* Every row: o [B,H,Sq,d], lse [B,H,Sq] (doubles). */
int oracle_attention(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B, int64_t H,
                     int64_t Sq, int64_t Sk, int64_t d, int causal, float scale, double *o,
                     double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (!o || !lse)
        return -1;
    int64_t n = B * H * Sq;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * 3 * (size_t)n);
    if (!rows)
        return -4;
    for (int64_t b = 0, r = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < Sq; ++i, ++r) {
                rows[3 * r] = b;
                rows[3 * r + 1] = h;
                rows[3 * r + 2] = i;
            }
    rc = oracle_attention_rows(q, k, v, B, H, Sq, Sk, d, causal, scale, rows, n, o, lse, nthreads);
    free(rows);
    return rc;
}

/*
 * The softmax row P_i (Chapter 2's definition) over all Sk keys: visible keys
 * get their probability, hidden keys 0. p: Sk doubles.
 */
int oracle_probs_row(const uint16_t *q, const uint16_t *k, int64_t B, int64_t H, int64_t Sq,
                     int64_t Sk, int64_t d, int causal, float scale, int64_t b, int64_t h,
                     int64_t i, double *p)
{
    int rc = check_args(q, k, k, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    int64_t r[3] = {b, h, i};
    if (!p || !row_in_range(r, B, H, Sq))
        return -3;
    int64_t nv = visible_keys(i, Sq, Sk, causal);
    for (int64_t j = 0; j < Sk; ++j)
        p[j] = 0.0;
    if (nv == 0)
        return 0;
    const uint16_t *qi = q + ((b * H + h) * Sq + i) * d;
    const uint16_t *kbh = k + (b * H + h) * Sk * d;
    score_row(qi, kbh, nv, d, (double)scale, p);
    double m = -INFINITY;
    for (int64_t j = 0; j < nv; ++j)
        if (p[j] > m)
            m = p[j];
    double l = 0.0;
    for (int64_t j = 0; j < nv; ++j)
        l += exp(p[j] - m);
    for (int64_t j = 0; j < nv; ++j)
        p[j] = exp(p[j] - m) / l;
    return 0;
}

/*
 * Online softmax, form 1 — page 1's pseudocode, over blocks of `block` visible
 * keys: new_max = max(running_max, rowmax(S_blk)); correction =
 * e^{running_max - new_max}; P = e^{S_blk - new_max}; accumulator =
 * accumulator * correction + P V_blk; running_sum = running_sum * correction +
 * rowsum(P); at the end O = accumulator / running_sum.
 */
static void online_form1_row(const uint16_t *qi, const uint16_t *kbh, const uint16_t *vbh,
                             int64_t nv, int64_t d, double scale, int64_t block, double *s,
                             double *acc, double *o, double *lse)
{
    double running_max = -INFINITY, running_sum = 0.0;
    for (int64_t t = 0; t < d; ++t)
        acc[t] = 0.0;
    for (int64_t j0 = 0; j0 < nv; j0 += block) {
        int64_t nb = (nv - j0 < block) ? nv - j0 : block;
        score_row(qi, kbh + j0 * d, nb, d, scale, s);
        double bmax = -INFINITY;
        for (int64_t j = 0; j < nb; ++j)
            if (s[j] > bmax)
                bmax = s[j];
        double new_max = running_max > bmax ? running_max : bmax;
        double correction = exp(running_max - new_max);
        double rowsum = 0.0;
        for (int64_t t = 0; t < d; ++t)
            acc[t] *= correction;
        for (int64_t j = 0; j < nb; ++j) {
            double pj = exp(s[j] - new_max);
            rowsum += pj;
            const uint16_t *vj = vbh + (j0 + j) * d;
            for (int64_t t = 0; t < d; ++t)
                acc[t] += pj * bf16_to_double(vj[t]);
        }
        running_sum = running_sum * correction + rowsum;
        running_max = new_max;
    }
    if (nv == 0) {
        for (int64_t t = 0; t < d; ++t)
            o[t] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int64_t t = 0; t < d; ++t)
        o[t] = acc[t] / running_sum;
    *lse = running_max + log(running_sum);
}

/*
 * Online softmax, form 2 — "Warmup Guide", Chapter 3: each block b gives its
 * local max m~_b and local exp-sum l~_b (and local unnormalised output
 * o~_b = sum e^{s - m~_b} v); then m_new = max(m, m~_b),
 * l_new = l e^{m - m_new} + l~_b e^{m~_b - m_new}, and O is corrected the same
 * way; divide by l once at the end.
 */
static void online_form2_row(const uint16_t *qi, const uint16_t *kbh, const uint16_t *vbh,
                             int64_t nv, int64_t d, double scale, int64_t block, double *s,
                             double *acc, double *blk, double *o, double *lse)
{
    double m = -INFINITY, l = 0.0;
    for (int64_t t = 0; t < d; ++t)
        acc[t] = 0.0;
    for (int64_t j0 = 0; j0 < nv; j0 += block) {
        int64_t nb = (nv - j0 < block) ? nv - j0 : block;
        score_row(qi, kbh + j0 * d, nb, d, scale, s);
        double mb = -INFINITY;
        for (int64_t j = 0; j < nb; ++j)
            if (s[j] > mb)
                mb = s[j];
        double lb = 0.0;
        for (int64_t t = 0; t < d; ++t)
            blk[t] = 0.0;
        for (int64_t j = 0; j < nb; ++j) {
            double e = exp(s[j] - mb);
            lb += e;
            const uint16_t *vj = vbh + (j0 + j) * d;
            for (int64_t t = 0; t < d; ++t)
                blk[t] += e * bf16_to_double(vj[t]);
        }
        double m_new = m > mb ? m : mb;
        double c_old = exp(m - m_new), c_blk = exp(mb - m_new);
        l = l * c_old + lb * c_blk;
        for (int64_t t = 0; t < d; ++t)
            acc[t] = acc[t] * c_old + blk[t] * c_blk;
        m = m_new;
    }
    if (nv == 0) {
        for (int64_t t = 0; t < d; ++t)
            o[t] = 0.0;
        *lse = -INFINITY;
        return;
    }
    for (int64_t t = 0; t < d; ++t)
        o[t] = acc[t] / l;
    *lse = m + log(l);
}

/* Online forms over a list of rows; form is 1 or 2; block >= 1. */
int oracle_online_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                       int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal, float scale,
                       int64_t block, int form, const int64_t *rows, int64_t n, double *o,
                       double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (block < 1 || (form != 1 && form != 2) || n < 0 || (n > 0 && (!rows || !o || !lse)))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (!row_in_range(rows + 3 * r, B, H, Sq))
            return -3;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)(block + 2 * d));
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            if (!s)
                continue;
            int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            const uint16_t *qi = q + ((b * H + h) * Sq + i) * d;
            const uint16_t *kbh = k + (b * H + h) * Sk * d;
            const uint16_t *vbh = v + (b * H + h) * Sk * d;
            int64_t nv = visible_keys(i, Sq, Sk, causal);
            if (form == 1)
                online_form1_row(qi, kbh, vbh, nv, d, (double)scale, block, s, s + block,
                                 o + r * d, lse + r);
            else
                online_form2_row(qi, kbh, vbh, nv, d, (double)scale, block, s, s + block,
                                 s + block + d, o + r * d, lse + r);
        }
        free(s);
    }
    return failed ? -4 : 0;
}

/*
 * Split-KV with a final combine ("Lecture 06", section 5, Flash-Decoding).
 * The visible keys of each row are cut at the key indices in `bounds`
 * (n_chunks + 1 ascending values, bounds[0] = 0, bounds[n_chunks] = Sk); each
 * chunk [bounds[c], bounds[c+1]) intersected with the visible keys gives a
 * partial (o_c normalised over the chunk, lse_c) by the definition; then
 *   lse = M + ln sum_c e^{lse_c - M},  M = max_c lse_c,
 *   o   = sum_c e^{lse_c - lse} o_c.
 * Chunks with no visible key have lse_c = -inf and weight 0.
 */
int oracle_split_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                      int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal, float scale,
                      const int64_t *bounds, int64_t n_chunks, const int64_t *rows, int64_t n,
                      double *o, double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (!bounds || n_chunks < 1 || bounds[0] != 0 || bounds[n_chunks] != Sk)
        return -1;
    for (int64_t c = 0; c < n_chunks; ++c)
        if (bounds[c + 1] < bounds[c])
            return -1;
    if (n < 0 || (n > 0 && (!rows || !o || !lse)))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (!row_in_range(rows + 3 * r, B, H, Sq))
            return -3;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        size_t sz = (size_t)Sk + (size_t)(n_chunks * (d + 1));
        double *s = (double *)malloc(sizeof(double) * sz);
        if (!s) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            if (!s)
                continue;
            double *part_o = s + Sk, *part_lse = part_o + n_chunks * d;
            int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            const uint16_t *qi = q + ((b * H + h) * Sq + i) * d;
            const uint16_t *kbh = k + (b * H + h) * Sk * d;
            const uint16_t *vbh = v + (b * H + h) * Sk * d;
            int64_t nv = visible_keys(i, Sq, Sk, causal);
            for (int64_t c = 0; c < n_chunks; ++c) {
                int64_t j0 = bounds[c], j1 = bounds[c + 1];
                if (j1 > nv)
                    j1 = nv;
                definition_row(qi, kbh, vbh, j0, j1 > j0 ? j1 : j0, d, (double)scale, s,
                               part_o + c * d, part_lse + c);
            }
            double M = -INFINITY;
            for (int64_t c = 0; c < n_chunks; ++c)
                if (part_lse[c] > M)
                    M = part_lse[c];
            double *orow = o + r * d;
            for (int64_t t = 0; t < d; ++t)
                orow[t] = 0.0;
            if (M == -INFINITY) {
                lse[r] = -INFINITY;
                continue;
            }
            double sum = 0.0;
            for (int64_t c = 0; c < n_chunks; ++c)
                sum += exp(part_lse[c] - M);
            double L = M + log(sum);
            for (int64_t c = 0; c < n_chunks; ++c) {
                double w = exp(part_lse[c] - L);
                for (int64_t t = 0; t < d; ++t)
                    orow[t] += w * part_o[c * d + t];
            }
            lse[r] = L;
        }
        free(s);
    }
    return failed ? -4 : 0;
}

/*
 * The final combine of Flash-Decoding ("Lecture 06", section 5) on its own,
 * for partials computed elsewhere (another process, another device):
 * o_parts [n_parts, n_rows, d] (each normalised over its part of the keys),
 * lse_parts [n_parts, n_rows]; writes o [n_rows, d] and lse [n_rows] with the
 * same log-sum-exp weighting as oracle_split_rows. A part with lse = -inf
 * has weight 0; rows where every part is -inf get o = 0, lse = -inf.
 */
int oracle_combine(int64_t n_parts, int64_t n_rows, int64_t d, const double *o_parts,
                   const double *lse_parts, double *o, double *lse)
{
    if (n_parts < 1 || n_rows < 0 || d < 1 || !o_parts || !lse_parts || !o || !lse)
        return -1;
    for (int64_t r = 0; r < n_rows; ++r) {
        double M = -INFINITY;
        for (int64_t c = 0; c < n_parts; ++c)
            if (lse_parts[c * n_rows + r] > M)
                M = lse_parts[c * n_rows + r];
        double *orow = o + r * d;
        for (int64_t t = 0; t < d; ++t)
            orow[t] = 0.0;
        if (M == -INFINITY) {
            lse[r] = -INFINITY;
            continue;
        }
        double sum = 0.0;
        for (int64_t c = 0; c < n_parts; ++c)
            sum += exp(lse_parts[c * n_rows + r] - M);
        double L = M + log(sum);
        for (int64_t c = 0; c < n_parts; ++c) {
            double w = exp(lse_parts[c * n_rows + r] - L);
            const double *prow = o_parts + (c * n_rows + r) * d;
            for (int64_t t = 0; t < d; ++t)
                orow[t] += w * prow[t];
        }
        lse[r] = L;
    }
    return 0;
}

/*
 * The definition with an explicit visibility mask instead of the causal rule:
 * "Warmup Guide — Inference Optimization at Depth", Chapter 4 applies a mask
 * to S before the softmax; here visible[(b * Sq + i) * Sk + j] != 0 means key
 * j enters row i of batch element b (for every head). This covers the
 * tree-structured verify step of "Lecture 06 — Making Decode Fast", section 3
 * (several candidate continuations verified in one pass, each seeing the
 * cache and its own ancestors), where the visible keys of a row are not a
 * prefix. Rows with no visible key: o = 0, lse = -inf.
 * o: [B,H,Sq,d], lse: [B,H,Sq].
 */
int oracle_attention_masked(const uint16_t *q, const uint16_t *k, const uint16_t *v, int64_t B,
                            int64_t H, int64_t Sq, int64_t Sk, int64_t d, const uint8_t *visible,
                            float scale, double *o, double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (!visible || !o || !lse)
        return -1;
    set_threads(nthreads);
    const double sc = (double)scale;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Sk);
        int64_t *idx = (int64_t *)malloc(sizeof(int64_t) * (size_t)Sk);
        if (!s || !idx) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < B * H * Sq; ++r) {
            if (!s || !idx)
                continue;
            const int64_t b = r / (H * Sq), h = (r / Sq) % H, i = r % Sq;
            const uint16_t *qi = q + r * d;
            const uint16_t *kbh = k + (b * H + h) * Sk * d;
            const uint16_t *vbh = v + (b * H + h) * Sk * d;
            const uint8_t *vis = visible + (b * Sq + i) * Sk;
            double *orow = o + r * d;
            int64_t n = 0;
            for (int64_t j = 0; j < Sk; ++j)
                if (vis[j])
                    idx[n++] = j;
            for (int64_t t = 0; t < d; ++t)
                orow[t] = 0.0;
            if (n == 0) {
                lse[r] = -INFINITY;
                continue;
            }
            /* scores of the visible keys, then the two-pass safe softmax */
            for (int64_t a = 0; a < n; ++a) {
                const uint16_t *kj = kbh + idx[a] * d;
                double dot = 0.0;
                for (int64_t t = 0; t < d; ++t)
                    dot += bf16_to_double(qi[t]) * bf16_to_double(kj[t]);
                s[a] = sc * dot;
            }
            double m = -INFINITY;
            for (int64_t a = 0; a < n; ++a)
                if (s[a] > m)
                    m = s[a];
            double l = 0.0;
            for (int64_t a = 0; a < n; ++a)
                l += exp(s[a] - m);
            for (int64_t a = 0; a < n; ++a) {
                const double pj = exp(s[a] - m) / l;
                const uint16_t *vj = vbh + idx[a] * d;
                for (int64_t t = 0; t < d; ++t)
                    orow[t] += pj * bf16_to_double(vj[t]);
            }
            lse[r] = m + log(l);
        }
        free(s);
        free(idx);
    }
    return failed ? -4 : 0;
}

/*
 * Gradients of the definition, given the upstream gradient dO: the backward
 * pass the pages describe ("Warmup Guide — Inference Optimization at Depth",
 * Chapter 4: recompute the probability tiles from Q and K instead of storing
 * P). Here P is simply recomputed row by row from the definition (fp64), and
 * the chain rule of O = softmax(scale * Q K^T + mask) V gives, per row i:
 *   dP_ij = dO_i . v_j,       D_i = sum_j P_ij dP_ij,
 *   dS_ij = P_ij (dP_ij - D_i),
 *   dQ_i  = scale * sum_j dS_ij k_j,
 *   dK_j += scale * dS_ij q_i,   dV_j += P_ij dO_i.
 * q, k, v, dO: bf16 bits ([B,H,Sq,d], [B,H,Sk,d] x2, [B,H,Sq,d]); outputs
 * dq [B,H,Sq,d], dk and dv [B,H,Sk,d] (doubles). Rows with no visible key
 * contribute nothing.
 */
int oracle_attention_backward(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                              const uint16_t *dout, int64_t B, int64_t H, int64_t Sq, int64_t Sk,
                              int64_t d, int causal, float scale, double *dq, double *dk,
                              double *dv, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (!dout || !dq || !dk || !dv)
        return -1;
    set_threads(nthreads);
    const double sc = (double)scale;
    int failed = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)Sk);
        double *dp = (double *)malloc(sizeof(double) * (size_t)Sk);
        if (!p || !dp) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < B * H; ++bh) {
            if (!p || !dp)
                continue;
            const uint16_t *kbh = k + bh * Sk * d, *vbh = v + bh * Sk * d;
            double *dkbh = dk + bh * Sk * d, *dvbh = dv + bh * Sk * d;
            for (int64_t t = 0; t < Sk * d; ++t)
                dkbh[t] = dvbh[t] = 0.0;
            for (int64_t i = 0; i < Sq; ++i) {
                const uint16_t *qi = q + (bh * Sq + i) * d;
                const uint16_t *doi = dout + (bh * Sq + i) * d;
                double *dqi = dq + (bh * Sq + i) * d;
                for (int64_t t = 0; t < d; ++t)
                    dqi[t] = 0.0;
                const int64_t nv = visible_keys(i, Sq, Sk, causal);
                if (nv == 0)
                    continue;
                /* P_i by the definition (two-pass safe softmax) */
                score_row(qi, kbh, nv, d, sc, p);
                double m = -INFINITY;
                for (int64_t j = 0; j < nv; ++j)
                    if (p[j] > m)
                        m = p[j];
                double l = 0.0;
                for (int64_t j = 0; j < nv; ++j)
                    l += exp(p[j] - m);
                for (int64_t j = 0; j < nv; ++j)
                    p[j] = exp(p[j] - m) / l;
                /* dP_ij = dO_i . v_j and D_i = sum_j P_ij dP_ij */
                double D = 0.0;
                for (int64_t j = 0; j < nv; ++j) {
                    const uint16_t *vj = vbh + j * d;
                    double acc = 0.0;
                    for (int64_t t = 0; t < d; ++t)
                        acc += bf16_to_double(doi[t]) * bf16_to_double(vj[t]);
                    dp[j] = acc;
                    D += p[j] * acc;
                }
                for (int64_t j = 0; j < nv; ++j) {
                    const double ds = p[j] * (dp[j] - D);
                    const uint16_t *kj = kbh + j * d;
                    double *dkj = dkbh + j * d, *dvj = dvbh + j * d;
                    for (int64_t t = 0; t < d; ++t) {
                        dqi[t] += sc * ds * bf16_to_double(kj[t]);
                        dkj[t] += sc * ds * bf16_to_double(qi[t]);
                        dvj[t] += p[j] * bf16_to_double(doi[t]);
                    }
                }
            }
        }
        free(p);
        free(dp);
    }
    return failed ? -4 : 0;
}

/*
 * The same gradients for chosen rows of one (b, h): dQ of the query rows in
 * qrows, and dK, dV of the key rows in krows. Every query row's softmax row
 * and D_i are recomputed from the definition (parallel over query rows), so
 * this reaches long sequences where the full backward above would be slow.
 * bh selects the head; dq_rows [nq, d], dk_rows and dv_rows [nk, d].
 */
int oracle_attention_backward_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                                   const uint16_t *dout, int64_t B, int64_t H, int64_t Sq,
                                   int64_t Sk, int64_t d, int causal, float scale, int64_t bh,
                                   const int64_t *qrows, int64_t nq, const int64_t *krows,
                                   int64_t nk, double *dq_rows, double *dk_rows, double *dv_rows,
                                   int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (!dout || bh < 0 || bh >= B * H || nq < 0 || nk < 0 || (nq && (!qrows || !dq_rows)) ||
        (nk && (!krows || !dk_rows || !dv_rows)))
        return -1;
    for (int64_t a = 0; a < nq; ++a)
        if (qrows[a] < 0 || qrows[a] >= Sq)
            return -3;
    for (int64_t a = 0; a < nk; ++a)
        if (krows[a] < 0 || krows[a] >= Sk)
            return -3;
    set_threads(nthreads);
    const double sc = (double)scale;
    const uint16_t *kbh = k + bh * Sk * d, *vbh = v + bh * Sk * d;
    for (int64_t t = 0; t < nk * d; ++t)
        dk_rows[t] = dv_rows[t] = 0.0;
    /* which query rows want dQ: position in qrows, or -1 */
    int64_t *qslot = (int64_t *)malloc(sizeof(int64_t) * (size_t)Sq);
    if (!qslot)
        return -4;
    for (int64_t i = 0; i < Sq; ++i)
        qslot[i] = -1;
    for (int64_t a = 0; a < nq; ++a)
        qslot[qrows[a]] = a;
    int failed = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)Sk);
        double *dp = (double *)malloc(sizeof(double) * (size_t)Sk);
        double *pk = (double *)calloc((size_t)(2 * nk * d + 1), sizeof(double));
        if (!p || !dp || !pk) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 16)
        for (int64_t i = 0; i < Sq; ++i) {
            if (!p || !dp || !pk)
                continue;
            const int64_t nv = visible_keys(i, Sq, Sk, causal);
            const uint16_t *qi = q + (bh * Sq + i) * d, *doi = dout + (bh * Sq + i) * d;
            if (nv == 0)
                continue;
            score_row(qi, kbh, nv, d, sc, p);
            double m = -INFINITY;
            for (int64_t j = 0; j < nv; ++j)
                if (p[j] > m)
                    m = p[j];
            double l = 0.0;
            for (int64_t j = 0; j < nv; ++j)
                l += exp(p[j] - m);
            for (int64_t j = 0; j < nv; ++j)
                p[j] = exp(p[j] - m) / l;
            double D = 0.0;
            for (int64_t j = 0; j < nv; ++j) {
                const uint16_t *vj = vbh + j * d;
                double acc = 0.0;
                for (int64_t t = 0; t < d; ++t)
                    acc += bf16_to_double(doi[t]) * bf16_to_double(vj[t]);
                dp[j] = acc;
                D += p[j] * acc;
            }
            if (qslot[i] >= 0) {
                double *dqi = dq_rows + qslot[i] * d;
                for (int64_t t = 0; t < d; ++t)
                    dqi[t] = 0.0;
                for (int64_t j = 0; j < nv; ++j) {
                    const double ds = p[j] * (dp[j] - D);
                    const uint16_t *kj = kbh + j * d;
                    for (int64_t t = 0; t < d; ++t)
                        dqi[t] += sc * ds * bf16_to_double(kj[t]);
                }
            }
            for (int64_t a = 0; a < nk; ++a) {
                const int64_t j = krows[a];
                if (j >= nv)
                    continue;
                const double ds = p[j] * (dp[j] - D);
                for (int64_t t = 0; t < d; ++t) {
                    pk[a * d + t] += sc * ds * bf16_to_double(qi[t]);
                    pk[nk * d + a * d + t] += p[j] * bf16_to_double(doi[t]);
                }
            }
        }
        if (pk) {
#pragma omp critical
            for (int64_t t = 0; t < nk * d; ++t) {
                dk_rows[t] += pk[t];
                dv_rows[t] += pk[nk * d + t];
            }
        }
        free(p);
        free(dp);
        free(pk);
    }
    free(qslot);
    return failed ? -4 : 0;
}

/* ---------------------------------------------------------------- FP8 forward
 *
 * "FlashAttention, speculative decoding, quantisation and parallelism", The
 * problem it solves (FlashAttention-3 targets Hopper's asynchrony and FP8),
 * and "Lecture 06", section 5 (FlashAttention-3: FP8 support, FP8 up to about
 * 1.2 PFLOP/s): the same forward with Q, K and V stored as 8-bit floats. The
 * pages name FP8 and nothing else about it; the readings taken here:
 *   - the format is E4M3 without infinities ("e4m3fn"): 1 sign bit, 4
 *     exponent bits with bias 7, 3 mantissa bits; exponent field 0 holds the
 *     subnormals m/8 * 2^-6; S.1111.111 is NaN; the largest finite value is
 *     1.75 * 2^8 = 448;
 *   - one fp32 descale per tensor: the value an input byte stands for is
 *     descale * decode(byte);
 *   - the second product runs in FP8 as well, so P is rounded to E4M3 before
 *     it multiplies V. The rounding is taken against a power of two at the
 *     row's max: with x_j = s_j * log2(e) and M = ceil(max_j x_j), the weight
 *     used is P_j = 2^-7 * e4m3(2^7 * 2^(x_j - M)) (round to nearest, ties to
 *     even). M is an integer, so rounding against any other integer
 *     reference gives the same P_j up to an exact power of two (outside the
 *     subnormal range): a streaming kernel that settles its reference late
 *     reaches the same weights;
 *   - the row sum l = sum_j 2^(x_j - M) is taken before the rounding, so the
 *     LSE is the definition's;
 *   - o = sum_j P_j v_j / l and lse = ln 2 * (M + log2 l).
 * With quantize_p = 0 the weights are not rounded and the result is the
 * definition of attention on the decoded inputs.
 */

/* ln 2 (strict C11 has no M_LN2). */
static const double kLn2 = 0.693147180559945309417232121458176568;

/* Exact E4M3 -> double from the bit fields. */
static double e4m3_to_double(uint8_t x)
{
    const int e = (x >> 3) & 15, m = x & 7;
    double mag;
    if (e == 15 && m == 7)
        return NAN;
    if (e == 0)
        mag = ldexp((double)m, -9);        /* m/8 * 2^-6 */
    else
        mag = ldexp(8.0 + m, e - 10);      /* (1 + m/8) * 2^(e-7) */
    return (x & 0x80) ? -mag : mag;
}

/*
 * Round a finite double to the nearest E4M3 value, ties to the even mantissa,
 * magnitudes above 448 clamped to 448. The spacing in the binade [2^e, 2^e+1)
 * is 2^(e-3) (three mantissa bits); below 2^-6 it is the subnormal 2^-9.
 */
static double e4m3_round(double y)
{
    const double a = fabs(y);
    if (a == 0.0 || a != a)
        return y;
    int k;
    frexp(a, &k);                  /* a = f 2^k with f in [0.5, 1): floor(log2 a) = k - 1 */
    int e = k - 1;
    if (e < -6)
        e = -6;
    const double q = ldexp(1.0, e - 3);
    const double r = a / q;        /* exact: q is a power of two */
    double n = floor(r);
    const double frac = r - n;
    if (frac > 0.5 || (frac == 0.5 && fmod(n, 2.0) == 1.0))
        n += 1.0;
    double out = n * q;
    if (out > 448.0)
        out = 448.0;
    return y < 0 ? -out : out;
}

/* Decode n bytes (for the pins). */
int oracle_e4m3_decode(const uint8_t *x, int64_t n, double *out)
{
    if (n < 0 || (n > 0 && (!x || !out)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_to_double(x[i]);
    return 0;
}

/* Round n doubles to E4M3 values (for the pins). */
int oracle_e4m3_round(const double *y, int64_t n, double *out)
{
    if (n < 0 || (n > 0 && (!y || !out)))
        return -1;
    for (int64_t i = 0; i < n; ++i)
        out[i] = e4m3_round(y[i]);
    return 0;
}

/* One FP8 row over keys [0, n): the steps listed above. x: n doubles of scratch. */
static void fp8_row(const uint8_t *qi, const uint8_t *kbh, const uint8_t *vbh, int64_t n, int64_t d,
                    double scale, double dq, double dk, double dv, int quantize_p, double *x,
                    double *o, double *lse)
{
    for (int64_t t = 0; t < d; ++t)
        o[t] = 0.0;
    if (n <= 0) {
        *lse = -INFINITY;
        return;
    }
    /* s_j = scale * (dq q_i) . (dk k_j); x_j = s_j log2(e) */
    double mx = -INFINITY;
    for (int64_t j = 0; j < n; ++j) {
        const uint8_t *kj = kbh + j * d;
        double dot = 0.0;
        for (int64_t t = 0; t < d; ++t)
            dot += (dq * e4m3_to_double(qi[t])) * (dk * e4m3_to_double(kj[t]));
        x[j] = scale * dot / kLn2;
        if (x[j] > mx)
            mx = x[j];
    }
    const double M = quantize_p ? ceil(mx) : mx;
    double l = 0.0;
    for (int64_t j = 0; j < n; ++j)
        l += exp2(x[j] - M);
    for (int64_t j = 0; j < n; ++j) {
        double p = exp2(x[j] - M);
        if (quantize_p)
            p = ldexp(e4m3_round(ldexp(p, 7)), -7);
        const uint8_t *vj = vbh + j * d;
        for (int64_t t = 0; t < d; ++t)
            o[t] += p * (dv * e4m3_to_double(vj[t]));
    }
    for (int64_t t = 0; t < d; ++t)
        o[t] /= l;
    *lse = kLn2 * (M + log2(l));
}

/*
 * FP8 forward for a list of rows. q: E4M3 bytes [B,H,Sq,d]; k, v: [B,H,Sk,d];
 * rows: n triples (b,h,i); o: n*d doubles; lse: n doubles.
 */
int oracle_attention_fp8_rows(const uint8_t *q, const uint8_t *k, const uint8_t *v, int64_t B,
                              int64_t H, int64_t Sq, int64_t Sk, int64_t d, int causal, float scale,
                              float q_descale, float k_descale, float v_descale, int quantize_p,
                              const int64_t *rows, int64_t n, double *o, double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (n < 0 || (n > 0 && (!rows || !o || !lse)))
        return -1;
    for (int64_t r = 0; r < n; ++r)
        if (!row_in_range(rows + 3 * r, B, H, Sq))
            return -3;
    set_threads(nthreads);
    int failed = 0;
#pragma omp parallel
    {
        double *x = (double *)malloc(sizeof(double) * (size_t)Sk);
        if (!x) {
#pragma omp atomic write
            failed = 1;
        }
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n; ++r) {
            if (!x)
                continue;
            int64_t b = rows[3 * r], h = rows[3 * r + 1], i = rows[3 * r + 2];
            const uint8_t *qi = q + ((b * H + h) * Sq + i) * d;
            const uint8_t *kbh = k + (b * H + h) * Sk * d;
            const uint8_t *vbh = v + (b * H + h) * Sk * d;
            fp8_row(qi, kbh, vbh, visible_keys(i, Sq, Sk, causal), d, (double)scale,
                    (double)q_descale, (double)k_descale, (double)v_descale, quantize_p, x,
                    o + r * d, lse + r);
        }
        free(x);
    }
    return failed ? -4 : 0;
}

/* Every row: o [B,H,Sq,d], lse [B,H,Sq] (doubles). */
int oracle_attention_fp8(const uint8_t *q, const uint8_t *k, const uint8_t *v, int64_t B, int64_t H,
                         int64_t Sq, int64_t Sk, int64_t d, int causal, float scale,
                         float q_descale, float k_descale, float v_descale, int quantize_p,
                         double *o, double *lse, int nthreads)
{
    int rc = check_args(q, k, v, B, H, Sq, Sk, d);
    if (rc)
        return rc;
    if (!o || !lse)
        return -1;
    int64_t n = B * H * Sq;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * 3 * (size_t)n);
    if (!rows)
        return -4;
    for (int64_t b = 0, r = 0; b < B; ++b)
        for (int64_t h = 0; h < H; ++h)
            for (int64_t i = 0; i < Sq; ++i, ++r) {
                rows[3 * r] = b;
                rows[3 * r + 1] = h;
                rows[3 * r + 2] = i;
            }
    rc = oracle_attention_fp8_rows(q, k, v, B, H, Sq, Sk, d, causal, scale, q_descale, k_descale,
                                   v_descale, quantize_p, rows, n, o, lse, nthreads);
    free(rows);
    return rc;
}
