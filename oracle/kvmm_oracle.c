/*
 * kvmm_oracle.c -- plain, slow CPU oracle for query-aware MinMax page
 * selection followed by sparse paged GQA decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path links, loads or
 * calls this file: it is used by the tests, by the smoke check and by the
 * CPU-baseline leg of the benchmark.  It shares no code, header, table or
 * helper with the CUDA library; the two only ever see the same input bytes.
 *
 * Every computation is written straight from its definition, one unit
 * (batch b, layer l, KV head h) at a time, in double precision, with no
 * blocking, fusion or reordering:
 *
 *   FlexiCache: Leveraging Temporal Stability of Attention Heads for
 *   Efficient KV Cache Management (blog summary of the MLSys'26 paper)
 *     - "Core method, 2. MinMax-metadata page scoring": every KV page keeps
 *       the per-channel minimum and maximum of its keys; the query and these
 *       bounds give an estimate of the largest dot product the page can
 *       produce; the top-K pages are chosen per (layer, KV head).
 *     - "Core method, 3. Periodic reranking and incremental promotion":
 *       after a rerank only (current top-K minus previous top-K) is moved.
 *     - "System design, head-level block table": the block table is
 *       [batch, layer, head, logical_block]; evicted slots point at a null
 *       block that is never dereferenced.
 *     - "Core method, 4" and "System design" (physical block reuse): after a
 *       rerank the promoted pages are brought from the host KV into the
 *       physical blocks of the evicted pages.
 *     - "Core method, 1. Stability-differentiated placement": decode
 *       attention runs over the top-K pages only.
 *     - "Core insight: attention heads differ in temporal stability": the
 *       top-K sets of a head are compared a few steps apart with the
 *       Random-Corrected Overlap (1 = identical sets, 0 = the overlap of
 *       random sets), aggregated over a window W; the least stable quarter
 *       of the heads is unstable.
 *   KVDrive: A Holistic Multi-Tier KV Cache Management System for
 *   Long-Context LLM Inference, "Background and key observations": Quest
 *   multiplies the query with the keys' channel-wise min and max.
 *   KVDrive, "Method details": each page's mean key is its representative
 *   in the index; the mean-key scorer ranks pages by q . mean.
 *
 * Readings taken where the pages are silent (the plainest one the rest of
 *   the pages supports; none of these points is printed on either page):
 *   - page score for one query head: sum_d max(q_d*min_d, q_d*max_d), the
 *     exact maximum of q.k over the box [min, max];
 *   - GQA: the KV head's score is the SUM of its query heads' scores
 *     (group_reduce = 0); group_reduce = 1 takes the MAX instead;
 *   - top-K ties go to the lower logical page index; if a unit has no more
 *     than K pages, all of them are selected; the selection is emitted in
 *     ascending page order;
 *   - a partial last page uses only its valid tokens (< seq_len);
 *   - min/max of bf16 values is taken in value order with -0 < +0, so the
 *     result is a unique bf16 bit pattern;
 *   - attention scale defaults to D^-1/2; output and log-sum-exp in double;
 *     a unit with no valid token yields output 0 and lse = -inf.
 *   - a page's mean key is its keys' fp32 sum in token order over their
 *     count, rounded to bf16 nearest-even (the rounding decides the stored
 *     code, so it is taken in the kernel's precision); its score for head g
 *     is q_g . mean in double;
 *   - promotion pairs promoted[i] with evicted[i] (both ascending) for
 *     i < min(np, ne): the evicted page's block goes to the promoted page,
 *     the evicted entry becomes the null block; surplus evicted blocks are
 *     freed in order, surplus promoted pages stay unplaced;
 *   - RCO(A, B) = (|A n B| - |A||B|/P) / (min(|A|,|B|) - |A||B|/P): the
 *     overlap minus that of random subsets of the same sizes among P pages,
 *     over its largest possible value (evaluated as the ratio of the exact
 *     integers P|A n B| - |A||B| and P min(|A|,|B|) - |A||B|); 1 when the two
 *     are equal (every page selected, or P = 0); P is the later (larger) page
 *     count of the two
 *     steps; a head's stability is the mean over the window's pairs (and
 *     over the batch); round(frac * heads) heads of lowest stability are
 *     unstable, ties to the lower index.
 *
 * bf16 values are passed as their raw 16-bit patterns (uint16_t).
 *
 * Pool layouts: k_pool is [n_phys][T][D] (token-major); v_pool is
 * [n_phys][D][T] (each page's values stored dimension-major, as paged
 * serving engines lay out the value cache).
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Device-error bits, defined here on their own (same meaning as the
 * library's): a selected logical page whose table entry is the null block,
 * and a table entry outside the physical pool. */
#define ORACLE_ERR_NULL_BLOCK 1
#define ORACLE_ERR_OUT_OF_RANGE 2

static double bf16_value(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* a strictly before b in the order used for min/max: by value, and -0 < +0 */
static int bf16_before(uint16_t a, uint16_t b)
{
    double x = bf16_value(a), y = bf16_value(b);
    if (x < y) return 1;
    if (x > y) return 0;
    return (a & 0x8000u) && !(b & 0x8000u);
}

/* Resolve a logical page through the unit's block-table row.
 * Returns the physical page, or -1 after setting the matching error bit. */
static int64_t resolve_page(const int32_t* bt_row, int32_t logical, int64_t n_phys, int32_t* err)
{
    int32_t phys = bt_row[logical];
    if (phys < 0) {
        *err |= ORACLE_ERR_NULL_BLOCK;
        return -1;
    }
    if ((int64_t)phys >= n_phys) {
        *err |= ORACLE_ERR_OUT_OF_RANGE;
        return -1;
    }
    return phys;
}

/* Number of valid tokens of logical page p in a sequence of seq_len tokens. */
static int32_t valid_tokens(int32_t p, int32_t T, int32_t seq_len)
{
    int64_t first = (int64_t)p * T;
    if (first >= seq_len) return 0;
    int64_t n = (int64_t)seq_len - first;
    return n < T ? (int32_t)n : T;
}

/* ---------------------------------------------------------------------------
 * Append: write new token rows into their pages through the block table.
 * Token tok_begin + j takes row j of new_k / new_v ([n][D]).
 * Returns error bits; rows whose page is null or out of range are skipped.
 */
int32_t oracle_unit_append(uint16_t* k_pool, uint16_t* v_pool, int64_t n_phys, int32_t T, int32_t D,
                           const int32_t* bt_row, int32_t tok_begin, int32_t tok_end,
                           const uint16_t* new_k, const uint16_t* new_v)
{
    int32_t err = 0;
    for (int32_t t = tok_begin; t < tok_end; ++t) {
        int64_t phys = resolve_page(bt_row, t / T, n_phys, &err);
        if (phys < 0) continue;
        int64_t row = phys * T + (t % T);
        for (int32_t d = 0; d < D; ++d) {
            k_pool[row * D + d] = new_k[(int64_t)(t - tok_begin) * D + d];
            v_pool[(phys * D + d) * T + (t % T)] = new_v[(int64_t)(t - tok_begin) * D + d];
        }
    }
    return err;
}

/* ---------------------------------------------------------------------------
 * MinMax metadata of logical pages [page_begin, page_end) of one unit:
 * meta[p][0][d] = min over the page's valid tokens of k[t][d],
 * meta[p][1][d] = max over the same tokens.  Pages with no valid token and
 * pages whose entry is null / out of range are left untouched.
 */
int32_t oracle_unit_minmax(const uint16_t* k_pool, int64_t n_phys, int32_t T, int32_t D,
                           const int32_t* bt_row, int32_t seq_len, int32_t page_begin,
                           int32_t page_end, uint16_t* meta)
{
    int32_t err = 0;
    for (int32_t p = page_begin; p < page_end; ++p) {
        int32_t n = valid_tokens(p, T, seq_len);
        if (n == 0) continue;
        int64_t phys = resolve_page(bt_row, p, n_phys, &err);
        if (phys < 0) continue;
        const uint16_t* page = k_pool + phys * T * D;
        uint16_t* mn = meta + (int64_t)p * 2 * D;
        uint16_t* mx = mn + D;
        for (int32_t d = 0; d < D; ++d) {
            uint16_t lo = page[d], hi = page[d];
            for (int32_t r = 1; r < n; ++r) {
                uint16_t x = page[(int64_t)r * D + d];
                if (bf16_before(x, lo)) lo = x;
                if (bf16_before(hi, x)) hi = x;
            }
            mn[d] = lo;
            mx[d] = hi;
        }
    }
    return err;
}

/* ---------------------------------------------------------------------------
 * Page scores of one unit.  q is [G][D] (the query heads of the KV head's
 * group), meta is [P][2][D].  For query head g:
 *     s_g(p) = sum_d max(q[g][d] * min_p[d], q[g][d] * max_p[d])
 * and the unit's score is sum_g s_g(p) (group_reduce 0) or max_g s_g(p)
 * (group_reduce 1).
 */
void oracle_unit_scores(const uint16_t* q, int32_t G, int32_t D, const uint16_t* meta, int32_t P,
                        int32_t group_reduce, double* scores)
{
    for (int32_t p = 0; p < P; ++p) {
        const uint16_t* mn = meta + (int64_t)p * 2 * D;
        const uint16_t* mx = mn + D;
        double total = 0.0;
        for (int32_t g = 0; g < G; ++g) {
            double s = 0.0;
            for (int32_t d = 0; d < D; ++d) {
                double qd = bf16_value(q[(int64_t)g * D + d]);
                double a = qd * bf16_value(mn[d]);
                double b = qd * bf16_value(mx[d]);
                s += (a > b) ? a : b;
            }
            if (group_reduce == 1)
                total = (g == 0 || s > total) ? s : total;
            else
                total += s;
        }
        scores[p] = total;
    }
}

/* ---------------------------------------------------------------------------
 * Top-K: order the pages by (score descending, page index ascending), keep
 * the first min(K, P), and return them in ascending page order.
 */
typedef struct {
    double score;
    int32_t page;
} scored_page;

static int by_score_then_page(const void* a, const void* b)
{
    const scored_page* x = (const scored_page*)a;
    const scored_page* y = (const scored_page*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->page > y->page) - (x->page < y->page);
}

static int by_int(const void* a, const void* b)
{
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

int32_t oracle_topk(const double* scores, int32_t P, int32_t K, int32_t* sel)
{
    if (P <= 0 || K <= 0) return 0;
    scored_page* order = (scored_page*)malloc(sizeof(scored_page) * (size_t)P);
    if (!order) return -1;
    for (int32_t p = 0; p < P; ++p) {
        order[p].score = scores[p];
        order[p].page = p;
    }
    qsort(order, (size_t)P, sizeof(scored_page), by_score_then_page);
    int32_t n = K < P ? K : P;
    for (int32_t i = 0; i < n; ++i) sel[i] = order[i].page;
    free(order);
    qsort(sel, (size_t)n, sizeof(int32_t), by_int);
    return n;
}

/* ---------------------------------------------------------------------------
 * Set difference a \ b of two ascending lists, in ascending order.
 * promoted = cur \ prev, evicted = prev \ cur.
 */
int32_t oracle_set_difference(const int32_t* a, int32_t na, const int32_t* b, int32_t nb, int32_t* out)
{
    int32_t n = 0;
    for (int32_t i = 0; i < na; ++i) {
        int found = 0;
        for (int32_t j = 0; j < nb; ++j)
            if (b[j] == a[i]) found = 1;
        if (!found) out[n++] = a[i];
    }
    return n;
}

/* ---------------------------------------------------------------------------
 * Softmax attention of G query heads over an explicit list of n tokens
 * (rows[t] = phys * T + r: token r of physical page phys, in the order given):
 *     z_t = scale * sum_d q[g][d] * k_t[d]
 *     out[g] = sum_t exp(z_t - m) v_t / sum_t exp(z_t - m),   m = max_t z_t
 *     lse[g] = m + log(sum_t exp(z_t - m))
 */
static void attend_rows(const uint16_t* q, int32_t G, int32_t D, int32_t T, const uint16_t* k_pool,
                        const uint16_t* v_pool, const int64_t* rows, int64_t n, double scale,
                        double* out, double* lse)
{
    double* z = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    for (int32_t g = 0; g < G; ++g) {
        double* o = out + (int64_t)g * D;
        for (int32_t d = 0; d < D; ++d) o[d] = 0.0;
        if (n == 0 || !z) {
            lse[g] = -INFINITY;
            continue;
        }
        double m = -INFINITY;
        for (int64_t t = 0; t < n; ++t) {
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d)
                dot += bf16_value(q[(int64_t)g * D + d]) * bf16_value(k_pool[rows[t] * D + d]);
            z[t] = dot * scale;
            if (z[t] > m) m = z[t];
        }
        double denom = 0.0;
        for (int64_t t = 0; t < n; ++t) {
            double w = exp(z[t] - m);
            denom += w;
            int64_t phys = rows[t] / T, r = rows[t] % T;
            for (int32_t d = 0; d < D; ++d) o[d] += w * bf16_value(v_pool[(phys * D + d) * T + r]);
        }
        for (int32_t d = 0; d < D; ++d) o[d] /= denom;
        lse[g] = m + log(denom);
    }
    free(z);
}

/* Sparse decode attention of one unit over its selected logical pages
 * sel[0..cnt), each resolved through the block-table row; tokens at or past
 * seq_len are not attended; null / out-of-range entries set their error bit
 * and contribute nothing.  scale <= 0 means D^-1/2. */
int32_t oracle_unit_sparse_attention(const uint16_t* q, int32_t G, int32_t D, int32_t T,
                                     const uint16_t* k_pool, const uint16_t* v_pool,
                                     int64_t n_phys, const int32_t* bt_row, int32_t seq_len,
                                     const int32_t* sel, int32_t cnt, double scale, double* out,
                                     double* lse)
{
    int32_t err = 0;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * ((size_t)cnt * T + 1));
    int64_t n = 0;
    for (int32_t i = 0; i < cnt; ++i) {
        int32_t nv = valid_tokens(sel[i], T, seq_len);
        if (nv == 0) continue;
        int64_t phys = resolve_page(bt_row, sel[i], n_phys, &err);
        if (phys < 0) continue;
        for (int32_t r = 0; r < nv; ++r) rows[n++] = phys * T + r;
    }
    attend_rows(q, G, D, T, k_pool, v_pool, rows, n, scale, out, lse);
    free(rows);
    return err;
}

/* Dense decode attention of one unit: every token t < seq_len, in token
 * order, each found through the block-table row. */
int32_t oracle_unit_dense_attention(const uint16_t* q, int32_t G, int32_t D, int32_t T,
                                    const uint16_t* k_pool, const uint16_t* v_pool,
                                    int64_t n_phys, const int32_t* bt_row, int32_t seq_len,
                                    double scale, double* out, double* lse)
{
    int32_t err = 0;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * ((size_t)seq_len + 1));
    int64_t n = 0;
    for (int32_t t = 0; t < seq_len; ++t) {
        int64_t phys = resolve_page(bt_row, t / T, n_phys, &err);
        if (phys < 0) continue;
        rows[n++] = phys * T + (t % T);
    }
    attend_rows(q, G, D, T, k_pool, v_pool, rows, n, scale, out, lse);
    free(rows);
    return err;
}

/* ---------------------------------------------------------------------------
 * One decode step of one unit, in the method's order (the CPU baseline):
 *   append the new token and refresh the MinMax of its page; if the unit is
 *   rescored this step, score every page, select the top-K and list
 *   promoted = cur \ prev and evicted = prev \ cur, then make cur the unit's
 *   selection; otherwise keep the previous selection; finally run sparse
 *   attention over the selection.
 * sel / sel_cnt hold the previous selection on entry and the current one on
 * return.  scores is caller scratch of P entries.
 */
int32_t oracle_unit_step(uint16_t* k_pool, uint16_t* v_pool, int64_t n_phys, int32_t T, int32_t D,
                         const int32_t* bt_row, int32_t seq_len, const uint16_t* new_k,
                         const uint16_t* new_v, uint16_t* meta, const uint16_t* q, int32_t G,
                         int32_t rescore, int32_t K, int32_t group_reduce, int32_t* sel,
                         int32_t* sel_cnt, int32_t* promoted, int32_t* n_promoted, int32_t* evicted,
                         int32_t* n_evicted, double* scores, double scale, double* out, double* lse)
{
    int32_t err = 0;
    int32_t P = (seq_len + T - 1) / T;
    if (new_k && new_v && seq_len > 0) {
        err |= oracle_unit_append(k_pool, v_pool, n_phys, T, D, bt_row, seq_len - 1, seq_len, new_k, new_v);
        err |= oracle_unit_minmax(k_pool, n_phys, T, D, bt_row, seq_len, P - 1, P, meta);
    }
    *n_promoted = 0;
    *n_evicted = 0;
    if (rescore) {
        int32_t* cur = (int32_t*)malloc(sizeof(int32_t) * (size_t)(K > 0 ? K : 1));
        oracle_unit_scores(q, G, D, meta, P, group_reduce, scores);
        int32_t n = oracle_topk(scores, P, K, cur);
        *n_promoted = oracle_set_difference(cur, n, sel, *sel_cnt, promoted);
        *n_evicted = oracle_set_difference(sel, *sel_cnt, cur, n, evicted);
        memcpy(sel, cur, sizeof(int32_t) * (size_t)n);
        *sel_cnt = n;
        free(cur);
    }
    err |= oracle_unit_sparse_attention(q, G, D, T, k_pool, v_pool, n_phys, bt_row, seq_len, sel,
                                        *sel_cnt, scale, out, lse);
    return err;
}

/* ------------------------------------------------------------------------
 * Temporal stability (FlexiCache, "Core insight: attention heads differ in
 * temporal stability").
 */

/* |A n B| of two sets of distinct page indices, in any order: every pair. */
static int32_t overlap_count(const int32_t* a, int32_t na, const int32_t* b, int32_t nb)
{
    int32_t n = 0;
    for (int32_t i = 0; i < na; ++i)
        for (int32_t j = 0; j < nb; ++j)
            if (a[i] == b[j]) {
                ++n;
                break;
            }
    return n;
}

/* Random-Corrected Overlap of sets A and B drawn from P pages:
 *   (|A n B| - |A||B|/P) / (min(|A|,|B|) - |A||B|/P),
 * |A||B|/P the expected overlap of random subsets of those sizes, min the
 * largest possible.  Numerator and denominator are multiplied by P > 0, so
 * both are exact integers and the value is one correctly rounded division. */
double oracle_rco(const int32_t* a, int32_t na, const int32_t* b, int32_t nb, int32_t P)
{
    if (P <= 0) return 1.0;
    const int64_t chance_p = (int64_t)na * nb;         /* P * expected overlap */
    const int64_t best_p = (int64_t)(na < nb ? na : nb) * P; /* P * largest overlap */
    if (best_p - chance_p <= 0) return 1.0;
    return (double)((int64_t)overlap_count(a, na, b, nb) * P - chance_p) / (double)(best_p - chance_p);
}

/* A unit's stability over a window of n recorded steps, newest first: step t
 * holds cnt[t] pages at idx + t * kmax, taken over pages[t] pages.  The mean
 * of RCO(step t, step t + lag) over t = 0 .. n - lag - 1, P the larger of the
 * two page counts.  NaN when there is no pair. */
double oracle_unit_stability(const int32_t* idx, const int32_t* cnt, const int32_t* pages, int32_t kmax,
                             int32_t n, int32_t lag)
{
    double sum = 0.0;
    int32_t pairs = 0;
    for (int32_t t = 0; t + lag < n; ++t) {
        const int32_t P = pages[t] > pages[t + lag] ? pages[t] : pages[t + lag];
        sum += oracle_rco(idx + (int64_t)t * kmax, cnt[t], idx + (int64_t)(t + lag) * kmax, cnt[t + lag], P);
        ++pairs;
    }
    return pairs ? sum / (double)pairs : NAN;
}

/* unstable[i] = 1 for the round(frac * n) entries of lowest stability (ties:
 * lower index first), else 0.  round() rounds half up: floor(x + 0.5). */
void oracle_classify(const double* stability, int32_t n, double frac, uint8_t* unstable)
{
    const int32_t k = (int32_t)floor(frac * (double)n + 0.5);
    for (int32_t i = 0; i < n; ++i) {
        int32_t rank = 0;
        for (int32_t j = 0; j < n; ++j)
            if (stability[j] < stability[i] || (stability[j] == stability[i] && j < i)) ++rank;
        unstable[i] = rank < k ? 1 : 0;
    }
}

/* ------------------------------------------------------------------------
 * Promotion of one unit (FlexiCache, "Core method, 3" / "Core method, 4" /
 * "System design, head-level block table"): the pairs i < m = min(np, ne)
 * move the block of evicted[i] to promoted[i] and copy the host store's page
 * promoted[i] (keys [T][D] and values [D][T], host_k/host_v hold the unit's
 * Pmax pages) into it; evicted entries become -1; the blocks of evicted[i],
 * i >= m, are returned in freed[i - m] (-1 for a skipped entry).  A pair
 * whose evicted entry is null / out of range, or whose pages lie outside
 * [0, Pmax), moves nothing and sets its error bit.  Returns the error bits;
 * *moved receives the pages moved.
 */
int32_t oracle_unit_promote(int32_t* bt_row, int32_t Pmax, int64_t n_phys, const int32_t* promoted, int32_t np,
                            const int32_t* evicted, int32_t ne, const uint16_t* host_k, const uint16_t* host_v,
                            uint16_t* k_pool, uint16_t* v_pool, int32_t T, int32_t D, int32_t* freed,
                            int32_t* moved)
{
    int32_t err = 0;
    const int32_t m = np < ne ? np : ne;
    const int64_t page = (int64_t)T * D;
    int64_t* block = (int64_t*)malloc(sizeof(int64_t) * (size_t)(ne > 0 ? ne : 1));
    /* the evicted entries: read their blocks, then null them */
    for (int32_t i = 0; i < ne; ++i) {
        block[i] = -1;
        if (evicted[i] < 0 || evicted[i] >= Pmax) {
            err |= ORACLE_ERR_OUT_OF_RANGE;
            continue;
        }
        const int32_t ph = bt_row[evicted[i]];
        if (ph < 0)
            err |= ORACLE_ERR_NULL_BLOCK;
        else if (ph >= n_phys)
            err |= ORACLE_ERR_OUT_OF_RANGE;
        else
            block[i] = ph;
        bt_row[evicted[i]] = -1;
    }
    int32_t n = 0;
    for (int32_t i = 0; i < m; ++i) {
        if (promoted[i] < 0 || promoted[i] >= Pmax) {
            err |= ORACLE_ERR_OUT_OF_RANGE;
            continue;
        }
        if (block[i] < 0) continue;
        bt_row[promoted[i]] = (int32_t)block[i];
        memcpy(k_pool + block[i] * page, host_k + (int64_t)promoted[i] * page, sizeof(uint16_t) * (size_t)page);
        memcpy(v_pool + block[i] * page, host_v + (int64_t)promoted[i] * page, sizeof(uint16_t) * (size_t)page);
        ++n;
    }
    for (int32_t i = m; i < ne; ++i)
        if (freed) freed[i - m] = (int32_t)block[i];
    free(block);
    *moved = n;
    return err;
}

/* Changed entries of a block table (FlexiCache, "System design, head-level
 * block table": dirty tracking synchronises only what changed):
 * table[idx[i]] = val[i] in order; an index outside [0, entries) or a value
 * outside [-1, n_phys) is skipped and sets ORACLE_ERR_OUT_OF_RANGE. */
int32_t oracle_table_update(int32_t* table, int64_t entries, int64_t n_phys, const int64_t* idx,
                            const int32_t* val, int64_t n)
{
    int32_t err = 0;
    for (int64_t i = 0; i < n; ++i) {
        if (idx[i] < 0 || idx[i] >= entries || val[i] < -1 || val[i] >= n_phys) {
            err |= ORACLE_ERR_OUT_OF_RANGE;
            continue;
        }
        table[idx[i]] = val[i];
    }
    return err;
}

/* ------------------------------------------------------------------------
 * The mean-key scorer (KVDrive, "Method details": each page's mean key is
 * its representative).
 */

/* float -> bf16 bit pattern, rounding to nearest, ties to even (finite x) */
static uint16_t bf16_round_nearest_even(float x)
{
    uint32_t u;
    memcpy(&u, &x, sizeof(u));
    const uint32_t lsb = (u >> 16) & 1u;
    u += 0x7fffu + lsb;
    return (uint16_t)(u >> 16);
}

/* mean[p][d] for logical pages [page_begin, page_end) with valid tokens:
 * the fp32 sum of k[t][d] over the page's valid tokens in token order,
 * divided by their count, rounded to bf16.  Null / out-of-range entries
 * set their error bit and the page is left untouched. */
int32_t oracle_unit_meankey(const uint16_t* k_pool, int64_t n_phys, int32_t T, int32_t D, const int32_t* bt_row,
                            int32_t seq_len, int32_t page_begin, int32_t page_end, uint16_t* mean)
{
    int32_t err = 0;
    for (int32_t p = page_begin; p < page_end; ++p) {
        const int32_t n = valid_tokens(p, T, seq_len);
        if (n == 0) continue;
        const int64_t phys = resolve_page(bt_row, p, n_phys, &err);
        if (phys < 0) continue;
        const uint16_t* page = k_pool + phys * T * D;
        for (int32_t d = 0; d < D; ++d) {
            float acc = 0.0f;
            for (int32_t r = 0; r < n; ++r) acc += (float)bf16_value(page[(int64_t)r * D + d]);
            mean[(int64_t)p * D + d] = bf16_round_nearest_even(acc / (float)n);
        }
    }
    return err;
}

/* s(p) = sum_g q_g . mean_p (group_reduce 0) or max_g (group_reduce 1), in double */
void oracle_unit_mean_scores(const uint16_t* q, int32_t G, int32_t D, const uint16_t* mean, int32_t P,
                             int32_t group_reduce, double* scores)
{
    for (int32_t p = 0; p < P; ++p) {
        double heads = 0.0; /* the group's reduction */
        for (int32_t g = 0; g < G; ++g) {
            double s = 0.0;
            for (int32_t d = 0; d < D; ++d)
                s += bf16_value(q[(int64_t)g * D + d]) * bf16_value(mean[(int64_t)p * D + d]);
            if (group_reduce == 1)
                heads = (g == 0 || s > heads) ? s : heads;
            else
                heads = heads + s;
        }
        scores[p] = heads;
    }
}

/* Dense attention mass of every page: mass[g][p] = sum over the page's valid
 * tokens of softmax_t(scale * q_g . k_t), the softmax taken over every token
 * below seq_len (through the block table).  A page whose entry is null
 * contributes 0.  scale <= 0 means D^-1/2. */
int32_t oracle_unit_page_mass(const uint16_t* q, int32_t G, int32_t D, int32_t T, const uint16_t* k_pool,
                              int64_t n_phys, const int32_t* bt_row, int32_t seq_len, double scale, double* mass)
{
    int32_t err = 0;
    if (scale <= 0.0) scale = 1.0 / sqrt((double)D);
    const int32_t P = (seq_len + T - 1) / T;
    double* z = (double*)malloc(sizeof(double) * (size_t)(seq_len > 0 ? seq_len : 1));
    int64_t* row = (int64_t*)malloc(sizeof(int64_t) * (size_t)(seq_len > 0 ? seq_len : 1));
    for (int32_t t = 0; t < seq_len; ++t) {
        const int64_t phys = resolve_page(bt_row, t / T, n_phys, &err);
        row[t] = phys < 0 ? -1 : phys * T + t % T;
    }
    for (int32_t g = 0; g < G; ++g) {
        double m = -INFINITY;
        for (int32_t t = 0; t < seq_len; ++t) {
            z[t] = -INFINITY;
            if (row[t] < 0) continue;
            double dot = 0.0;
            for (int32_t d = 0; d < D; ++d)
                dot += bf16_value(q[(int64_t)g * D + d]) * bf16_value(k_pool[row[t] * D + d]);
            z[t] = dot * scale;
            if (z[t] > m) m = z[t];
        }
        double denom = 0.0;
        for (int32_t t = 0; t < seq_len; ++t) denom += (row[t] < 0) ? 0.0 : exp(z[t] - m);
        for (int32_t p = 0; p < P; ++p) mass[(int64_t)g * P + p] = 0.0;
        for (int32_t t = 0; t < seq_len; ++t)
            if (row[t] >= 0) mass[(int64_t)g * P + t / T] += exp(z[t] - m) / denom;
    }
    free(z);
    free(row);
    return err;
}

/* ------------------------------------------------------------------------
 * The centroid level of KVDrive's index ("Method details": each page's mean
 * key is its representative, and higher-level centroids group similar pages;
 * "the trade-off between block size and centroid count": the centroid count
 * is proportional to the context, and the grouping is by similarity, with
 * half the centroids a spatial blocking of the pages needs).  The page names
 * no clustering algorithm.  The reading taken: Lloyd's k-means over a unit's
 * pages' mean keys, started from spatial blocks of R consecutive pages
 * (n_c = ceil(P / R) centroids; n_iter = 0 leaves the spatial blocks), with
 *   - the assignment: page p joins the centroid j of least squared Euclidean
 *     distance sum_d (m_pd - c_jd)^2, ties to the lower j;
 *   - the update: c_j = bf16 nearest-even of (the fp32 sum of its members'
 *     mean keys in page order) / (their count); a centroid left with no
 *     member keeps its value.
 * Both steps are decisions or stored codes, so they are taken in the
 * precision and order the GPU kernel uses: the distance accumulates
 * fmaf(x, x, acc) over d = 0 .. D-1 in fp32 with x = m_pd - c_jd, the sum
 * adds the members in page order in fp32, and the quotient is an fp32
 * division.  The search then scores the centroids like pages (q . c, the
 * group reduced by sum or max, in double), expands the M best centroids
 * (ties to the lower centroid) into their member pages, and keeps the K
 * best of those pages by their mean-key scores (ties to the lower page),
 * ascending.
 */
static void centroid_update(const uint16_t* mean, int32_t P, int32_t D, int32_t n_c, const int32_t* assign,
                            uint16_t* cent, int32_t* off, int32_t* members)
{
    for (int32_t j = 0; j <= n_c; ++j) off[j] = 0;
    for (int32_t p = 0; p < P; ++p) off[assign[p] + 1] += 1;
    for (int32_t j = 0; j < n_c; ++j) off[j + 1] += off[j];
    int32_t* fill = (int32_t*)malloc(sizeof(int32_t) * (size_t)(n_c > 0 ? n_c : 1));
    for (int32_t j = 0; j < n_c; ++j) fill[j] = off[j];
    for (int32_t p = 0; p < P; ++p) members[fill[assign[p]]++] = p; /* page order within a group */
    free(fill);
    for (int32_t j = 0; j < n_c; ++j) {
        const int32_t n = off[j + 1] - off[j];
        if (n == 0) continue; /* keeps its value */
        for (int32_t d = 0; d < D; ++d) {
            float acc = 0.0f;
            for (int32_t k = off[j]; k < off[j + 1]; ++k) acc += (float)bf16_value(mean[(int64_t)members[k] * D + d]);
            cent[(int64_t)j * D + d] = bf16_round_nearest_even(acc / (float)n);
        }
    }
}

static void centroid_assign(const uint16_t* mean, int32_t P, int32_t D, int32_t n_c, const uint16_t* cent,
                            int32_t* assign)
{
    for (int32_t p = 0; p < P; ++p) {
        float best = 0.0f;
        int32_t arg = 0;
        for (int32_t j = 0; j < n_c; ++j) {
            float acc = 0.0f;
            for (int32_t d = 0; d < D; ++d) {
                const float x = (float)bf16_value(mean[(int64_t)p * D + d]) - (float)bf16_value(cent[(int64_t)j * D + d]);
                acc = fmaf(x, x, acc);
            }
            if (j == 0 || acc < best) {
                best = acc;
                arg = j;
            }
        }
        assign[p] = arg;
    }
}

/* Builds a unit's centroids from its P pages' mean keys mean[P][D]: cent[n_c][D], assign[P], off[n_c + 1]
 * and members[P] (the pages of centroid j are members[off[j] .. off[j+1]), ascending).  Returns n_c. */
int32_t oracle_centroid_build(const uint16_t* mean, int32_t P, int32_t D, int32_t R, int32_t n_iter, uint16_t* cent,
                              int32_t* assign, int32_t* off, int32_t* members)
{
    const int32_t n_c = (P + R - 1) / R;
    for (int32_t p = 0; p < P; ++p) assign[p] = p / R; /* spatial blocks */
    centroid_update(mean, P, D, n_c, assign, cent, off, members);
    for (int32_t it = 0; it < n_iter; ++it) {
        centroid_assign(mean, P, D, n_c, cent, assign);
        centroid_update(mean, P, D, n_c, assign, cent, off, members);
    }
    return n_c;
}

/* The two-level search of one unit: centroid scores cs[n_c]; the M best centroids; their member pages
 * (cand[0 .. *n_cand), ascending; pages < P) with their mean-key scores ps[*n_cand]; the K best of those
 * pages into sel (ascending).  Returns the selection's size. */
int32_t oracle_centroid_select(const uint16_t* q, int32_t G, int32_t D, const uint16_t* mean, int32_t P,
                               const uint16_t* cent, int32_t n_c, const int32_t* off, const int32_t* members, int32_t M,
                               int32_t K, int32_t group_reduce, double* cs, int32_t* chosen, int32_t* cand,
                               int32_t* n_cand, double* ps, int32_t* sel)
{
    oracle_unit_mean_scores(q, G, D, cent, n_c, group_reduce, cs);
    const int32_t nm = oracle_topk(cs, n_c, M, chosen);
    uint8_t* take = (uint8_t*)calloc((size_t)(P > 0 ? P : 1), 1);
    for (int32_t i = 0; i < nm; ++i)
        for (int32_t k = off[chosen[i]]; k < off[chosen[i] + 1]; ++k) take[members[k]] = 1;
    int32_t n = 0;
    for (int32_t p = 0; p < P; ++p)
        if (take[p]) cand[n++] = p;
    free(take);
    *n_cand = n;
    uint16_t* rows = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)(n > 0 ? n : 1) * (size_t)D);
    for (int32_t i = 0; i < n; ++i) memcpy(rows + (int64_t)i * D, mean + (int64_t)cand[i] * D, sizeof(uint16_t) * (size_t)D);
    oracle_unit_mean_scores(q, G, D, rows, n, group_reduce, ps);
    free(rows);
    const int32_t cnt = oracle_topk(ps, n, K, sel); /* positions, ascending */
    for (int32_t i = 0; i < cnt; ++i) sel[i] = cand[sel[i]];
    return cnt;
}
