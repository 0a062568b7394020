/*
 * CPU oracle for query-aware (Quest-style) sparse decode attention over a
 * paged KV cache.  TEST INFRASTRUCTURE ONLY: the tests, the smoke check and
 * the benchmark's CPU-baseline leg are the only callers.  Nothing on the
 * product path links or calls this file, and it shares no code with the CUDA
 * library (its own bf16 helpers, its own loops).
 *
 * What it follows:
 *  - "add-sparse-method" skill page, "Placement Rules" 3-4: metadata is
 *    updated after KV is written (on_kv_stored), and the decode-time view is
 *    built from the current layer's q (build_decode_view).
 *  - SparseEngine summary page, section "method key points": Quest performs
 *    query-relevant page selection over per-method cache metadata, and the
 *    attention backend consumes the resulting view.
 *  - The method statement these pages leave open is fixed as follows: each
 *    page stores the per-channel min and max of its keys; a page's score is
 *    the upper bound sum_i max(q_i*kmax_i, q_i*kmin_i), summed over the query
 *    heads of one kv group; each (request, kv head) keeps its top-K pages,
 *    ties going to the lower page index; exact softmax attention runs over
 *    only those pages.
 *
 * Selection options (the pages describe none of them; the readings taken):
 *  - per_q_head: every query head selects its own pages by its own bound
 *    (no sum over the kv group); sel_idx then has one row per query head and
 *    each head attends only its row's pages.
 *  - sink_pages / window_pages: the first sink_pages and the last
 *    window_pages logical pages of a request are always kept.  They rank
 *    above every other page, among themselves by lower page index, and they
 *    count toward the budget K.
 *
 * FP8 pages (the pages name a quantized attention view but define no codec;
 * the reading taken): every (token, kv head) row of K and of V is stored as
 * 128 e4m3 codes and one fp32 scale s = amax(|row|) / 448; a value x is
 * coded as e4m3(x / s), rounded to nearest with ties to even and saturated
 * to +-448 (s = 0 and all codes 0 for an all-zero row); it decodes to
 * e4m3_value(code) * s.  The page metadata stays the bf16 min / max of the
 * keys as appended (before coding), so selection does not change.
 *
 * It is written literally: the score uses the max-form above (not any
 * rearrangement of it), ranking is a full sort, attention is two passes
 * over an explicit score vector.  Accumulation is fp32 in the loop order
 * written (heads, then channels; tokens in ascending page order).
 *
 * Layouts (bf16 values are passed as uint16 bit patterns):
 *   k_pool, v_pool  [n_phys][Hkv][P][D]
 *   meta            [n_phys][Hkv][2][D]   ([0] = kmin, [1] = kmax)
 *   q               [B][Hq][D]            query head h belongs to kv group h / (Hq/Hkv)
 *   page_table      [B][max_pages]        logical page -> physical page
 *   seq_lens        [B]
 *   sel_idx         [B][Hkv][K]           selected logical pages, ascending, -1 padded
 *   sel_cnt         [B][Hkv]
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Threads the row loops below may use: OpenMP's count in a -fopenmp build,
 * else 1. */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

static float bf16_bits_to_float(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return f;
}

/* Exact when f already holds a bf16 value (its low 16 bits are zero). */
static uint16_t float_to_bf16_bits_exact(float f) {
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/*
 * Append T tokens: copy each token's key and value row into its slot, then
 * recompute, from scratch, the key min/max of every page this call touched,
 * over that page's filled offsets [0, filled).  Pages fill in offset order
 * without holes, so a page's fill after this call is one past the largest
 * offset written to it here.
 */
int oracle_update_meta(uint16_t* k_pool, uint16_t* v_pool, uint16_t* meta,
                       int64_t n_phys, int Hkv, int P, int D,
                       const uint16_t* k_new, const uint16_t* v_new,
                       const int32_t* slot_mapping, int64_t T) {
    int32_t* fill = (int32_t*)calloc((size_t)n_phys, sizeof(int32_t));
    if (!fill) return -1;
    const size_t row = (size_t)D;
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t page = slot / P;
        int off = (int)(slot % P);
        if (slot < 0 || page >= n_phys) { free(fill); return -2; }
        for (int h = 0; h < Hkv; ++h) {
            size_t dst = (((size_t)page * Hkv + h) * P + off) * row;
            size_t src = ((size_t)t * Hkv + h) * row;
            memcpy(k_pool + dst, k_new + src, row * sizeof(uint16_t));
            memcpy(v_pool + dst, v_new + src, row * sizeof(uint16_t));
        }
        if (off + 1 > fill[page]) fill[page] = off + 1;
    }
    for (int64_t page = 0; page < n_phys; ++page) {
        int filled = fill[page];
        if (filled == 0) continue;
        for (int h = 0; h < Hkv; ++h) {
            uint16_t* mn = meta + (((size_t)page * Hkv + h) * 2 + 0) * row;
            uint16_t* mx = meta + (((size_t)page * Hkv + h) * 2 + 1) * row;
            for (int i = 0; i < D; ++i) {
                float lo = INFINITY, hi = -INFINITY;
                for (int o = 0; o < filled; ++o) {
                    float k = bf16_bits_to_float(k_pool[(((size_t)page * Hkv + h) * P + o) * row + i]);
                    if (k < lo) lo = k;
                    if (k > hi) hi = k;
                }
                mn[i] = float_to_bf16_bits_exact(lo);
                mx[i] = float_to_bf16_bits_exact(hi);
            }
        }
    }
    free(fill);
    return 0;
}

/*
 * Upper-bound score of one page for one kv group:
 *   s = sum over query heads h of the group, sum over channels i, of
 *       max(q[h][i] * kmax[i], q[h][i] * kmin[i]).
 */
static float page_bound(const uint16_t* q_group, int G, int D,
                        const uint16_t* kmin, const uint16_t* kmax) {
    float s = 0.0f;
    for (int h = 0; h < G; ++h) {
        for (int i = 0; i < D; ++i) {
            float qi = bf16_bits_to_float(q_group[(size_t)h * D + i]);
            float a = qi * bf16_bits_to_float(kmax[i]);
            float c = qi * bf16_bits_to_float(kmin[i]);
            s += (a > c) ? a : c;
        }
    }
    return s;
}

typedef struct {
    float score;
    int32_t page;
    int32_t forced;   /* 1: a sink or window page */
} scored_page;

/* Forced pages first, among themselves by lower index; then higher score first,
 * equal scores: lower logical page index first. */
static int by_score_then_index(const void* pa, const void* pb) {
    const scored_page* a = (const scored_page*)pa;
    const scored_page* b = (const scored_page*)pb;
    if (a->forced != b->forced) return a->forced ? -1 : 1;
    if (a->forced) return (a->page < b->page) ? -1 : (a->page > b->page);   /* forced: by index alone */
    if (a->score > b->score) return -1;
    if (a->score < b->score) return 1;
    return (a->page < b->page) ? -1 : (a->page > b->page);
}

static int by_int_ascending(const void* pa, const void* pb) {
    int32_t a = *(const int32_t*)pa, b = *(const int32_t*)pb;
    return (a < b) ? -1 : (a > b);
}

/*
 * For every request b and selection row r -- kv group r, or query head r when
 * per_q_head -- score each of the request's n_b = ceil(len_b / P) logical
 * pages with the bound of the row's query heads (the group's G heads, or the
 * one head) against the metadata of the row's kv head, keep the min(K, n_b)
 * first pages under the order (forced desc, score desc, page asc), and emit
 * their logical indices ascending.  R = per_q_head ? Hq : Hkv rows.
 * scores (nullable) receives [B][R][max_pages] fp32 (the bound, also for
 * forced pages), entries past n_b untouched.
 *
 * select_row computes one row (request b, row r); `list` holds max_pages
 * entries of scratch.
 */
static int select_row(const uint16_t* q, const uint16_t* meta, const int32_t* page_table,
                      const int32_t* seq_lens, int Hq, int Hkv, int D, int P, int max_pages, int K,
                      int64_t n_phys, int per_q_head, int sink_pages, int window_pages, int b, int r,
                      scored_page* list, int32_t* sel_idx, int32_t* sel_cnt, float* scores) {
    const int G = Hq / Hkv;
    const int R = per_q_head ? Hq : Hkv;
    int n = (seq_lens[b] + P - 1) / P;
    if (n < 1 || n > max_pages) return -2;
    const int g = per_q_head ? r / G : r;
    const int first_head = per_q_head ? r : g * G;
    const int heads = per_q_head ? 1 : G;
    const uint16_t* qr = q + ((size_t)b * Hq + (size_t)first_head) * D;
    for (int p = 0; p < n; ++p) {
        int64_t phys = page_table[(size_t)b * max_pages + p];
        if (phys < 0 || phys >= n_phys) return -2;
        const uint16_t* kmin = meta + (((size_t)phys * Hkv + g) * 2 + 0) * D;
        const uint16_t* kmax = meta + (((size_t)phys * Hkv + g) * 2 + 1) * D;
        list[p].score = page_bound(qr, heads, D, kmin, kmax);
        list[p].page = p;
        list[p].forced = (p < sink_pages || p >= n - window_pages) ? 1 : 0;
        if (scores) scores[((size_t)b * R + r) * max_pages + p] = list[p].score;
    }
    qsort(list, (size_t)n, sizeof(scored_page), by_score_then_index);
    int m = n < K ? n : K;
    int32_t* out = sel_idx + ((size_t)b * R + r) * K;
    for (int j = 0; j < m; ++j) out[j] = list[j].page;
    qsort(out, (size_t)m, sizeof(int32_t), by_int_ascending);
    for (int j = m; j < K; ++j) out[j] = -1;
    sel_cnt[(size_t)b * R + r] = m;
    return 0;
}

/* Rows are independent: a build with OpenMP (-fopenmp) hands them to the
 * host's threads, each with its own scratch; without it the loop runs in
 * order on one thread.  Either way every row is computed by select_row alone.
 */
int oracle_select_ex(const uint16_t* q, const uint16_t* meta,
                     const int32_t* page_table, const int32_t* seq_lens,
                     int B, int Hq, int Hkv, int D, int P, int max_pages, int K,
                     int64_t n_phys, int per_q_head, int sink_pages, int window_pages,
                     int32_t* sel_idx, int32_t* sel_cnt, float* scores) {
    if (Hq % Hkv != 0 || K < 1 || sink_pages < 0 || window_pages < 0) return -1;
    const int R = per_q_head ? Hq : Hkv;
    const int64_t rows = (int64_t)B * R;
    int rc = 0;
#pragma omp parallel
    {
        scored_page* list = (scored_page*)malloc((size_t)max_pages * sizeof(scored_page));
#pragma omp for schedule(dynamic, 1)
        for (int64_t row = 0; row < rows; ++row) {
            int e = list ? select_row(q, meta, page_table, seq_lens, Hq, Hkv, D, P, max_pages, K, n_phys,
                                      per_q_head, sink_pages, window_pages, (int)(row / R), (int)(row % R), list,
                                      sel_idx, sel_cnt, scores)
                         : -1;
            if (e) {
#pragma omp atomic write
                rc = e;
            }
        }
        free(list);
    }
    return rc;
}

/*
 * The selection step alone, on given scores: for each of the rows, keep the
 * min(K, n_pages[row]) pages of scores[row][0 .. n) that come first under
 * (score desc, page asc) -- the order oracle_select_ex uses, with no forced
 * pages -- and emit their indices ascending, padded with -1.
 */
int oracle_topk(const float* scores, const int32_t* n_pages, int rows, int max_pages, int K,
                int32_t* sel_idx, int32_t* sel_cnt) {
    if (K < 1 || rows < 0 || max_pages < 1) return -1;
    scored_page* list = (scored_page*)malloc((size_t)max_pages * sizeof(scored_page));
    if (!list) return -1;
    for (int r = 0; r < rows; ++r) {
        const int n = n_pages[r];
        if (n < 0 || n > max_pages) { free(list); return -2; }
        for (int p = 0; p < n; ++p) {
            list[p].score = scores[(size_t)r * max_pages + p];
            list[p].page = p;
            list[p].forced = 0;
        }
        qsort(list, (size_t)n, sizeof(scored_page), by_score_then_index);
        const int m = n < K ? n : K;
        int32_t* out = sel_idx + (size_t)r * K;
        for (int j = 0; j < m; ++j) out[j] = list[j].page;
        qsort(out, (size_t)m, sizeof(int32_t), by_int_ascending);
        for (int j = m; j < K; ++j) out[j] = -1;
        sel_cnt[r] = m;
    }
    free(list);
    return 0;
}

/* The base method: one row per kv group, no forced pages. */
int oracle_select(const uint16_t* q, const uint16_t* meta,
                  const int32_t* page_table, const int32_t* seq_lens,
                  int B, int Hq, int Hkv, int D, int P, int max_pages, int K,
                  int64_t n_phys, int32_t* sel_idx, int32_t* sel_cnt, float* scores) {
    return oracle_select_ex(q, meta, page_table, seq_lens, B, Hq, Hkv, D, P, max_pages, K, n_phys, 0, 0, 0,
                            sel_idx, sel_cnt, scores);
}

/*
 * Exact softmax attention of every query head over the tokens of a page
 * list: all n_b logical pages when sel_idx is NULL (dense), else the
 * sel_cnt[b][r] pages of sel_idx[b][r], r = the head's kv group g, or the
 * head itself when per_q_head (sel_idx then has Hq rows per request).  The last logical page n_b - 1 holds
 * len_b - P*(n_b - 1) tokens; every other page holds P.
 *   z_t = (q . k_t) * scale;  m = max z;  l = sum exp(z - m);
 *   out = sum exp(z_t - m) v_t / l;  lse = m + ln(l).
 * out is fp32 [B][Hq][D]; lse fp32 [B][Hq].
 */
/* One query head (request b, head h) of oracle_decode_ex; z, tok_page and
 * tok_off hold max_pages * P entries of scratch. */
static int decode_head(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                       const int32_t* page_table, const int32_t* seq_lens, int Hq, int Hkv, int D, int P,
                       int max_pages, int64_t n_phys, const int32_t* sel_idx, const int32_t* sel_cnt, int K,
                       int per_q_head, float scale, int b, int h, float* z, int32_t* tok_page, int32_t* tok_off,
                       float* out, float* lse) {
    const int G = Hq / Hkv;
    const int R = per_q_head ? Hq : Hkv;
    int len = seq_lens[b];
    int n = (len + P - 1) / P;
    if (n < 1 || n > max_pages) return -2;
    int g = h / G;
    int r = per_q_head ? h : g;
    int count = sel_idx ? sel_cnt[(size_t)b * R + r] : n;
    if (count < 0 || count > (sel_idx ? K : n)) return -2;
    /* Gather the attended tokens as (physical page, offset). */
    int ntok = 0;
    for (int j = 0; j < count; ++j) {
        int p = sel_idx ? sel_idx[((size_t)b * R + r) * K + j] : j;
        if (p < 0 || p >= n) return -2;
        int64_t phys = page_table[(size_t)b * max_pages + p];
        if (phys < 0 || phys >= n_phys) return -2;
        int valid = (p == n - 1) ? len - P * (n - 1) : P;
        for (int o = 0; o < valid; ++o) {
            tok_page[ntok] = (int32_t)phys;
            tok_off[ntok] = o;
            ++ntok;
        }
    }
    const uint16_t* qh = q + ((size_t)b * Hq + h) * D;
    float* o_row = out + ((size_t)b * Hq + h) * D;
    float m = -INFINITY;
    for (int t = 0; t < ntok; ++t) {
        const uint16_t* k = k_pool + (((size_t)tok_page[t] * Hkv + g) * P + tok_off[t]) * D;
        float dot = 0.0f;
        for (int i = 0; i < D; ++i) dot += bf16_bits_to_float(qh[i]) * bf16_bits_to_float(k[i]);
        z[t] = dot * scale;
        if (z[t] > m) m = z[t];
    }
    float l = 0.0f;
    for (int i = 0; i < D; ++i) o_row[i] = 0.0f;
    for (int t = 0; t < ntok; ++t) {
        float w = expf(z[t] - m);
        l += w;
        const uint16_t* v = v_pool + (((size_t)tok_page[t] * Hkv + g) * P + tok_off[t]) * D;
        for (int i = 0; i < D; ++i) o_row[i] += w * bf16_bits_to_float(v[i]);
    }
    if (ntok == 0) {
        lse[(size_t)b * Hq + h] = -INFINITY;
        return 0;
    }
    for (int i = 0; i < D; ++i) o_row[i] /= l;
    lse[(size_t)b * Hq + h] = m + logf(l);
    return 0;
}

/*
 * Exact softmax attention of every query head over the tokens of a page
 * list: all n_b logical pages when sel_idx is NULL (dense), else the
 * sel_cnt[b][r] pages of sel_idx[b][r], r = the head's kv group g, or the
 * head itself when per_q_head (sel_idx then has Hq rows per request).  The last logical page n_b - 1 holds
 * len_b - P*(n_b - 1) tokens; every other page holds P.
 *   z_t = (q . k_t) * scale;  m = max z;  l = sum exp(z - m);
 *   out = sum exp(z_t - m) v_t / l;  lse = m + ln(l).
 * out is fp32 [B][Hq][D]; lse fp32 [B][Hq].  Heads are independent: an
 * OpenMP build hands them to the host's threads (each with its own scratch),
 * a plain build runs them in order; each head is computed by decode_head alone.
 */
int oracle_decode_ex(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                     const int32_t* page_table, const int32_t* seq_lens,
                     int B, int Hq, int Hkv, int D, int P, int max_pages, int64_t n_phys,
                     const int32_t* sel_idx, const int32_t* sel_cnt, int K, int per_q_head, float scale,
                     float* out, float* lse) {
    if (Hq % Hkv != 0) return -1;
    const int64_t heads = (int64_t)B * Hq;
    int rc = 0;
#pragma omp parallel
    {
        float* z = (float*)malloc((size_t)max_pages * P * sizeof(float));
        int32_t* tok_page = (int32_t*)malloc((size_t)max_pages * P * sizeof(int32_t));
        int32_t* tok_off = (int32_t*)malloc((size_t)max_pages * P * sizeof(int32_t));
        const int ok = z && tok_page && tok_off;
#pragma omp for schedule(dynamic, 1)
        for (int64_t bh = 0; bh < heads; ++bh) {
            int e = ok ? decode_head(q, k_pool, v_pool, page_table, seq_lens, Hq, Hkv, D, P, max_pages, n_phys,
                                     sel_idx, sel_cnt, K, per_q_head, scale, (int)(bh / Hq), (int)(bh % Hq), z,
                                     tok_page, tok_off, out, lse)
                       : -1;
            if (e) {
#pragma omp atomic write
                rc = e;
            }
        }
        free(z);
        free(tok_page);
        free(tok_off);
    }
    return rc;
}

/* The base method: one selection row per kv group. */
int oracle_decode(const uint16_t* q, const uint16_t* k_pool, const uint16_t* v_pool,
                  const int32_t* page_table, const int32_t* seq_lens,
                  int B, int Hq, int Hkv, int D, int P, int max_pages, int64_t n_phys,
                  const int32_t* sel_idx, const int32_t* sel_cnt, int K, float scale,
                  float* out, float* lse) {
    return oracle_decode_ex(q, k_pool, v_pool, page_table, seq_lens, B, Hq, Hkv, D, P, max_pages, n_phys,
                            sel_idx, sel_cnt, K, 0, scale, out, lse);
}

/* ---------------------------------------------------------------- FP8 (e4m3) pages
 * e4m3: sign bit, 4 exponent bits with bias 7, 3 mantissa bits; exponent 0
 * holds the subnormals m * 2^-9; codes 0x7F / 0xFF are NaN; there are no
 * infinities; the largest finite value is 0x7E = 448. */
float oracle_e4m3_value(uint8_t c) {
    const int sgn = c >> 7, e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const float v = (e == 0) ? ldexpf((float)m, -9) : ldexpf((float)(8 + m), e - 10);
    return sgn ? -v : v;
}

/* Nearest e4m3 value, ties to the even code, saturating to +-448; NaN -> 0x7F. */
uint8_t oracle_e4m3_encode(float x) {
    if (isnan(x)) return 0x7F;
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    float a = fabsf(x);
    if (a >= 448.0f) return sgn | 0x7E;
    if (a == 0.0f) return sgn;
    /* Spacing of e4m3 values around a: 2^(E - 3) for a in [2^E, 2^(E+1)),
     * E >= -6; 2^-9 below 2^-6 (subnormals). */
    int E = ilogbf(a);
    if (E < -6) E = -6;
    const int qe = E - 3;
    const float r = rintf(ldexpf(a, -qe));     /* integer multiple of the spacing; rintf rounds half to even */
    const float v = ldexpf(r, qe);             /* exact e4m3 value (r = 16 carries into the next binade) */
    if (v >= 448.0f) return sgn | 0x7E;
    if (v == 0.0f) return sgn;
    int ev = ilogbf(v);
    if (ev < -6) return sgn | (uint8_t)ldexpf(v, 9);                 /* subnormal: m = v * 2^9 */
    const int m = (int)ldexpf(v, 3 - ev) - 8;                         /* v = (8 + m) * 2^(ev - 3) */
    return sgn | (uint8_t)(((ev + 7) << 3) | m);
}

/*
 * Codes and scales of T appended tokens into FP8 pools at their slots:
 *   k8, v8  [n_phys][Hkv][P][D] e4m3 codes;  ks, vs  [n_phys][Hkv][P] fp32 scales.
 * (The bf16 rows and the metadata go through oracle_update_meta.)
 */
int oracle_quantize_rows(uint8_t* k8, uint8_t* v8, float* ks, float* vs,
                         int64_t n_phys, int Hkv, int P, int D,
                         const uint16_t* k_new, const uint16_t* v_new,
                         const int32_t* slot_mapping, int64_t T) {
    for (int64_t t = 0; t < T; ++t) {
        int64_t slot = slot_mapping[t];
        int64_t page = slot / P;
        int off = (int)(slot % P);
        if (slot < 0 || page >= n_phys) return -2;
        for (int h = 0; h < Hkv; ++h) {
            for (int which = 0; which < 2; ++which) {
                const uint16_t* src = (which ? v_new : k_new) + ((size_t)t * Hkv + h) * D;
                uint8_t* dst = (which ? v8 : k8) + (((size_t)page * Hkv + h) * P + off) * D;
                float* sc = (which ? vs : ks) + ((size_t)page * Hkv + h) * P + off;
                float amax = 0.0f;
                for (int i = 0; i < D; ++i) {
                    float a = fabsf(bf16_bits_to_float(src[i]));
                    if (a > amax) amax = a;
                }
                const float scale = amax / 448.0f;
                *sc = scale;
                for (int i = 0; i < D; ++i)
                    dst[i] = scale > 0.0f ? oracle_e4m3_encode(bf16_bits_to_float(src[i]) / scale) : 0;
            }
        }
    }
    return 0;
}

/*
 * oracle_decode over FP8 pages: key and value elements are
 * e4m3_value(code) * scale of their row (fp32), otherwise as oracle_decode_ex.
 */
int oracle_decode_fp8(const uint16_t* q, const uint8_t* k8, const uint8_t* v8, const float* ks, const float* vs,
                      const int32_t* page_table, const int32_t* seq_lens,
                      int B, int Hq, int Hkv, int D, int P, int max_pages, int64_t n_phys,
                      const int32_t* sel_idx, const int32_t* sel_cnt, int K, int per_q_head, float scale,
                      float* out, float* lse) {
    if (Hq % Hkv != 0) return -1;
    const int G = Hq / Hkv;
    const int R = per_q_head ? Hq : Hkv;
    float* z = (float*)malloc((size_t)max_pages * P * sizeof(float));
    int64_t* tok_row = (int64_t*)malloc((size_t)max_pages * P * sizeof(int64_t));
    if (!z || !tok_row) { free(z); free(tok_row); return -1; }
    int rc = 0;
    for (int b = 0; b < B && rc == 0; ++b) {
        int len = seq_lens[b];
        int n = (len + P - 1) / P;
        if (n < 1 || n > max_pages) { rc = -2; break; }
        for (int h = 0; h < Hq && rc == 0; ++h) {
            int g = h / G;
            int r = per_q_head ? h : g;
            int count = sel_idx ? sel_cnt[(size_t)b * R + r] : n;
            if (count < 0 || count > (sel_idx ? K : n)) { rc = -2; break; }
            int ntok = 0;   /* attended tokens as row indices into [n_phys][Hkv][P] */
            for (int j = 0; j < count; ++j) {
                int p = sel_idx ? sel_idx[((size_t)b * R + r) * K + j] : j;
                if (p < 0 || p >= n) { rc = -2; break; }
                int64_t phys = page_table[(size_t)b * max_pages + p];
                if (phys < 0 || phys >= n_phys) { rc = -2; break; }
                int valid = (p == n - 1) ? len - P * (n - 1) : P;
                for (int o = 0; o < valid; ++o) tok_row[ntok++] = (phys * Hkv + g) * P + o;
            }
            if (rc) break;
            const uint16_t* qh = q + ((size_t)b * Hq + h) * D;
            float* o_row = out + ((size_t)b * Hq + h) * D;
            float m = -INFINITY;
            for (int t = 0; t < ntok; ++t) {
                const uint8_t* k = k8 + (size_t)tok_row[t] * D;
                float dot = 0.0f;
                for (int i = 0; i < D; ++i) dot += bf16_bits_to_float(qh[i]) * (oracle_e4m3_value(k[i]) * ks[tok_row[t]]);
                z[t] = dot * scale;
                if (z[t] > m) m = z[t];
            }
            float l = 0.0f;
            for (int i = 0; i < D; ++i) o_row[i] = 0.0f;
            for (int t = 0; t < ntok; ++t) {
                float w = expf(z[t] - m);
                l += w;
                const uint8_t* v = v8 + (size_t)tok_row[t] * D;
                for (int i = 0; i < D; ++i) o_row[i] += w * (oracle_e4m3_value(v[i]) * vs[tok_row[t]]);
            }
            if (ntok == 0) {
                lse[(size_t)b * Hq + h] = -INFINITY;
                continue;
            }
            for (int i = 0; i < D; ++i) o_row[i] /= l;
            lse[(size_t)b * Hq + h] = m + logf(l);
        }
    }
    free(z);
    free(tok_row);
    return rc;
}
