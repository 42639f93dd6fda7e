/*
 * oracle.c -- plain, slow CPU reference of the batched speculative-decoding verify
 * step. TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the CPU-baseline
 * leg of the benchmark call it; the product path never does.
 *
 * Everything is computed in fp64 with straight loops in the order the definitions
 * are written, so that each function can be checked against its source by eye.
 * Nothing here is shared with the CUDA library: no header, helper or table.
 * The only parallelism is an OpenMP loop over independent (row, head) items, which
 * changes no arithmetic.
 *
 * Sources (web pages; function or section named on each):
 *  - span-02 `engine/crates/model/src/spec.rs`: module documentation (verify of B
 *    branches with KV appended in place at pos..pos+k, emit only on equality with
 *    the argmax of the row before, rollback = advancing pos, kv_hi = position),
 *    `SpecReq` (page of position p is pages[p / page_size]), `greedy_logprob`
 *    (first maximum wins), `Spec::body_inner` (step order).
 *  - memra-engine 0.70.0 `src/spec.rs`, `full_attn_verify`: row r attends keys
 *    [0, base_len + r + 1).
 *  - DSSD-dev `dssd/fast.py`, `_attention` (CPU reference: SDPA per row over its exact
 *    key list, GQA by consecutive grouping) and `generate_spec` (accept loop, then the
 *    correction / bonus token target[len(committed)]).
 *  - oxinfer 0.0.5 `src/qwen_mtp.rs`: module documentation (x = fc([rmsnorm_emb(embed
 *    (x_{i+1})), rmsnorm_hidden(h_i)]), fc [H, 2H], embedding first) and
 *    `speculative_accept` (greedy case: accept iff the draft is the argmax).
 *  - OCP 8-bit floating point specification, E4M3 (bias 7, max 448, no infinities,
 *    S.1111.111 is NaN, subnormals m * 2^-9): the FP8 page format.
 *
 * Readings where the pages are silent (all listed in the design notes):
 *  - pos[b] is the position of the branch's first verify row = committed tokens.
 *  - KV page layout [num_pages][Hkv][page_size][d]; q head h uses kv head h / G.
 *  - FP8: code = e4m3(float(x) / scale) with IEEE fp32 division, round to nearest
 *    even, saturating to +-448 (satfinite); value = decode(code) * scale.
 *  - The argmax decision is taken on the fp32-rounded logit (the pages' argmax runs
 *    on fp32 logits, flashrt-structures whole_step.py `generate_speculative`).
 *  - MTP concat halves are rounded to bf16 before fc; x is rounded to bf16.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_ERR_PAGE 1
#define ORC_ERR_COVER 2
#define ORC_ERR_TOKEN 4
#define ORC_ERR_D2T 8
#define ORC_ERR_POS 16
#define ORC_ERR_TREE 32
#define ORC_ERR_SLOT 64

int orc_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_threads(int n) {
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* ------------------------------------------------------------------------------------
 * Number formats
 * ---------------------------------------------------------------------------------- */

/* bfloat16 -> double: the 16 bits are the top half of an IEEE binary32. */
double orc_bf16_to_double(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* double -> bfloat16, round to nearest, ties to even, written from the definition:
 * find the two neighbouring bf16 values and pick the nearer (even one on a tie).
 * NaN -> canonical quiet NaN 0x7FC0; overflow rounds to +-inf as IEEE does. */
uint16_t orc_double_to_bf16(double x) {
    if (isnan(x)) return 0x7FC0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (a == 0.0) return sign;
    if (isinf(a)) return sign | 0x7F80;
    /* bf16: 8 exponent bits (bias 127), 7 stored mantissa bits. */
    int e;
    frexp(a, &e);              /* a = f * 2^e, f in [0.5, 1) -> unbiased exponent e-1 */
    int ue = e - 1;
    if (ue < -126) ue = -126;  /* subnormal range shares the quantum of 2^-126 */
    double quantum = ldexp(1.0, ue - 7);
    double lo = floor(a / quantum) * quantum;  /* exact: a/quantum is a power-of-two scaling */
    double hi = lo + quantum;
    double r;
    if (a - lo < hi - a) r = lo;
    else if (a - lo > hi - a) r = hi;
    else r = (fmod(lo / quantum, 2.0) == 0.0) ? lo : hi;
    if (r >= ldexp(1.0, 128)) return sign | 0x7F80;
    float f = (float)r;        /* exact: r has at most 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, 4);
    return (uint16_t)(sign | ((u >> 16) & 0x7FFF));
}

/* E4M3 code -> value (OCP FP8: sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent 0 is subnormal m/8 * 2^-6; S.1111.111 is NaN; no infinities). */
double orc_e4m3_decode(uint8_t c) {
    int s = (c >> 7) & 1, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return NAN;
    if (e == 0) v = ldexp((double)m / 8.0, -6);
    else v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return s ? -v : v;
}

/* fp32 value -> E4M3 code, round to nearest even, saturating to the largest finite
 * magnitude 448 (the "satfinite" behaviour); NaN -> 0x7F. Written as a search over the
 * 127 non-negative finite codes, whose values increase with the code: find the largest
 * code whose value is <= |x| (binary search), then the nearer of it and its successor
 * wins, a tie going to the even code (mantissa LSB 0). */
uint8_t orc_e4m3_encode(float xf) {
    double x = (double)xf;
    if (isnan(x)) return 0x7F;
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs(x);
    if (a >= 448.0) return sign | 0x7E;
    int lo_c = 0, hi_c = 0x7E;          /* invariant: value(lo_c) <= a < value(hi_c) */
    while (hi_c - lo_c > 1) {
        int mid = (lo_c + hi_c) / 2;
        if (orc_e4m3_decode((uint8_t)mid) <= a) lo_c = mid;
        else hi_c = mid;
    }
    int best = lo_c;
    double lo = orc_e4m3_decode((uint8_t)best);
    if (lo == a) return sign | (uint8_t)best;
    double hi = orc_e4m3_decode((uint8_t)(best + 1));
    int pick;
    if (a - lo < hi - a) pick = best;
    else if (a - lo > hi - a) pick = best + 1;
    else pick = (best % 2 == 0) ? best : best + 1;
    return sign | (uint8_t)pick;
}

/* ------------------------------------------------------------------------------------
 * Paged KV pool
 * ---------------------------------------------------------------------------------- */

typedef struct {
    void *k_pool, *v_pool;            /* uint16 bf16 bits or uint8 E4M3 codes */
    const float *k_scale, *v_scale;   /* [num_pages][Hkv] (FP8 only) */
    const int32_t *page_table;        /* [B][max_pages] */
    int32_t num_pages, max_pages, page_size, n_kv_heads, head_dim, kv_dtype;
} orc_kv;

static size_t pool_index(const orc_kv *kv, int page, int g, int slot) {
    return (((size_t)page * kv->n_kv_heads + g) * kv->page_size + slot) * kv->head_dim;
}

/* Resolve position p of page-table row b to (page, slot). Returns an error bit or 0. */
static int locate(const orc_kv *kv, int b, int p, int *page, int *slot) {
    if (p < 0) return ORC_ERR_POS;
    int pi = p / kv->page_size;
    if (pi >= kv->max_pages) return ORC_ERR_COVER;
    int pg = kv->page_table[(size_t)b * kv->max_pages + pi];
    if (pg < 0 || pg >= kv->num_pages) return ORC_ERR_PAGE;
    *page = pg;
    *slot = p % kv->page_size;
    return 0;
}

/* Write n_rows K/V rows; row i goes to page-table row row_branch[i] at position
 * row_pos[i] (span-02 spec.rs, `SpecReq`: "its KV slot is page pages[pos / 16]").
 * bf16 pool: bit copy. FP8 pool: code = e4m3(float(x) / scale[page][g]).
 * Returns the OR of the error bits of skipped rows. Rows must name distinct positions. */
int orc_kv_write_rows(const orc_kv *kv, const int32_t *row_branch, const int32_t *row_pos,
                      int n_rows, const uint16_t *k_rows, const uint16_t *v_rows) {
    int err = 0;
    const int Hkv = kv->n_kv_heads, d = kv->head_dim;
    /* rows are independent (they target distinct positions) */
#pragma omp parallel for schedule(static) reduction(| : err)
    for (int i = 0; i < n_rows; ++i) {
        int page, slot;
        int e = locate(kv, row_branch[i], row_pos[i], &page, &slot);
        if (e) { err |= e; continue; }
        for (int g = 0; g < Hkv; ++g) {
            const uint16_t *ks = k_rows + ((size_t)i * Hkv + g) * d;
            const uint16_t *vs = v_rows + ((size_t)i * Hkv + g) * d;
            size_t dst = pool_index(kv, page, g, slot);
            if (kv->kv_dtype == 0) {
                memcpy((uint16_t *)kv->k_pool + dst, ks, (size_t)d * 2);
                memcpy((uint16_t *)kv->v_pool + dst, vs, (size_t)d * 2);
            } else {
                float sk = kv->k_scale[(size_t)page * Hkv + g];
                float sv = kv->v_scale[(size_t)page * Hkv + g];
                for (int c = 0; c < d; ++c) {
                    float xk = (float)orc_bf16_to_double(ks[c]);
                    float xv = (float)orc_bf16_to_double(vs[c]);
                    ((uint8_t *)kv->k_pool)[dst + c] = orc_e4m3_encode(xk / sk);
                    ((uint8_t *)kv->v_pool)[dst + c] = orc_e4m3_encode(xv / sv);
                }
            }
        }
    }
    return err;
}

/* The verify-step append: branch b's k+1 new rows go to positions pos[b]..pos[b]+k
 * (span-02 spec.rs, module documentation). Row r = b*(k+1)+j. */
int orc_kv_append(const orc_kv *kv, const int32_t *pos, int B, int k,
                  const uint16_t *k_new, const uint16_t *v_new) {
    int R = B * (k + 1);
    int32_t *rb = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    int32_t *rp = (int32_t *)malloc(sizeof(int32_t) * (size_t)(R > 0 ? R : 1));
    for (int b = 0; b < B; ++b)
        for (int j = 0; j <= k; ++j) {
            rb[b * (k + 1) + j] = b;
            rp[b * (k + 1) + j] = pos[b] + j;
        }
    int err = orc_kv_write_rows(kv, rb, rp, R, k_new, v_new);
    free(rb);
    free(rp);
    return err;
}

/* Value of element c of (page, kv head g, slot) in the K (which=0) or V (1) pool. */
static double kv_value(const orc_kv *kv, int which, int page, int g, int slot, int c) {
    size_t i = pool_index(kv, page, g, slot) + c;
    if (kv->kv_dtype == 0) {
        const uint16_t *pool = (const uint16_t *)(which ? kv->v_pool : kv->k_pool);
        return orc_bf16_to_double(pool[i]);
    }
    const uint8_t *pool = (const uint8_t *)(which ? kv->v_pool : kv->k_pool);
    const float *sc = which ? kv->v_scale : kv->k_scale;
    return orc_e4m3_decode(pool[i]) * (double)sc[(size_t)page * kv->n_kv_heads + g];
}

/* ------------------------------------------------------------------------------------
 * Verify attention
 * ---------------------------------------------------------------------------------- */

/* One output vector: row r of branch b at position p, q head h.
 *   s_t = scale * sum_c q[c] * K_t[c],  t = 0..p   (keys of branch b, kv head h/G)
 *   o   = sum_t exp(s_t - max s) V_t / sum_t exp(s_t - max s)
 * memra-engine spec.rs `full_attn_verify`: row r sees keys [0, base_len + r + 1);
 * span-02 spec.rs: kv_hi = position. Returns an error bit or 0. */
static int attn_one(const orc_kv *kv, int b, int p, int g, const uint16_t *q, double scale,
                    double *o, double *s /* scratch [p+1] */) {
    const int d = kv->head_dim;
    double mx = -INFINITY;
    for (int t = 0; t <= p; ++t) {
        int page, slot;
        int e = locate(kv, b, t, &page, &slot);
        if (e) return e;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += orc_bf16_to_double(q[c]) * kv_value(kv, 0, page, g, slot, c);
        s[t] = scale * dot;
        if (s[t] > mx) mx = s[t];
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    double den = 0.0;
    for (int t = 0; t <= p; ++t) {
        int page, slot;
        locate(kv, b, t, &page, &slot);
        double w = exp(s[t] - mx);
        den += w;
        for (int c = 0; c < d; ++c) o[c] += w * kv_value(kv, 1, page, g, slot, c);
    }
    for (int c = 0; c < d; ++c) o[c] /= den;
    return 0;
}

/* All R = B*(k+1) rows x Hq heads. q bf16 [R][Hq][d]; out fp64 [R][Hq][d].
 * Row r = b*(k+1)+j sits at position pos[b]+j. Rows whose key path hits a bad page
 * are left as NaN and reported. */
int orc_verify_attn(const orc_kv *kv, const int32_t *pos, int B, int k, int n_q_heads,
                    const uint16_t *q, double scale, double *out) {
    const int d = kv->head_dim, Hq = n_q_heads, G = n_q_heads / kv->n_kv_heads;
    const int R = B * (k + 1);
    int err = 0;
    int maxp = 0;
    for (int b = 0; b < B; ++b)
        if (pos[b] + k + 1 > maxp) maxp = pos[b] + k + 1;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int item = 0; item < R * Hq; ++item) {
        int r = item / Hq, h = item % Hq, b = r / (k + 1), j = r % (k + 1);
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxp + 1));
        double *o = out + ((size_t)r * Hq + h) * d;
        int e = (pos[b] < 0) ? ORC_ERR_POS
                             : attn_one(kv, b, pos[b] + j, h / G, q + ((size_t)r * Hq + h) * d, scale, o, s);
        if (e) {
            for (int c = 0; c < d; ++c) o[c] = NAN;
            err |= e;
        }
        free(s);
    }
    return err;
}

/* ---- tree / star verify (a next row) -------------------------------------------------
 * DSSD-dev `_set_rows` / `_star_cycle`: a tree row reads the contiguous committed prefix
 * (keys t < cl at their own index) and then the slots of its own path; chains are the case
 * slot = position. Here the k+1 verify rows of branch b own the slots pos_b .. pos_b+k
 * (row j writes slot pos_b+j), and row j's path is given as a bit mask over them:
 * anc_mask[b][j] bit i set = row j reads slot pos_b+i (its ancestors and itself). Keys
 * are visited in ascending slot order, as in attn_one; a chain's masks (bits 0..j) give
 * attn_one's key set exactly. */
static int attn_keys(const orc_kv *kv, int b, const int32_t *keys, int n_keys, int g, const uint16_t *q,
                     double scale, double *o, double *s) {
    const int d = kv->head_dim;
    double mx = -INFINITY;
    for (int i = 0; i < n_keys; ++i) {
        int page, slot;
        int e = locate(kv, b, keys[i], &page, &slot);
        if (e) return e;
        double dot = 0.0;
        for (int c = 0; c < d; ++c) dot += orc_bf16_to_double(q[c]) * kv_value(kv, 0, page, g, slot, c);
        s[i] = scale * dot;
        if (s[i] > mx) mx = s[i];
    }
    for (int c = 0; c < d; ++c) o[c] = 0.0;
    double den = 0.0;
    for (int i = 0; i < n_keys; ++i) {
        int page, slot;
        locate(kv, b, keys[i], &page, &slot);
        double w = exp(s[i] - mx);
        den += w;
        for (int c = 0; c < d; ++c) o[c] += w * kv_value(kv, 1, page, g, slot, c);
    }
    for (int c = 0; c < d; ++c) o[c] /= den;
    return 0;
}

int orc_verify_attn_tree(const orc_kv *kv, const int32_t *pos, int B, int k, int n_q_heads,
                         const uint16_t *q, double scale, const int32_t *anc_mask, double *out) {
    const int d = kv->head_dim, Hq = n_q_heads, G = n_q_heads / kv->n_kv_heads;
    const int R = B * (k + 1);
    int err = 0;
    int maxp = 0;
    for (int b = 0; b < B; ++b)
        if (pos[b] + k + 1 > maxp) maxp = pos[b] + k + 1;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int item = 0; item < R * Hq; ++item) {
        int r = item / Hq, h = item % Hq, b = r / (k + 1);
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxp + 1));
        int32_t *keys = (int32_t *)malloc(sizeof(int32_t) * (size_t)(maxp + 1));
        double *o = out + ((size_t)r * Hq + h) * d;
        /* row j of a branch is a tree node: it sees itself and only earlier rows (its
         * ancestors), so bit j is set and no bit above j */
        const int j = r % (k + 1);
        const uint32_t m = (uint32_t)anc_mask[r];
        int e = pos[b] < 0 ? ORC_ERR_POS : 0, n = 0;
        if (!((m >> j) & 1u) || ((m >> j) >> 1) != 0) e |= ORC_ERR_TREE;
        if (!e) {
            for (int t = 0; t < pos[b]; ++t) keys[n++] = t;
            for (int i = 0; i <= k; ++i)
                if ((anc_mask[r] >> i) & 1) keys[n++] = pos[b] + i;
            e = n ? attn_keys(kv, b, keys, n, h / G, q + ((size_t)r * Hq + h) * d, scale, o, s) : ORC_ERR_POS;
        }
        if (e) {
            for (int c = 0; c < d; ++c) o[c] = NAN;
            err |= e;
        }
        free(keys);
        free(s);
    }
    return err;
}

/* A chosen subset of (row, head) outputs, for full-size checks:
 * items[i] = r * Hq + h; out fp64 [n_items][d]. */
int orc_verify_attn_items(const orc_kv *kv, const int32_t *pos, int B, int k, int n_q_heads,
                          const uint16_t *q, double scale, const int32_t *items, int n_items,
                          double *out) {
    const int d = kv->head_dim, Hq = n_q_heads, G = n_q_heads / kv->n_kv_heads;
    int err = 0;
    int maxp = 0;
    for (int b = 0; b < B; ++b)
        if (pos[b] + k + 1 > maxp) maxp = pos[b] + k + 1;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int i = 0; i < n_items; ++i) {
        int r = items[i] / Hq, h = items[i] % Hq, b = r / (k + 1), j = r % (k + 1);
        double *s = (double *)malloc(sizeof(double) * (size_t)(maxp + 1));
        double *o = out + (size_t)i * d;
        int e = attn_one(kv, b, pos[b] + j, h / G, q + ((size_t)r * Hq + h) * d, scale, o, s);
        if (e) {
            for (int c = 0; c < d; ++c) o[c] = NAN;
            err |= e;
        }
        free(s);
    }
    (void)B;
    return err;
}

/* ------------------------------------------------------------------------------------
 * LM head with argmax
 * ---------------------------------------------------------------------------------- */

/* Row m: logit[v] = sum_h hidden[m][h] * W[v][h] in fp64 (every bf16 x bf16 product is
 * exact in fp64); the decision is taken on the fp32-rounded logits: the id is the
 * first v whose logit is strictly greater than every earlier one (span-02 spec.rs,
 * `greedy_logprob`: first maximum). With d2t the id becomes d2t[id] (oxinfer
 * qwen_mtp.rs, trimmed draft head). Also returns the fp64 max logit and the fp64 gap
 * between the winner and the best other logit (the margin). */
static void lmhead_row(const uint16_t *hidden_row, const uint16_t *W, int V, int H,
                       int32_t *id, double *max_logit, double *gap) {
    int best = -1;
    float bestf = 0.0f;
    double best64 = 0.0, second64 = -INFINITY;
    double *hd = (double *)malloc(sizeof(double) * (size_t)H);
    for (int c = 0; c < H; ++c) hd[c] = orc_bf16_to_double(hidden_row[c]);
    for (int v = 0; v < V; ++v) {
        const uint16_t *w = W + (size_t)v * H;
        double acc = 0.0;
        for (int c = 0; c < H; ++c) acc += hd[c] * orc_bf16_to_double(w[c]);
        float f = (float)acc;
        if (best < 0 || f > bestf) {
            if (best >= 0 && best64 > second64) second64 = best64;
            best = v;
            bestf = f;
            best64 = acc;
        } else if (acc > second64) {
            second64 = acc;
        }
    }
    free(hd);
    *id = best;
    if (max_logit) *max_logit = best64;
    if (gap) *gap = best64 - second64;
}

int orc_lmhead_argmax(const uint16_t *hidden, const uint16_t *W, int M, int V, int H,
                      const int32_t *d2t, int d2t_limit, int32_t *ids, double *max_logit,
                      double *gap) {
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1) reduction(| : err)
    for (int m = 0; m < M; ++m) {
        int32_t id;
        lmhead_row(hidden + (size_t)m * H, W, V, H, &id, max_logit ? &max_logit[m] : 0,
                   gap ? &gap[m] : 0);
        if (d2t) {
            int32_t t = d2t[id];
            if (t < 0 || t >= d2t_limit) {
                err |= ORC_ERR_D2T;
                t = -1;
            }
            id = t;
        }
        ids[m] = id;
    }
    return err;
}

/* Plain logits, fp64 [M][V] (for row-invariance and tolerance checks on small sizes). */
void orc_lmhead_logits(const uint16_t *hidden, const uint16_t *W, int M, int V, int H,
                       double *logits) {
#pragma omp parallel for schedule(static)
    for (int m = 0; m < M; ++m)
        for (int v = 0; v < V; ++v) {
            double acc = 0.0;
            for (int c = 0; c < H; ++c)
                acc += orc_bf16_to_double(hidden[(size_t)m * H + c]) * orc_bf16_to_double(W[(size_t)v * H + c]);
            logits[(size_t)m * V + v] = acc;
        }
}

/* ------------------------------------------------------------------------------------
 * Greedy chain acceptance
 * ---------------------------------------------------------------------------------- */

/* DSSD-dev fast.py `generate_spec`: walk the drafts, stop at the first one that differs
 * from the target token of its row, then append target[len(committed)] (correction or
 * bonus). span-02 spec.rs: the draft at verify row j+1 is compared with the argmax of
 * verify row j; new position = pos + accepted + 1. */
void orc_accept(const int32_t *drafts, const int32_t *ids, const int32_t *pos, int B, int k,
                int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted, int32_t *out_pos,
                int32_t *out_next) {
    for (int b = 0; b < B; ++b) {
        const int32_t *target = ids + (size_t)b * (k + 1);
        int32_t *emit = out_tokens + (size_t)b * (k + 1);
        int n = 0;
        for (int i = 0; i < k; ++i) {
            int32_t d = drafts[(size_t)b * k + i];
            if (d != target[i]) break;
            emit[n++] = d;
        }
        int a = n;
        emit[n++] = target[a];
        for (int j = n; j <= k; ++j) emit[j] = -1;
        out_n[b] = n;
        out_accepted[b] = a;
        out_pos[b] = pos[b] + a + 1;
        out_next[b] = target[a];
    }
}

/* Stop tokens and a generation budget on top of the greedy run. DSSD-dev dssd/fast.py,
 * `_commit`: a cycle's committed tokens are appended one by one and the loop breaks right
 * after the first token the stop rule fires on (that token is kept), or once the output
 * reaches the generation limit max_new; span-02 engine/crates/model/src/spec.rs,
 * `Spec::body_inner`: the device acceptance call takes a small stop-id buffer (initialised
 * to -1, i.e. unused entries) and a token limit (1 << 30 = none). The run of branch b
 * (drafts[0..a) then ids[b(k+1)+a]) is cut after its first token that is in the stop
 * set, then to at most budget[b] tokens (budget NULL: no limit; a negative entry counts
 * as 0). n = tokens kept, accepted = drafts among them, new_pos = pos + n, next = the
 * last kept token (-1 when none), done = the kept run ends on a stop token or used the
 * whole budget. */
void orc_accept_stop(const int32_t *drafts, const int32_t *ids, const int32_t *pos, int B, int k,
                     const int32_t *stop, int n_stop, const int32_t *budget, int32_t *out_tokens,
                     int32_t *out_n, int32_t *out_accepted, int32_t *out_pos, int32_t *out_next,
                     int32_t *out_done) {
    for (int b = 0; b < B; ++b) {
        const int32_t *target = ids + (size_t)b * (k + 1);
        int32_t run[64];
        int a = 0;
        while (a < k && drafts[(size_t)b * k + a] == target[a]) {
            run[a] = drafts[(size_t)b * k + a];
            ++a;
        }
        run[a] = target[a];
        int n = a + 1, stopped = 0;
        for (int i = 0; i <= a; ++i) {
            int hit = 0;
            for (int j = 0; j < n_stop; ++j)
                if (stop[j] >= 0 && stop[j] == run[i]) hit = 1;
            if (hit) {
                n = i + 1;
                stopped = 1;
                break;
            }
        }
        int capped = 0;
        if (budget) {
            int cap = budget[b] < 0 ? 0 : budget[b];
            if (n > cap) {
                n = cap;
                stopped = 0; /* the stop token was cut off */
            }
            if (n == cap) capped = 1;
        }
        int32_t *emit = out_tokens + (size_t)b * (k + 1);
        for (int j = 0; j <= k; ++j) emit[j] = j < n ? run[j] : -1;
        out_n[b] = n;
        out_accepted[b] = a < n ? a : n;
        out_pos[b] = pos[b] + n;
        out_next[b] = n > 0 ? run[n - 1] : -1;
        out_done[b] = stopped || capped;
    }
}

/* Tree acceptance (greedy). DSSD-dev `_star_cycle`: a child is accepted when its token is
 * the target's choice at its parent (the root's argmax for a depth-1 star), and the
 * committed tokens are that choice followed by the accepted child's own choice. Here the
 * k+1 rows of branch b form a tree: row 0 is the root (the fed token), row j >= 1 carries
 * draft token drafts[b][j-1] and has parent[b][j] < j. From the root, the walk moves to the
 * lowest-numbered child whose token equals the current row's argmax ids[b(k+1)+cur], and
 * stops when none does. Emitted: the accepted drafts in walk order, then the last row's
 * argmax (the bonus); path[b][0] = 0 and path[b][i] = the i-th accepted row, -1 after.
 * A parent array with parent[j] outside [0, j) gives an error bit and no walk past it.
 * With parent[j] = j-1 this is orc_accept. */
int orc_accept_tree(const int32_t *drafts, const int32_t *ids, const int32_t *pos, const int32_t *parent,
                    int B, int k, int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted,
                    int32_t *out_pos, int32_t *out_next, int32_t *out_path) {
    int err = 0;
    for (int b = 0; b < B; ++b) {
        const int32_t *target = ids + (size_t)b * (k + 1);
        const int32_t *par = parent + (size_t)b * (k + 1);
        int32_t *emit = out_tokens + (size_t)b * (k + 1);
        int32_t *path = out_path + (size_t)b * (k + 1);
        for (int j = 1; j <= k; ++j)
            if (par[j] < 0 || par[j] >= j) err |= ORC_ERR_TREE;
        int cur = 0, a = 0;
        path[0] = 0;
        for (;;) {
            int next = -1;
            for (int c = cur + 1; c <= k; ++c)
                if (par[c] == cur && drafts[(size_t)b * k + c - 1] == target[cur]) { next = c; break; }
            if (next < 0) break;
            emit[a] = drafts[(size_t)b * k + next - 1];
            path[++a] = next;
            cur = next;
        }
        emit[a] = target[cur];
        for (int j = a + 1; j <= k; ++j) { emit[j] = -1; path[j] = -1; }
        out_n[b] = a + 1;
        out_accepted[b] = a;
        out_pos[b] = pos[b] + a + 1;
        out_next[b] = target[cur];
    }
    return err;
}

/* KV compaction after a tree walk (DSSD-dev `_star_cycle`: the accepted child's K/V is
 * copied to slot pos0+1). Accepted row path[b][i] (written at slot pos_b + path[b][i])
 * moves to slot pos_b + i, for i = 1..accepted[b], in ascending i: a path's rows increase,
 * so a source is never overwritten before it is read. bf16 pools copy bits; FP8 pools
 * decode with the source page's scale and re-encode with the destination page's scale. */
int orc_kv_compact(const orc_kv *kv, const int32_t *pos, const int32_t *path, const int32_t *accepted, int B,
                   int k) {
    int err = 0;
    const int Hkv = kv->n_kv_heads, d = kv->head_dim;
    for (int b = 0; b < B; ++b)
        for (int i = 1; i <= accepted[b]; ++i) {
            const int src_row = path[(size_t)b * (k + 1) + i];
            if (src_row == i) continue;
            int sp, ss, dp, ds;
            int e = locate(kv, b, pos[b] + src_row, &sp, &ss) | locate(kv, b, pos[b] + i, &dp, &ds);
            if (e) { err |= e; continue; }
            for (int g = 0; g < Hkv; ++g) {
                size_t src = pool_index(kv, sp, g, ss), dst = pool_index(kv, dp, g, ds);
                if (kv->kv_dtype == 0) {
                    memcpy((uint16_t *)kv->k_pool + dst, (uint16_t *)kv->k_pool + src, (size_t)d * 2);
                    memcpy((uint16_t *)kv->v_pool + dst, (uint16_t *)kv->v_pool + src, (size_t)d * 2);
                } else {
                    for (int c = 0; c < d; ++c) {
                        double xk = kv_value(kv, 0, sp, g, ss, c), xv = kv_value(kv, 1, sp, g, ss, c);
                        ((uint8_t *)kv->k_pool)[dst + c] =
                            orc_e4m3_encode((float)xk / kv->k_scale[(size_t)dp * Hkv + g]);
                        ((uint8_t *)kv->v_pool)[dst + c] =
                            orc_e4m3_encode((float)xv / kv->v_scale[(size_t)dp * Hkv + g]);
                    }
                }
            }
        }
    return err;
}

/* Speculative sampling acceptance (the next row f4). oxinfer `speculative_accept`: a draft d
 * drawn from q is kept with probability min(1, p(d) / q(d)), otherwise replaced by a token
 * drawn from the normalised max(0, p - q) (from p when that is all zero); DSSD-dev
 * `_sample_verify`: walk the chain, stop at the first rejection, and sample the bonus from
 * the last row's p after a full acceptance. The random numbers are inputs here (u in
 * [0, 1)): u_acc[b][i] for draft i's test, u_res[b] for the one token drawn at the end.
 * p_j = softmax(logits[b(k+1)+j] / temperature) in fp64; q [B][k][V] are the draft
 * distributions (probabilities). Drawing t from a non-negative weight vector w uses the
 * inverse CDF in index order: the smallest t whose running sum exceeds u * sum(w). */
static int draw_index(const double *w, int V, double u) {
    double tot = 0.0;
    for (int t = 0; t < V; ++t) tot += w[t];
    double c = 0.0, lim = u * tot;
    for (int t = 0; t < V; ++t) {
        c += w[t];
        if (c > lim) return t;
    }
    for (int t = V - 1; t >= 0; --t)
        if (w[t] > 0.0) return t;
    return 0;
}

static void softmax_t(const float *z, int V, double temperature, double *p) {
    double mx = -INFINITY;
    for (int t = 0; t < V; ++t)
        if ((double)z[t] / temperature > mx) mx = (double)z[t] / temperature;
    double den = 0.0;
    for (int t = 0; t < V; ++t) {
        p[t] = exp((double)z[t] / temperature - mx);
        den += p[t];
    }
    for (int t = 0; t < V; ++t) p[t] /= den;
}

/* A draft is a sample of q, so 0 <= d < V and q(d) > 0; a draft outside the vocabulary or
 * one that q gives no probability cannot have been drawn: it is an input error
 * (ORC_ERR_TOKEN) and is rejected (the replacement is drawn from the residual). */
int orc_accept_sample(const int32_t *drafts, const float *logits, const float *q, const int32_t *pos, int B,
                      int k, int V, double temperature, const float *u_acc, const float *u_res,
                      int32_t *out_tokens, int32_t *out_n, int32_t *out_accepted, int32_t *out_pos,
                      int32_t *out_next) {
    int err = 0;
#pragma omp parallel for schedule(dynamic, 16) reduction(| : err)
    for (int b = 0; b < B; ++b) {
        double *p = (double *)malloc(sizeof(double) * (size_t)V);
        double *w = (double *)malloc(sizeof(double) * (size_t)V);
        int32_t *emit = out_tokens + (size_t)b * (k + 1);
        int a = 0, last = -1;
        for (int i = 0; i < k; ++i) {
            softmax_t(logits + ((size_t)b * (k + 1) + i) * V, V, temperature, p);
            const int d = drafts[(size_t)b * k + i];
            const float *qi = q + ((size_t)b * k + i) * V;
            const int valid = d >= 0 && d < V && (double)qi[d] > 0.0;
            if (!valid) err |= ORC_ERR_TOKEN;
            const double pd = valid ? p[d] : 0.0, qd = valid ? (double)qi[d] : 1.0;
            if (valid && (pd >= qd || (double)u_acc[(size_t)b * k + i] < pd / qd)) {
                emit[a++] = d;
                continue;
            }
            int any = 0;
            for (int t = 0; t < V; ++t) {
                w[t] = p[t] - (double)qi[t];
                if (w[t] < 0.0) w[t] = 0.0;
                if (w[t] > 0.0) any = 1;
            }
            last = draw_index(any ? w : p, V, (double)u_res[b]);
            break;
        }
        if (last < 0) {  /* every draft kept: the bonus from the last row's p */
            softmax_t(logits + ((size_t)b * (k + 1) + a) * V, V, temperature, p);
            last = draw_index(p, V, (double)u_res[b]);
        }
        emit[a] = last;
        for (int j = a + 1; j <= k; ++j) emit[j] = -1;
        out_n[b] = a + 1;
        out_accepted[b] = a;
        out_pos[b] = pos[b] + a + 1;
        out_next[b] = last;
        free(p);
        free(w);
    }
    return err;
}

/* ------------------------------------------------------------------------------------
 * MTP draft-head input
 * ---------------------------------------------------------------------------------- */

/* oxinfer qwen_mtp.rs, module documentation:
 *   x = fc([rmsnorm_emb(embed(x_{i+1})), rmsnorm_hidden(h_i)])   fc: [H, 2H]
 * rmsnorm(y; g)_i = y_i / sqrt(mean(y^2) + eps) * g_i (fp64 here). The two halves are
 * rounded to bf16 (the concat is a bf16 activation), fc sums in fp64.
 * concat_out bf16 [M][2H]; x_out fp64 [M][H]. A token outside [0, V) gives a zero
 * embedding half and an error bit. */
int orc_mtp_input(const int32_t *tok, const uint16_t *E, const uint16_t *h, const float *g_emb,
                  const float *g_hid, double eps, const uint16_t *W_fc, int M, int H, int V,
                  uint16_t *concat_out, double *x_out) {
    int err = 0;
    for (int m = 0; m < M; ++m) {
        uint16_t *c = concat_out + (size_t)m * 2 * H;
        int t = tok[m];
        if (t < 0 || t >= V) {
            err |= ORC_ERR_TOKEN;
            for (int i = 0; i < H; ++i) c[i] = 0;
        } else {
            const uint16_t *e = E + (size_t)t * H;
            double ss = 0.0;
            for (int i = 0; i < H; ++i) {
                double y = orc_bf16_to_double(e[i]);
                ss += y * y;
            }
            double inv = 1.0 / sqrt(ss / H + eps);
            for (int i = 0; i < H; ++i) c[i] = orc_double_to_bf16(orc_bf16_to_double(e[i]) * inv * (double)g_emb[i]);
        }
        const uint16_t *hr = h + (size_t)m * H;
        double ss = 0.0;
        for (int i = 0; i < H; ++i) {
            double y = orc_bf16_to_double(hr[i]);
            ss += y * y;
        }
        double inv = 1.0 / sqrt(ss / H + eps);
        for (int i = 0; i < H; ++i) c[H + i] = orc_double_to_bf16(orc_bf16_to_double(hr[i]) * inv * (double)g_hid[i]);
    }
#pragma omp parallel for schedule(static)
    for (int item = 0; item < M * H; ++item) {
        int m = item / H, o = item % H;
        const uint16_t *c = concat_out + (size_t)m * 2 * H;
        const uint16_t *w = W_fc + (size_t)o * 2 * H;
        double acc = 0.0;
        for (int i = 0; i < 2 * H; ++i) acc += orc_bf16_to_double(w[i]) * orc_bf16_to_double(c[i]);
        x_out[item] = acc;
    }
    return err;
}

/* ------------------------------------------------------------------------------------
 * The draft head's remembered hidden rows (span-02 engine/crates/model/src/spec.rs,
 * `Spec::body_inner`): a step gathers h[b] = hpool[hslot[b]] before drafting and scatters
 * the acceptance's rows back, hpool[hslot[b]] = h[b], after it. Rows are bf16 bit patterns,
 * copied as they are; a slot outside [0, n_slots) is an error bit and its row is skipped.
 * ---------------------------------------------------------------------------------- */
int orc_h_gather(uint16_t *h_out, const uint16_t *hpool, const int32_t *hslot, int B, int H, int n_slots) {
    int err = 0;
    for (int b = 0; b < B; ++b) {
        const int s = hslot[b];
        if (s < 0 || s >= n_slots) {
            err |= ORC_ERR_SLOT;
            continue;
        }
        for (int i = 0; i < H; ++i) h_out[(size_t)b * H + i] = hpool[(size_t)s * H + i];
    }
    return err;
}

int orc_h_scatter(uint16_t *hpool, const uint16_t *h_in, const int32_t *hslot, int B, int H, int n_slots) {
    int err = 0;
    for (int b = 0; b < B; ++b) {
        const int s = hslot[b];
        if (s < 0 || s >= n_slots) {
            err |= ORC_ERR_SLOT;
            continue;
        }
        for (int i = 0; i < H; ++i) hpool[(size_t)s * H + i] = h_in[(size_t)b * H + i];
    }
    return err;
}
