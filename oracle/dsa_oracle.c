/*
 * CPU oracle for the DSA decode/prefill hot path (lightning indexer + Top-K + sparse flash attention).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may load this library: only the tests, the
 * package smoke check and the benchmark's CPU-baseline leg do.  It shares no code, header, table or
 * constant with the CUDA library; its inputs come from the seeded generator and its arithmetic is
 * written here from the definitions, in double precision, as plainly as possible.
 *
 * Sources (titles of the published articles the method is taken from):
 *  [A1] "Optimizing Inference for Hybrid Attention LLMs: Practices for Fast Adaptation",
 *       section 1 (sparse attention module bullet) and section 3.2 (index-gather-compute integration,
 *       paged KV management).
 *  [A2] "Optimizing Inference for Hybrid Attention Architectures: From Operator Fusion to Sequence
 *       Sharding", section "Breaking Down the Computational Path of Hybrid Attention", steps 1
 *       (index screening by the lightning indexer, head-importance weighting, Top-K) and 2 (sparse
 *       flash attention over the selected KV).
 *  [A3] "Day0 Inference Optimization for Next-Generation Hybrid-Architecture LLMs Based on CANN",
 *       section 2.1 (fused scoring/weighting/Top-K reading the paged K cache) and section 3.1 (FP8
 *       indexer inputs).
 *  [A4] "Day0 Inference Support and Performance Optimization for New LLM Architectures", sections 3.1
 *       (integrated indexer fusion: only Top-K indices leave the chip) and 3.2 (the sparse kernel
 *       reads only the selected positions' KV from the paged cache).
 *
 * The articles describe the steps in prose and print no formula.  Readings used here:
 *  - index score  I[t,s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d])   (no softmax, no bias);
 *  - FP8 inputs are E4M3 codes (OCP OFP8 definition) times one fp32 scale per row, applied literally;
 *  - MXFP8 inputs ([A1] section 1 and [A4] section 4.1: microscaled FP8, one scale per group of 32
 *    elements): E4M3 codes times one E8M0 scale per 32 consecutive elements of a row (OCP MX
 *    definition: the byte e means 2^(e - 127), 0xFF is NaN), applied literally;
 *  - query t of sequence b (n_b new tokens, L_b cached tokens including them) sits at position
 *    p = L_b - n_b + j and sees positions 0..p (causal, itself included);
 *  - Top-K orders by score descending, then position ascending; with fewer than K visible positions
 *    all are taken; the result is returned in ascending position order padded with -1;
 *  - attention over the selected rows: z = scale * q . kv (all 576 dims), softmax over the selected
 *    set, out = sum softmax * kv[:, :Dv] (V = leading Dv dims of the same latent row),
 *    lse = max z + log sum exp(z - max z) (natural log).  No selected row: out = 0, lse = -inf.
 *  - FP8 latent-KV cache ([A1] section 1 layered quantization; [A4] section 4 hierarchical quantization:
 *    FP8 with one scale per 128 elements of each token): the latent part (the leading Dv = 512 dims)
 *    is 4 tiles of 128 E4M3 codes, each with its own fp32 scale; the remaining 64 rotary dims stay bf16
 *    (576 is not a multiple of 128).  Row layout, 656 bytes: 512 codes, 4 fp32 scales, 64 bf16 values.
 *    An element is code value x its tile's scale, applied literally.
 *  - appending a step's rows ([A4] section 3.3, the K input of the indexer; quantisation as in [A1]
 *    section 1): query token t's new indexer key and latent-KV row go to the cache row of its own
 *    position p_t.  FP8 caches quantise dynamically: scale = absmax / 448 over the quantisation group
 *    (the indexer key row; each 128-element latent tile), 1 when the group is all zero, and
 *    code = E4M3(x / scale) rounded to nearest, ties to the even code, saturating at 448.  The pages fix
 *    no precision for this; absmax, scale and x / scale are taken in fp32 (IEEE, correctly rounded),
 *    the precision of the GPU kernel, so both make the same integer decisions.
 */
#include <math.h>
#include <omp.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

typedef struct {
    int32_t batch;
    int32_t total_q;
    int32_t num_pages;
    int32_t page_size;
    int32_t max_pages_per_seq;
    int32_t idx_heads;
    int32_t idx_dim;
    int32_t idx_fp8; /* 0: q_idx/k_idx are bf16 bits; 1: E4M3 codes with fp32 row scales;
                        2: E4M3 codes with one E8M0 scale byte per 32 elements (MXFP8) */
    int32_t top_k;
    int32_t attn_heads;
    int32_t kv_dim;
    int32_t v_dim;
    int32_t kv_fp8; /* 0: kv rows are bf16 bits; 1: the 656-byte FP8 layout above */
    double softmax_scale;
} oracle_dims;

enum { ORC_OK = 0, ORC_BAD_ARG = -1, ORC_BAD_PAGE = -2, ORC_BAD_POS = -3, ORC_NOMEM = -4 };

/* Threads the oracle's parallel loops use from now on (n >= 1); returns the previous maximum.  Used to
 * time the oracle on one core. */
int oracle_set_threads(int n) {
    int old = omp_get_max_threads();
    if (n >= 1) omp_set_num_threads(n);
    return old;
}

/* bf16 is the upper half of an IEEE binary32 value. */
double oracle_bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* OCP OFP8 E4M3: sign, 4 exponent bits (bias 7), 3 mantissa bits; exponent 0 is subnormal
 * (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
double oracle_e4m3_value(uint8_t code) {
    int sign = code >> 7;
    int e = (code >> 3) & 0xF;
    int m = code & 0x7;
    double v;
    if (e == 0xF && m == 0x7) return NAN;
    if (e == 0)
        v = ldexp((double)m / 8.0, -6);
    else
        v = ldexp(1.0 + (double)m / 8.0, e - 7);
    return sign ? -v : v;
}

/* E4M3 code of y: the nearest of the finite values (codes 0x00..0x7E and their negatives) by scanning
 * them all, ties to the even code; beyond 448 in magnitude the result is +-448 (saturation); NaN gives
 * 0x7F.  Zero keeps its sign. */
uint8_t oracle_e4m3_encode(float y) {
    if (y != y) return 0x7F;
    uint8_t sign = signbit(y) ? 0x80 : 0x00;
    double a = fabs((double)y);
    int best = 0;
    double best_err = INFINITY;
    for (int c = 0; c <= 0x7E; ++c) {
        double err = fabs(oracle_e4m3_value((uint8_t)c) - a);
        if (err < best_err || (err == best_err && (c & 1) == 0)) {
            best = c;
            best_err = err;
        }
    }
    return (uint8_t)(sign | best);
}

/* Dynamic E4M3 quantisation of one group of n values (see the readings at the top):
 * *scale = absmax / 448 in fp32 (1 for an all-zero group), codes[i] = E4M3(x[i] / *scale) in fp32. */
void oracle_quantize_group(const float* x, int32_t n, uint8_t* codes, float* scale) {
    float amax = 0.0f;
    for (int32_t i = 0; i < n; ++i)
        if (fabsf(x[i]) > amax) amax = fabsf(x[i]);
    float s = amax > 0.0f ? amax / 448.0f : 1.0f;
    for (int32_t i = 0; i < n; ++i) {
        float y = x[i] / s;
        codes[i] = oracle_e4m3_encode(y);
    }
    *scale = s;
}

/* Bytes of one latent-KV cache row. */
static int64_t kv_row_bytes(const oracle_dims* d) {
    if (!d->kv_fp8) return (int64_t)d->kv_dim * 2;
    return (int64_t)d->v_dim + 4 * (d->v_dim / 128) + 2 * ((int64_t)d->kv_dim - d->v_dim);
}

/* Element c of latent-KV cache row `row` (either layout). */
static double kv_elem(const oracle_dims* d, const void* kv_cache, int64_t row, int32_t c) {
    const uint8_t* r = (const uint8_t*)kv_cache + row * kv_row_bytes(d);
    uint16_t bits;
    if (!d->kv_fp8) {
        memcpy(&bits, r + 2 * (int64_t)c, 2);
        return oracle_bf16_value(bits);
    }
    if (c < d->v_dim) {
        float scale;
        memcpy(&scale, r + d->v_dim + 4 * (c / 128), 4);
        return oracle_e4m3_value(r[c]) * (double)scale;
    }
    memcpy(&bits, r + d->v_dim + 4 * (d->v_dim / 128) + 2 * (int64_t)(c - d->v_dim), 2);
    return oracle_bf16_value(bits);
}

/* OCP MX E8M0 scale: 2^(e - 127); 0xFF is NaN. */
double oracle_e8m0_value(uint8_t e) {
    if (e == 0xFF) return NAN;
    return ldexp(1.0, (int)e - 127);
}

/* Sequence of query token t and its causal position. */
static int query_locate(const oracle_dims* d, const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t t,
                        int32_t* b_out, int64_t* p_out) {
    if (t < 0 || t >= d->total_q) return ORC_BAD_ARG;
    for (int32_t b = 0; b < d->batch; ++b) {
        if (t >= cu_q_lens[b] && t < cu_q_lens[b + 1]) {
            int32_t n = cu_q_lens[b + 1] - cu_q_lens[b];
            int32_t L = seq_lens[b];
            if (n > L) return ORC_BAD_POS;
            *b_out = b;
            *p_out = (int64_t)L - n + (t - cu_q_lens[b]);
            return ORC_OK;
        }
    }
    return ORC_BAD_ARG;
}

/* Physical row of logical position s of sequence b ([A1] 3.2 paged KV management). */
static int page_row(const oracle_dims* d, const int32_t* page_table, int32_t b, int64_t s, int64_t* row) {
    int64_t lp = s / d->page_size;
    if (lp >= d->max_pages_per_seq) return ORC_BAD_POS;
    int32_t pg = page_table[(int64_t)b * d->max_pages_per_seq + lp];
    if (pg < 0 || pg >= d->num_pages) return ORC_BAD_PAGE;
    *row = (int64_t)pg * d->page_size + s % d->page_size;
    return ORC_OK;
}

static double idx_elem(const oracle_dims* d, const void* base, const float* scales, int64_t row, int32_t col) {
    if (d->idx_fp8 == 2) {  /* scales: E8M0 bytes [rows][idx_dim / 32] */
        const uint8_t* p = (const uint8_t*)base;
        const uint8_t* e = (const uint8_t*)scales;
        return oracle_e4m3_value(p[row * d->idx_dim + col]) * oracle_e8m0_value(e[row * (d->idx_dim / 32) + col / 32]);
    }
    if (d->idx_fp8) {
        const uint8_t* p = (const uint8_t*)base;
        return oracle_e4m3_value(p[row * d->idx_dim + col]) * (double)scales[row];
    }
    const uint16_t* p = (const uint16_t*)base;
    return oracle_bf16_value(p[row * d->idx_dim + col]);
}

/*
 * Index scores of query t against every visible position 0..p ([A2] step 1; [A3] 2.1):
 * scores[s] = sum_h w[t,h] * max(0, sum_d q[t,h,d] * k[s,d]).  Returns the count p+1 (>= 0) or an
 * error code (< 0).  `scores` must hold at least p+1 values.
 */
int64_t oracle_index_scores(const oracle_dims* d, const void* q_idx, const float* q_scale, const float* w,
                            const void* k_cache, const float* k_scale, const int32_t* page_table,
                            const int32_t* seq_lens, const int32_t* cu_q_lens, int32_t t, double* scores) {
    int32_t b;
    int64_t p;
    int rc = query_locate(d, seq_lens, cu_q_lens, t, &b, &p);
    if (rc) return rc;
    const int32_t H = d->idx_heads, D = d->idx_dim;
    /* qT[j][h] = q[t,h,j]: the query stored dimension-major, so that the dot products of all heads advance
     * together, one dimension at a time.  Every dot product still adds its terms in dimension order
     * (j = 0, 1, ...), exactly as the definition reads; only independent dot products are interleaved. */
    double* qT = (double*)malloc(sizeof(double) * (size_t)H * (size_t)D);
    double* k = (double*)malloc(sizeof(double) * (size_t)D);
    double* dot = (double*)malloc(sizeof(double) * (size_t)H);
    if (!qT || !k || !dot) {
        free(qT);
        free(k);
        free(dot);
        return ORC_NOMEM;
    }
    for (int32_t h = 0; h < H; ++h)
        for (int32_t j = 0; j < D; ++j)
            qT[j * H + h] = idx_elem(d, q_idx, q_scale, (int64_t)t * H + h, j);
    for (int64_t s = 0; s <= p; ++s) {
        int64_t row;
        rc = page_row(d, page_table, b, s, &row);
        if (rc) {
            free(qT);
            free(k);
            free(dot);
            return rc;
        }
        for (int32_t j = 0; j < D; ++j) k[j] = idx_elem(d, k_cache, k_scale, row, j);
        for (int32_t h = 0; h < H; ++h) dot[h] = 0.0;
        for (int32_t j = 0; j < D; ++j)
            for (int32_t h = 0; h < H; ++h) dot[h] += qT[j * H + h] * k[j];
        double I = 0.0;
        for (int32_t h = 0; h < H; ++h) {
            double relu = dot[h] > 0.0 ? dot[h] : 0.0;
            I += (double)w[(int64_t)t * H + h] * relu;
        }
        scores[s] = I;
    }
    free(qT);
    free(k);
    free(dot);
    return p + 1;
}

typedef struct {
    double score;
    int64_t pos;
} scored_pos;

/* Score descending, then position ascending. */
static int by_score_then_pos(const void* a, const void* b) {
    const scored_pos* x = (const scored_pos*)a;
    const scored_pos* y = (const scored_pos*)b;
    if (x->score > y->score) return -1;
    if (x->score < y->score) return 1;
    return (x->pos > y->pos) - (x->pos < y->pos);
}

static int by_int32(const void* a, const void* b) {
    int32_t x = *(const int32_t*)a, y = *(const int32_t*)b;
    return (x > y) - (x < y);
}

/*
 * Top-K selection for the listed query tokens ([A2] step 1; [A4] 3.1: only the Top-K indices are
 * produced).  For each listed token i (global index tlist[i], or i itself when tlist is NULL):
 *   topk[i*K .. i*K+K-1]  = selected positions, ascending, padded with -1;
 *   kth[i]                = score of the last selected position in (score desc, pos asc) order;
 *   nsel[i]               = min(K, p+1).
 * Returns 0 or the first error code met.
 */
int oracle_indexer_topk(const oracle_dims* d, const void* q_idx, const float* q_scale, const float* w,
                        const void* k_cache, const float* k_scale, const int32_t* page_table,
                        const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* tlist, int32_t nt,
                        int32_t* topk, double* kth, int32_t* nsel) {
    int err = 0;
    const int32_t K = d->top_k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < nt; ++i) {
        int32_t t = tlist ? tlist[i] : i;
        int32_t b;
        int64_t p;
        int rc = query_locate(d, seq_lens, cu_q_lens, t, &b, &p);
        int32_t* out = topk + (int64_t)i * K;
        for (int32_t k = 0; k < K; ++k) out[k] = -1;
        if (rc) {
#pragma omp atomic write
            err = rc;
            continue;
        }
        int64_t n = p + 1;
        double* sc = (double*)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
        scored_pos* sp = (scored_pos*)malloc(sizeof(scored_pos) * (size_t)(n > 0 ? n : 1));
        if (!sc || !sp) {
            free(sc);
            free(sp);
#pragma omp atomic write
            err = ORC_NOMEM;
            continue;
        }
        int64_t got = oracle_index_scores(d, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens,
                                          cu_q_lens, t, sc);
        if (got < 0) {
            free(sc);
            free(sp);
#pragma omp atomic write
            err = (int)got;
            continue;
        }
        for (int64_t s = 0; s < n; ++s) {
            sp[s].score = sc[s] == 0.0 ? 0.0 : sc[s]; /* -0.0 ranks as +0.0 */
            sp[s].pos = s;
        }
        qsort(sp, (size_t)n, sizeof(scored_pos), by_score_then_pos);
        int32_t m = (int32_t)(n < K ? n : K);
        for (int32_t k = 0; k < m; ++k) out[k] = (int32_t)sp[k].pos;
        qsort(out, (size_t)m, sizeof(int32_t), by_int32);
        if (kth) kth[i] = m > 0 ? sp[m - 1].score : -INFINITY;
        if (nsel) nsel[i] = m;
        free(sc);
        free(sp);
    }
    return err;
}

/*
 * Sparse flash attention over the selected rows ([A2] step 2; [A4] 3.2; [A1] 3.2 gather):
 * for each listed token i and head h, with S = {topk[i, k] >= 0}:
 *   z_s = scale * sum_{c < kv_dim} q[t,h,c] * kv[s,c]
 *   out[i,h,:] = sum_s softmax(z)_s * kv[s, :v_dim],  lse[i,h] = logsumexp(z).
 * topk rows are indexed by list position i (row i belongs to token tlist[i]).
 * weights (optional, [nt, H, K]) receives softmax(z) in topk order (0 for -1 entries).
 */
int oracle_sparse_attn(const oracle_dims* d, const uint16_t* q, const void* kv_cache,
                       const int32_t* page_table, const int32_t* seq_lens, const int32_t* cu_q_lens,
                       const int32_t* topk, const int32_t* tlist, int32_t nt, double* out, double* lse,
                       double* weights) {
    int err = 0;
    const int32_t H = d->attn_heads, C = d->kv_dim, V = d->v_dim, K = d->top_k;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < nt; ++i) {
        int32_t t = tlist ? tlist[i] : i;
        int32_t b;
        int64_t p;
        int rc = query_locate(d, seq_lens, cu_q_lens, t, &b, &p);
        if (rc) {
#pragma omp atomic write
            err = rc;
            continue;
        }
        const int32_t* sel = topk + (int64_t)i * K;
        int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * (size_t)(K > 0 ? K : 1));
        double* z = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)H);
        /* the selected rows, decoded once (kv[k][c]), and the queries stored dimension-major (qT[c][h]) */
        double* kv = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1) * (size_t)C);
        double* qT = (double*)malloc(sizeof(double) * (size_t)C * (size_t)H);
        if (!rows || !z || !kv || !qT) {
            free(rows);
            free(z);
            free(kv);
            free(qT);
#pragma omp atomic write
            err = ORC_NOMEM;
            continue;
        }
        int bad = 0;
        for (int32_t k = 0; k < K; ++k) {
            rows[k] = -1;
            if (sel[k] < 0) continue;
            if (sel[k] > p) {
                bad = ORC_BAD_POS;
                break;
            }
            if (page_row(d, page_table, b, sel[k], &rows[k])) {
                bad = ORC_BAD_PAGE;
                break;
            }
        }
        if (bad) {
            free(rows);
            free(z);
            free(kv);
            free(qT);
#pragma omp atomic write
            err = bad;
            continue;
        }
        for (int32_t k = 0; k < K; ++k)
            if (rows[k] >= 0)
                for (int32_t c = 0; c < C; ++c) kv[(int64_t)k * C + c] = kv_elem(d, kv_cache, rows[k], c);
        for (int32_t h = 0; h < H; ++h)
            for (int32_t c = 0; c < C; ++c) qT[(int64_t)c * H + h] = oracle_bf16_value(q[((int64_t)t * H + h) * C + c]);
        /* z[k][h] = scale * sum_c q[t,h,c] kv[k,c]: every dot product adds its terms in dimension order; the
         * heads' dot products advance together */
        for (int32_t k = 0; k < K; ++k) {
            if (rows[k] < 0) continue;
            double* zk = z + (int64_t)k * H;
            for (int32_t h = 0; h < H; ++h) zk[h] = 0.0;
            for (int32_t c = 0; c < C; ++c) {
                const double v = kv[(int64_t)k * C + c];
                for (int32_t h = 0; h < H; ++h) zk[h] += qT[(int64_t)c * H + h] * v;
            }
            for (int32_t h = 0; h < H; ++h) zk[h] = d->softmax_scale * zk[h];
        }
        for (int32_t h = 0; h < H; ++h) {
            double zmax = -INFINITY;
            int32_t count = 0;
            for (int32_t k = 0; k < K; ++k) {
                if (rows[k] < 0) continue;
                const double zz = z[(int64_t)k * H + h];
                if (zz > zmax) zmax = zz;
                ++count;
            }
            double* o = out + ((int64_t)i * H + h) * V;
            for (int32_t v = 0; v < V; ++v) o[v] = 0.0;
            double* wrow = weights ? weights + ((int64_t)i * H + h) * K : NULL;
            if (wrow)
                for (int32_t k = 0; k < K; ++k) wrow[k] = 0.0;
            if (count == 0) {
                lse[(int64_t)i * H + h] = -INFINITY;
                continue;
            }
            double denom = 0.0;
            for (int32_t k = 0; k < K; ++k)
                if (rows[k] >= 0) denom += exp(z[(int64_t)k * H + h] - zmax);
            for (int32_t k = 0; k < K; ++k) {
                if (rows[k] < 0) continue;
                double a = exp(z[(int64_t)k * H + h] - zmax) / denom;
                if (wrow) wrow[k] = a;
                for (int32_t v = 0; v < V; ++v) o[v] += a * kv[(int64_t)k * C + v];
            }
            lse[(int64_t)i * H + h] = zmax + log(denom);
        }
        free(rows);
        free(z);
        free(kv);
        free(qT);
    }
    return err;
}

/*
 * Index scores of several query tokens at once (OpenMP over the list): row i of `scores` (stride
 * `stride` values) receives I[tlist[i], 0..p], the rest of the row is left untouched.  Returns 0 or
 * the first error code met.
 */
int oracle_index_scores_batch(const oracle_dims* d, const void* q_idx, const float* q_scale, const float* w,
                              const void* k_cache, const float* k_scale, const int32_t* page_table,
                              const int32_t* seq_lens, const int32_t* cu_q_lens, const int32_t* tlist, int32_t nt,
                              int64_t stride, double* scores) {
    int err = 0;
#pragma omp parallel for schedule(dynamic, 1)
    for (int32_t i = 0; i < nt; ++i) {
        int64_t got = oracle_index_scores(d, q_idx, q_scale, w, k_cache, k_scale, page_table, seq_lens, cu_q_lens,
                                          tlist[i], scores + (int64_t)i * stride);
        if (got < 0) {
#pragma omp atomic write
            err = (int)got;
        }
    }
    return err;
}

/*
 * Appending one decode/prefill step's rows to the paged caches (readings at the top): for every query
 * token t, its new indexer key k_new[t] (bf16 bits [T, Di], or NULL) goes to the indexer cache row of
 * position p_t (bf16 copy, or E4M3 codes with the row's scale in k_scale), and its new latent-KV row
 * kv_new[t] (bf16 bits [T, kv_dim], or NULL) to the latent-KV cache row of p_t (bf16 copy, or the FP8
 * layout).  Returns 0 or the first error code met (nothing is written for a token with an error).
 */
int oracle_append_rows(const oracle_dims* d, const uint16_t* k_new, const uint16_t* kv_new, const int32_t* page_table,
                       const int32_t* seq_lens, const int32_t* cu_q_lens, void* k_cache, float* k_scale,
                       void* kv_cache) {
    int err = 0;
    if (k_new && d->idx_fp8 == 2) return ORC_BAD_ARG; /* appending MXFP8 keys is not defined here */
    float* x = (float*)malloc(sizeof(float) * (size_t)(d->idx_dim > d->kv_dim ? d->idx_dim : d->kv_dim));
    if (!x) return ORC_NOMEM;
    for (int32_t t = 0; t < d->total_q; ++t) {
        int32_t b;
        int64_t p, row;
        int rc = query_locate(d, seq_lens, cu_q_lens, t, &b, &p);
        if (!rc) rc = page_row(d, page_table, b, p, &row);
        if (rc) {
            if (!err) err = rc;
            continue;
        }
        if (k_new) {
            const uint16_t* src = k_new + (int64_t)t * d->idx_dim;
            if (d->idx_fp8) {
                for (int32_t c = 0; c < d->idx_dim; ++c) x[c] = (float)oracle_bf16_value(src[c]);
                oracle_quantize_group(x, d->idx_dim, (uint8_t*)k_cache + row * d->idx_dim, &k_scale[row]);
            } else {
                memcpy((uint16_t*)k_cache + row * d->idx_dim, src, sizeof(uint16_t) * (size_t)d->idx_dim);
            }
        }
        if (kv_new) {
            const uint16_t* src = kv_new + (int64_t)t * d->kv_dim;
            uint8_t* dst = (uint8_t*)kv_cache + row * kv_row_bytes(d);
            if (d->kv_fp8) {
                for (int32_t c = 0; c < d->v_dim; ++c) x[c] = (float)oracle_bf16_value(src[c]);
                for (int32_t tile = 0; tile < d->v_dim / 128; ++tile) {
                    float scale;
                    oracle_quantize_group(x + 128 * tile, 128, dst + 128 * tile, &scale);
                    memcpy(dst + d->v_dim + 4 * tile, &scale, 4);
                }
                memcpy(dst + d->v_dim + 4 * (d->v_dim / 128), src + d->v_dim,
                       sizeof(uint16_t) * (size_t)(d->kv_dim - d->v_dim));
            } else {
                memcpy(dst, src, sizeof(uint16_t) * (size_t)d->kv_dim);
            }
        }
    }
    free(x);
    return err;
}
