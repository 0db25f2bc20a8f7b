/*
 * oracle.c -- plain fp64 CPU reference for paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline leg
 * use it.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes is the plain definition of scaled dot-product attention,
 *     out = softmax(Q K^T * scale) V,
 * as given in the GPU programming guide page ("From megabytes to megawatts: a
 * full guide to high-performance LLM and diffusion kernels with CUDA and Triton",
 * section "Decomposing multi-head attention (MHA)"), evaluated in double
 * precision, with no tiling, no online softmax and no split: scores for every
 * visible key, subtract the row maximum, exponentiate, normalise, weight V.
 * The online-softmax / split-KV algorithm the GPU path uses ("The Flash Attention
 * revolution" on the same page; "Parallel Tiled Softmax" in the five-step list
 * of the Triton unified-attention page, "What three things the IBM paper got
 * right") reaches this same result up to rounding order, so the definition is
 * the oracle.
 *
 * Readings where the pages are silent (each is also listed in the design notes):
 *  - Cache layout [num_blocks, page_size, num_kv_heads, head_dim], bf16; K and V
 *    are separate pools of the same layout.  Logical position j of sequence b
 *    lives in physical page block_table[b][j / page_size], slot j % page_size.
 *  - Grouped-query attention: query head h reads KV head h / (Hq / Hkv).
 *  - Causal masking is bottom-right aligned: sequence b has seq_lens[b] = L_b
 *    tokens of context including its n_b new tokens, which are the last n_b
 *    positions; new token i sits at p = L_b - n_b + i and sees keys 0..p.  The
 *    causal rule itself ("future tokens get -inf") is from "Flash Attention in
 *    Triton" on the GPU programming guide page.
 *  - scale is the float the caller passes, widened to double exactly.
 *
 * Parity pins (tests/test_oracle_pins.py): closed forms (single key, constant V,
 * zero keys -> mean of the visible rows, two-key logistic weights), row sums,
 * block-permutation and causal-hiding invariants, and the library special case
 * torch.nn.functional.scaled_dot_product_attention in fp64 with an explicit
 * bottom-right mask.  tests/test_oracle_mutants.py plants plausible mistakes in a
 * copy of this file and checks that some pin fails for each.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum {
    ORACLE_OK = 0,
    ORACLE_BAD_DIMS = 1,
    ORACLE_BAD_QUERY_START = 2,
    ORACLE_BAD_LENGTHS = 3,
    ORACLE_BAD_BLOCK = 4,
    ORACLE_BAD_ROW = 5,
    ORACLE_NO_MEMORY = 6,
};

typedef struct {
    int64_t num_tokens;   /* T  */
    int64_t num_seqs;     /* B  */
    int64_t num_q_heads;  /* Hq */
    int64_t num_kv_heads; /* Hkv */
    int64_t head_dim;     /* D  */
    int64_t page_size;    /* P  */
    int64_t num_blocks;   /* NB */
    int64_t max_pages;    /* block_table row length */
} oracle_dims;

/* bf16 -> double is exact: the bf16 bits are the top half of an fp32. */
static double bf16_value(uint16_t bits) {
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Checks the caller's contract; returns ORACLE_OK or the first violation. */
int oracle_validate(const oracle_dims* d, const int32_t* block_table, const int32_t* seq_lens,
                    const int32_t* query_start_loc) {
    if (d->num_tokens < 0 || d->num_seqs < 0 || d->num_q_heads <= 0 || d->num_kv_heads <= 0 ||
        d->head_dim <= 0 || d->page_size <= 0 || d->num_blocks <= 0 || d->max_pages < 0 ||
        d->num_q_heads % d->num_kv_heads != 0)
        return ORACLE_BAD_DIMS;
    if (query_start_loc[0] != 0 || query_start_loc[d->num_seqs] != d->num_tokens)
        return ORACLE_BAD_QUERY_START;
    for (int64_t b = 0; b < d->num_seqs; ++b) {
        int64_t n = (int64_t)query_start_loc[b + 1] - query_start_loc[b];
        int64_t L = seq_lens[b];
        if (n < 0) return ORACLE_BAD_QUERY_START;
        if (L < n || L > d->max_pages * d->page_size) return ORACLE_BAD_LENGTHS;
        int64_t pages = (L + d->page_size - 1) / d->page_size;
        for (int64_t pg = 0; pg < pages; ++pg) {
            int32_t blk = block_table[b * d->max_pages + pg];
            if (blk < 0 || blk >= d->num_blocks) return ORACLE_BAD_BLOCK;
        }
    }
    return ORACLE_OK;
}

/* Sequence that owns query token t (query_start_loc is non-decreasing). */
static int64_t owner_seq(const int32_t* qsl, int64_t num_seqs, int64_t t) {
    int64_t lo = 0, hi = num_seqs - 1;
    while (lo < hi) {
        int64_t mid = (lo + hi + 1) / 2;
        if (qsl[mid] <= t) lo = mid; else hi = mid - 1;
    }
    return lo;
}

/* Address of the D values of logical position j, KV head hk, of sequence b. */
static const uint16_t* cache_row(const uint16_t* cache, const oracle_dims* d, const int32_t* block_table,
                                 int64_t b, int64_t j, int64_t hk) {
    int64_t page = block_table[b * d->max_pages + j / d->page_size];
    int64_t slot = j % d->page_size;
    return cache + ((page * d->page_size + slot) * d->num_kv_heads + hk) * d->head_dim;
}

/*
 * One output row: query token t, query head h.
 *   out[D]      attention output in double
 *   weights[L]  optional: softmax weight of every position 0..L_b-1 (0 where masked)
 *   lse         optional: log(sum_j exp(s_j)) over the visible keys
 * scores is caller scratch of at least L_b doubles.
 */
static void one_row(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                    const int32_t* block_table, const int32_t* seq_lens, const int32_t* qsl,
                    const oracle_dims* d, double scale, int64_t t, int64_t h,
                    double* scores, double* out, double* weights, double* lse) {
    const int64_t D = d->head_dim;
    const int64_t group = d->num_q_heads / d->num_kv_heads;
    const int64_t b = owner_seq(qsl, d->num_seqs, t);
    const int64_t n = (int64_t)qsl[b + 1] - qsl[b];
    const int64_t L = seq_lens[b];
    const int64_t i = t - qsl[b];
    const int64_t p = L - n + i;          /* absolute position of this query */
    const int64_t hk = h / group;         /* the KV head this query head reads */
    const uint16_t* qrow = q + (t * d->num_q_heads + h) * D;

    /* s_j = scale * <q, k_j> for every visible key j <= p */
    double m = -INFINITY;
    for (int64_t j = 0; j <= p; ++j) {
        const uint16_t* krow = cache_row(k_cache, d, block_table, b, j, hk);
        double dot = 0.0;
        for (int64_t c = 0; c < D; ++c) dot += bf16_value(qrow[c]) * bf16_value(krow[c]);
        scores[j] = scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    /* softmax over the visible keys (the maximum is subtracted before exp) */
    double l = 0.0;
    for (int64_t j = 0; j <= p; ++j) {
        scores[j] = exp(scores[j] - m);
        l += scores[j];
    }
    /* out = sum_j w_j v_j with w_j = e_j / l */
    for (int64_t c = 0; c < D; ++c) out[c] = 0.0;
    for (int64_t j = 0; j <= p; ++j) {
        const double w = scores[j] / l;
        const uint16_t* vrow = cache_row(v_cache, d, block_table, b, j, hk);
        for (int64_t c = 0; c < D; ++c) out[c] += w * bf16_value(vrow[c]);
        if (weights) weights[j] = w;
    }
    if (weights)
        for (int64_t j = p + 1; j < L; ++j) weights[j] = 0.0;
    if (lse) *lse = m + log(l);
}

/*
 * Selected rows.  rows holds n_rows pairs (token, q_head).  out is [n_rows, D].
 * lse (optional) is [n_rows].  threads <= 0 uses the OpenMP default.
 * Returns ORACLE_OK or an error code; on error nothing is written.
 */
int oracle_attention_rows(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                          const int32_t* block_table, const int32_t* seq_lens,
                          const int32_t* query_start_loc, const oracle_dims* d, double scale,
                          const int64_t* rows, int64_t n_rows, double* out, double* lse, int threads) {
    int rc = oracle_validate(d, block_table, seq_lens, query_start_loc);
    if (rc) return rc;
    for (int64_t r = 0; r < n_rows; ++r)
        if (rows[2 * r] < 0 || rows[2 * r] >= d->num_tokens || rows[2 * r + 1] < 0 ||
            rows[2 * r + 1] >= d->num_q_heads)
            return ORACLE_BAD_ROW;
    int64_t max_ctx = 1;
    for (int64_t b = 0; b < d->num_seqs; ++b)
        if (seq_lens[b] > max_ctx) max_ctx = seq_lens[b];
    int failed = 0;
#ifdef _OPENMP
    const int nt = threads > 0 ? threads : omp_get_max_threads();
#pragma omp parallel num_threads(nt)
#endif
    {
        double* scores = (double*)malloc(sizeof(double) * (size_t)max_ctx);
        if (!scores) {
#ifdef _OPENMP
#pragma omp atomic write
#endif
            failed = 1;
        }
#ifdef _OPENMP
#pragma omp for schedule(dynamic, 1)
#endif
        for (int64_t r = 0; r < n_rows; ++r) {
            if (!scores) continue;
            one_row(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, d, scale,
                    rows[2 * r], rows[2 * r + 1], scores, out + r * d->head_dim, NULL,
                    lse ? lse + r : NULL);
        }
        free(scores);
    }
    return failed ? ORACLE_NO_MEMORY : ORACLE_OK;
}

/* Every row: out is [T, Hq, D], lse (optional) is [T, Hq]. */
int oracle_attention(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     const int32_t* block_table, const int32_t* seq_lens, const int32_t* query_start_loc,
                     const oracle_dims* d, double scale, double* out, double* lse, int threads) {
    int64_t n_rows = d->num_tokens * d->num_q_heads;
    int64_t* rows = (int64_t*)malloc(sizeof(int64_t) * 2 * (size_t)(n_rows ? n_rows : 1));
    if (!rows) return ORACLE_NO_MEMORY;
    for (int64_t t = 0; t < d->num_tokens; ++t)
        for (int64_t h = 0; h < d->num_q_heads; ++h) {
            rows[2 * (t * d->num_q_heads + h)] = t;
            rows[2 * (t * d->num_q_heads + h) + 1] = h;
        }
    int rc = oracle_attention_rows(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, d, scale,
                                   rows, n_rows, out, lse, threads);
    free(rows);
    return rc;
}

/* Softmax weights of one row over positions 0..L_b-1 (masked positions are 0). */
int oracle_attention_weights(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                             const int32_t* block_table, const int32_t* seq_lens,
                             const int32_t* query_start_loc, const oracle_dims* d, double scale,
                             int64_t t, int64_t h, double* weights, double* out) {
    int rc = oracle_validate(d, block_table, seq_lens, query_start_loc);
    if (rc) return rc;
    if (t < 0 || t >= d->num_tokens || h < 0 || h >= d->num_q_heads) return ORACLE_BAD_ROW;
    int64_t b = owner_seq(query_start_loc, d->num_seqs, t);
    int64_t L = seq_lens[b] > 0 ? seq_lens[b] : 1;
    double* scores = (double*)malloc(sizeof(double) * (size_t)L);
    if (!scores) return ORACLE_NO_MEMORY;
    one_row(q, k_cache, v_cache, block_table, seq_lens, query_start_loc, d, scale, t, h, scores, out,
            weights, NULL);
    free(scores);
    return ORACLE_OK;
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Paged KV-cache write: for every new token t with slot_mapping[t] = s >= 0,
 * copy k_new[t] and v_new[t] ([Hkv, D] each) into page s / page_size, slot
 * s % page_size of k_cache and v_cache.  A negative slot means "no write"
 * (padding).  This is how the new tokens' K and V reach the paged KV cache of
 * the Triton unified-attention page (section "Why is switching the card so
 * hard": the paged KV cache) before attention reads them through the block
 * table.  bf16 values are copied bit for bit.  Returns ORACLE_BAD_BLOCK, with
 * nothing written, if a slot lies past num_blocks * page_size.
 */
int oracle_cache_write(const uint16_t* k_new, const uint16_t* v_new, const int64_t* slot_mapping,
                       uint16_t* k_cache, uint16_t* v_cache, int64_t num_tokens, int64_t num_blocks,
                       int64_t page_size, int64_t num_kv_heads, int64_t head_dim) {
    const int64_t row = num_kv_heads * head_dim;  /* values of one token */
    for (int64_t t = 0; t < num_tokens; ++t)
        if (slot_mapping[t] >= num_blocks * page_size) return ORACLE_BAD_BLOCK;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t s = slot_mapping[t];
        if (s < 0) continue;
        const int64_t page = s / page_size, slot = s % page_size;
        memcpy(k_cache + (page * page_size + slot) * row, k_new + t * row, sizeof(uint16_t) * (size_t)row);
        memcpy(v_cache + (page * page_size + slot) * row, v_new + t * row, sizeof(uint16_t) * (size_t)row);
    }
    return ORACLE_OK;
}
