/*
 * Plain CPU oracle for the QSA indexer step (score every causally visible
 * compressed index-key position, then take the exact top-k).
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or call
 * this file: only the tests, the smoke check and the benchmark's CPU-baseline
 * leg use it.  It shares no code, header or constant with the CUDA library.
 *
 * What it follows (pages of the block_sparse_attention_select set):
 *  - "spec(MODEL-MM-QWEN4-EXP) ...", section "The component deep-dives":
 *    the index score is relu(q.k) summed over the index heads, one score per
 *    query token with no head axis, an MQA index with one key head of dim 128,
 *    compress ratio 4, the (position+1) % COMPRESS_RATIO == 0 boundary and
 *    "candidates counted as visible // compress_ratio".
 *  - "[Perf][Qwen4Exp] Admit the cuBLAS QSA indexer and exact top-k on Turing",
 *    section "Purpose": FP16 operands with FP32 accumulation, and an *exact*
 *    lexicographic top-k with a deterministic tie rule (a non-exact selector
 *    "can pick a different block set when scores tie at the cutoff").
 *  - The pages do not spell out how the heads are weighted or which of two
 *    equal scores wins.  Readings taken: ReLU per head first, then the
 *    per-row head weight, then the sum over the heads in order h = 0 .. H-1
 *    (logit = sum_h w[r,h] * ReLU(q[r,h] . k[j]); w may be any finite value,
 *    1/sqrt(head_dim) folded into it by the caller); the higher score first
 *    and, on equal scores, the lower position index; -0 and +0 are equal
 *    scores; positions j >= V_r are never candidates (their logits are -inf).
 *
 * Arithmetic: IEEE binary32, multiply then add in a fixed order, no fused
 * multiply-add (the build passes -ffp-contract=off).  Products of two binary16
 * values are exact in binary32, so only the additions round.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* IEEE 754 binary16 -> binary32, from the format's definition:
 * sign 1 bit, exponent 5 bits (bias 15), fraction 10 bits.
 * exponent 0: subnormal, value = fraction * 2^-24; exponent 31: inf / NaN. */
float oracle_half_to_float(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int expo = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    float mag;
    if (expo == 0) {
        mag = ldexpf((float)frac, -24);              /* exact: frac < 2^10 */
    } else if (expo == 31) {
        mag = frac ? NAN : INFINITY;
    } else {
        mag = ldexpf((float)(1024 + frac), expo - 25); /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -mag : mag;
}

/* Number of compressed positions a query at 0-based token position t sees.
 * Compressed position p covers tokens 4p .. 4p+3 (ratio 4) and is stored once
 * its last token exists, i.e. at the (position+1) % ratio == 0 boundary; the
 * count is therefore (t+1) // ratio ("visible // compress_ratio"). */
int64_t oracle_visible_positions(int64_t t, int32_t ratio)
{
    if (t < 0 || ratio <= 0) return 0;
    return (t + 1) / ratio;
}

/* logits[r, j] for every row r and 0 <= j < ld:
 *   j <  V_r : sum_{h=0..H-1} w[r,h] * max(q[r,h,:] . k_j, 0)      (then +0.0f)
 *   j >= V_r : -inf
 * where k_j = k_cache[block_table[row_req[r], j / P], j % P, :] and P is the
 * page size in positions.  q is [R, H, D] binary16, k_cache is
 * [num_pages, P, D] binary16, block_table is [num_reqs, max_pages]. */
void oracle_score(const uint16_t *q, const float *w, int32_t R, int32_t H, int32_t D,
                  const uint16_t *k_cache, int32_t num_pages, int32_t page_positions,
                  const int32_t *block_table, int32_t max_pages,
                  const int32_t *row_req, const int32_t *row_visible,
                  float *logits, int64_t ld, int32_t nthreads)
{
    (void)num_pages;
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int32_t r = 0; r < R; ++r) {
        float *out = logits + (int64_t)r * ld;
        const int32_t b = row_req[r];
        const int64_t V = row_visible[r];
        float *qf = (float *)malloc(sizeof(float) * (size_t)H * (size_t)D);
        float *kf = (float *)malloc(sizeof(float) * (size_t)D);
        for (int64_t i = 0; i < (int64_t)H * D; ++i)
            qf[i] = oracle_half_to_float(q[(int64_t)r * H * D + i]);
        for (int64_t j = 0; j < ld; ++j) {
            if (j >= V) { out[j] = -INFINITY; continue; }
            const int64_t page = block_table[(int64_t)b * max_pages + j / page_positions];
            const uint16_t *kj = k_cache + (page * page_positions + j % page_positions) * D;
            for (int32_t t = 0; t < D; ++t) kf[t] = oracle_half_to_float(kj[t]);
            float s = 0.0f;
            for (int32_t h = 0; h < H; ++h) {
                float dot = 0.0f;
                for (int32_t t = 0; t < D; ++t) dot = dot + qf[h * D + t] * kf[t];
                const float relu = dot > 0.0f ? dot : 0.0f;
                s = s + w[(int64_t)r * H + h] * relu;
            }
            out[j] = s + 0.0f;   /* a -0 (negative weight times +0) becomes +0 */
        }
        free(kf);
        free(qf);
    }
}

typedef struct { float v; int32_t j; } scored_t;

/* Strict total order of the selector: higher score first, then lower index. */
static int by_score_desc_index_asc(const void *pa, const void *pb)
{
    const scored_t *a = (const scored_t *)pa, *b = (const scored_t *)pb;
    if (a->v > b->v) return -1;
    if (a->v < b->v) return 1;
    return (a->j > b->j) - (a->j < b->j);
}

/* Exact top-k of row r over its visible positions 0 <= j < V_r: a full sort by
 * (score desc, index asc), truncated to min(k, V_r); the remaining output
 * slots hold index -1 and value -inf.  out_val may be NULL. */
void oracle_select(const float *logits, int64_t ld, int32_t R, const int32_t *row_visible,
                   int32_t k, int32_t *out_idx, float *out_val, int32_t nthreads)
{
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#pragma omp parallel for schedule(dynamic, 1)
#endif
    for (int32_t r = 0; r < R; ++r) {
        int64_t V = row_visible[r] < ld ? row_visible[r] : ld;
        if (V < 0) V = 0;
        scored_t *all = (scored_t *)malloc(sizeof(scored_t) * (size_t)(V > 0 ? V : 1));
        for (int64_t j = 0; j < V; ++j) {
            all[j].v = logits[(int64_t)r * ld + j];
            all[j].j = (int32_t)j;
        }
        qsort(all, (size_t)V, sizeof(scored_t), by_score_desc_index_asc);
        for (int64_t i = 0; i < k; ++i) {
            const int has = i < V;
            out_idx[(int64_t)r * k + i] = has ? all[i].j : -1;
            if (out_val) out_val[(int64_t)r * k + i] = has ? all[i].v : -INFINITY;
        }
        free(all);
    }
}

/* Independent selector for tiny inputs: k rounds of "take the largest score
 * not yet taken, the lowest index among equal scores". O(V * k). */
void oracle_select_bruteforce(const float *logits, int64_t ld, int32_t R,
                              const int32_t *row_visible, int32_t k,
                              int32_t *out_idx, float *out_val)
{
    for (int32_t r = 0; r < R; ++r) {
        int64_t V = row_visible[r] < ld ? row_visible[r] : ld;
        if (V < 0) V = 0;
        const float *row = logits + (int64_t)r * ld;
        unsigned char *taken = (unsigned char *)calloc((size_t)(V > 0 ? V : 1), 1);
        for (int64_t i = 0; i < k; ++i) {
            int64_t best = -1;
            for (int64_t j = 0; j < V; ++j) {
                if (taken[j]) continue;
                if (best < 0 || row[j] > row[best]) best = j;   /* strict: first max wins */
            }
            if (best >= 0) taken[best] = 1;
            out_idx[(int64_t)r * k + i] = (int32_t)best;
            if (out_val) out_val[(int64_t)r * k + i] = best >= 0 ? row[best] : -INFINITY;
        }
        free(taken);
    }
}

int32_t oracle_max_threads(void)
{
#ifdef _OPENMP
    return (int32_t)omp_get_max_threads();
#else
    return 1;
#endif
}
