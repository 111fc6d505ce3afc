/*
 * CPU oracle for the paged KV write and ragged paged attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark load this library.  It shares no code,
 * header, table or helper with the CUDA library: it is a plain, slow and
 * obviously correct restatement of what the pages define, one loop per
 * index, in double precision.
 *
 * Sources (page title, section):
 *  - "31. Engine v2: one core for every request", "Flattened ragged batches":
 *    position p of a request lives in slot table[p / bs] * bs + p % bs.
 *  - same page, "Attention over the pool": the pool per layer is
 *    [num_blocks, block_size, kv_heads, head_dim]; write_kv scatters the
 *    step's rows to their slots, a slot of -1 (padding row) goes to the
 *    pool's last slot (scratch block); the reference backend gives
 *    request r's t queries positions seq_len - t + i, each sees keys
 *    0 .. its position, padding requests (seq_len 0 or no rows) leave zeros;
 *    with a sliding window w > 0 a query at position p sees only the keys
 *    at positions above p - w (the backend's `window` argument).
 *  - vllm-lite README, grouped-query attention: query heads fold onto KV
 *    heads in contiguous groups, query head h reads KV head h / (Hq / Hkv).
 *  - attention itself: softmax(scale * q . k) weighted sum of v over the
 *    visible keys (exact attention; "vLLM: LLM Inference as a memory and
 *    scheduling problem", "FlashAttention is not PagedAttention").
 *
 * Readings where the pages are silent (each listed with the design notes):
 *  - values are bf16 bit patterns (uint16_t); widening to double is exact;
 *  - accumulation and exp are done in double; the output is double;
 *  - the scale is the caller's (1/sqrt(head_dim) when the caller passes 0).
 *
 * Every pin of this file is in tests/test_oracle_pins.py.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 bit pattern -> double, exact (bf16 is the top half of an IEEE float). */
static double widen(uint16_t b)
{
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* The slot formula of the batch builder: table[p / bs] * bs + p % bs. */
int64_t oracle_slot(const int32_t *table_row, int64_t p, int32_t bs)
{
    return (int64_t)table_row[p / bs] * bs + p % bs;
}

/*
 * write_kv: for every row i of the step, in order, copy k[i] and v[i]
 * ([Hkv][d] raw bf16 values) to the pool slot slot_mapping[i]; a negative
 * slot is a padding row and goes to the pool's last slot.
 * Returns 0, or -1 if a slot is out of the pool.
 */
int oracle_paged_kv_write(uint16_t *k_cache, uint16_t *v_cache,
                          const uint16_t *k, const uint16_t *v,
                          const int64_t *slot_mapping, int32_t num_tokens,
                          int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks_total)
{
    int64_t row = (int64_t)num_kv_heads * head_dim;      /* elements per slot */
    int64_t scratch = (int64_t)num_blocks_total * block_size - 1;
    for (int32_t i = 0; i < num_tokens; i++) {
        int64_t s = slot_mapping[i] >= 0 ? slot_mapping[i] : scratch;
        if (s > scratch)
            return -1;
        for (int32_t h = 0; h < num_kv_heads; h++) {
            for (int32_t e = 0; e < head_dim; e++) {
                int64_t dst = s * row + (int64_t)h * head_dim + e;
                int64_t src = (int64_t)i * row + (int64_t)h * head_dim + e;
                k_cache[dst] = k[src];
                v_cache[dst] = v[src];
            }
        }
    }
    return 0;
}

/* Everything one attention row needs.  A quantized pool gives k8/v8 codes
 * and ks/vs scales instead of k_cache/v_cache. */
struct problem {
    const uint16_t *q, *k_cache, *v_cache;
    const int32_t *qsl, *seq_lens, *block_table;
    int32_t stride, num_reqs, num_tokens, hq, hkv, d, bs, nb_total;
    double scale;
    int32_t window;                                 /* 0: none; else keys above p - window */
    const uint8_t *k8, *v8;                         /* E4M3 codes, or NULL */
    const float *ks, *vs;                           /* their per (slot, head) scales */
};

double oracle_e4m3_decode(uint8_t c);

/* element e of the K (which = 0) or V (1) row of `slot`, KV head kh */
static double pool_value(const struct problem *P, int which, int64_t slot, int32_t kh, int32_t e)
{
    int64_t row = slot * P->hkv + kh;
    if (P->k8) {
        const uint8_t *codes = which ? P->v8 : P->k8;
        const float *scales = which ? P->vs : P->ks;
        return oracle_e4m3_decode(codes[row * P->d + e]) * (double)scales[row];
    }
    return widen((which ? P->v_cache : P->k_cache)[row * P->d + e]);
}

/*
 * Output row (token n, query head h) of request r: the query sits at
 * position p = L - t + i and attends to keys j0..p of its context, read
 * through the block table: j0 = 0, or with a sliding window w the first
 * key above p - w.  scores[] holds p + 1 doubles.
 */
static int attend_row(const struct problem *P, int32_t r, int32_t n, int32_t h,
                      double *scores, double *out_row)
{
    int32_t begin = P->qsl[r], t = P->qsl[r + 1] - begin, L = P->seq_lens[r];
    int32_t i = n - begin;
    int32_t g = P->hq / P->hkv;
    int32_t kh = h / g;
    int64_t p = (int64_t)L - t + i;
    const uint16_t *qrow = P->q + ((int64_t)n * P->hq + h) * P->d;
    const int32_t *table = P->block_table + (int64_t)r * P->stride;

    for (int32_t e = 0; e < P->d; e++)
        out_row[e] = 0.0;
    if (L == 0 || t == 0)
        return 0;                                   /* padding request: zeros */

    int64_t j0 = 0;
    if (P->window > 0 && p - P->window + 1 > 0)
        j0 = p - P->window + 1;
    double m = -INFINITY;
    for (int64_t j = j0; j <= p; j++) {
        int32_t blk = table[j / P->bs];
        if (blk < 0 || blk >= P->nb_total)
            return -1;
        int64_t slot = (int64_t)blk * P->bs + j % P->bs;
        double s = 0.0;
        for (int32_t e = 0; e < P->d; e++)
            s += widen(qrow[e]) * pool_value(P, 0, slot, kh, e);
        s *= P->scale;
        scores[j] = s;
        if (s > m)
            m = s;
    }
    double l = 0.0;
    for (int64_t j = j0; j <= p; j++) {
        double w = exp(scores[j] - m);
        scores[j] = w;
        l += w;
    }
    for (int64_t j = j0; j <= p; j++) {
        int32_t blk = table[j / P->bs];
        int64_t slot = (int64_t)blk * P->bs + j % P->bs;
        for (int32_t e = 0; e < P->d; e++)
            out_row[e] += scores[j] * pool_value(P, 1, slot, kh, e);
    }
    for (int32_t e = 0; e < P->d; e++)
        out_row[e] /= l;
    return 0;
}

static int check_problem(const struct problem *P)
{
    if (P->hkv <= 0 || P->hq <= 0 || P->hq % P->hkv != 0 || P->d <= 0 || P->bs <= 0 || P->window < 0)
        return -2;
    if (P->qsl[0] != 0 || P->qsl[P->num_reqs] != P->num_tokens)
        return -2;
    for (int32_t r = 0; r < P->num_reqs; r++) {
        int32_t t = P->qsl[r + 1] - P->qsl[r];
        int32_t L = P->seq_lens[r];
        if (t < 0 || L < 0)
            return -2;
        if (L > 0 && t > L)
            return -2;
        if (L > 0 && (L + P->bs - 1) / P->bs > P->stride)
            return -2;
    }
    return 0;
}

/* request of every row: the r with qsl[r] <= n < qsl[r + 1] */
static int32_t *rows_to_requests(const struct problem *P)
{
    int32_t *owner = (int32_t *)malloc(sizeof(int32_t) * (size_t)(P->num_tokens > 0 ? P->num_tokens : 1));
    if (!owner)
        return NULL;
    for (int32_t r = 0; r < P->num_reqs; r++)
        for (int32_t n = P->qsl[r]; n < P->qsl[r + 1]; n++)
            owner[n] = r;
    return owner;
}

static int32_t max_seq(const struct problem *P)
{
    int32_t m = 1;
    for (int32_t r = 0; r < P->num_reqs; r++)
        if (P->seq_lens[r] > m)
            m = P->seq_lens[r];
    return m;
}

/*
 * Full ragged paged attention: out is double [num_tokens][hq][d].
 * nthreads > 1 splits the independent (row, head) outputs across OpenMP
 * threads; every output is computed by the same loop either way.
 * Returns 0, -1 on an out-of-pool block id, -2 on inconsistent metadata,
 * -3 when memory runs out.
 */
static int run_all_rows(const struct problem *PP, double *out, int32_t nthreads);

int oracle_ragged_paged_attention(double *out, const uint16_t *q,
                                  const uint16_t *k_cache, const uint16_t *v_cache,
                                  const int32_t *query_start_loc, const int32_t *seq_lens,
                                  const int32_t *block_table, int32_t block_table_stride,
                                  int32_t num_reqs, int32_t num_tokens,
                                  int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                  int32_t block_size, int32_t num_blocks_total,
                                  double scale, int32_t window, int32_t nthreads)
{
    struct problem P = {q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                        block_table_stride, num_reqs, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks_total, scale, window, NULL, NULL, NULL, NULL};
    return run_all_rows(&P, out, nthreads);
}

/* The same attention over a quantized pool: keys and values are E4M3 codes
 * times their (slot, head) scale, dequantized exactly in double. */
int oracle_ragged_paged_attention_fp8(double *out, const uint16_t *q,
                                      const uint8_t *k_codes, const uint8_t *v_codes,
                                      const float *k_scale, const float *v_scale,
                                      const int32_t *query_start_loc, const int32_t *seq_lens,
                                      const int32_t *block_table, int32_t block_table_stride,
                                      int32_t num_reqs, int32_t num_tokens,
                                      int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                                      int32_t block_size, int32_t num_blocks_total,
                                      double scale, int32_t window, int32_t nthreads)
{
    struct problem P = {q, NULL, NULL, query_start_loc, seq_lens, block_table,
                        block_table_stride, num_reqs, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks_total, scale, window,
                        k_codes, v_codes, k_scale, v_scale};
    return run_all_rows(&P, out, nthreads);
}

static int run_all_rows(const struct problem *PP, double *out, int32_t nthreads)
{
    struct problem P = *PP;
    int32_t num_tokens = P.num_tokens, num_q_heads = P.hq, head_dim = P.d;
    int rc = check_problem(&P);
    if (rc)
        return rc;
    int32_t *owner = rows_to_requests(&P);
    if (!owner)
        return -3;
    int32_t lmax = max_seq(&P);
    int64_t total = (int64_t)num_tokens * num_q_heads;
    int status = 0;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)lmax);
        int local = scores ? 0 : -3;
#pragma omp for schedule(dynamic, 1)
        for (int64_t x = 0; x < total; x++) {
            if (local)
                continue;
            int32_t n = (int32_t)(x / num_q_heads), h = (int32_t)(x % num_q_heads);
            int e = attend_row(&P, owner[n], n, h, scores, out + x * head_dim);
            if (e)
                local = e;
        }
        if (local) {
#pragma omp critical
            status = local;
        }
        free(scores);
    }
    free(owner);
    return status;
}

static int run_rows(const struct problem *PP, double *out, const int32_t *tokens, const int32_t *heads,
                    int32_t count, int32_t nthreads);

/*
 * Selected outputs only: for k < count, out[k][0..d) = output of row
 * tokens[k], query head heads[k].  Same arithmetic as above; for checking
 * sampled outputs of full-size workloads.
 */
int oracle_attention_rows(double *out, const int32_t *tokens, const int32_t *heads, int32_t count,
                          const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *query_start_loc, const int32_t *seq_lens,
                          const int32_t *block_table, int32_t block_table_stride,
                          int32_t num_reqs, int32_t num_tokens,
                          int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                          int32_t block_size, int32_t num_blocks_total,
                          double scale, int32_t window, int32_t nthreads)
{
    struct problem P = {q, k_cache, v_cache, query_start_loc, seq_lens, block_table,
                        block_table_stride, num_reqs, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks_total, scale, window, NULL, NULL, NULL, NULL};
    return run_rows(&P, out, tokens, heads, count, nthreads);
}

/* Selected outputs over a quantized pool. */
int oracle_attention_rows_fp8(double *out, const int32_t *tokens, const int32_t *heads, int32_t count,
                              const uint16_t *q, const uint8_t *k_codes, const uint8_t *v_codes,
                              const float *k_scale, const float *v_scale,
                              const int32_t *query_start_loc, const int32_t *seq_lens,
                              const int32_t *block_table, int32_t block_table_stride,
                              int32_t num_reqs, int32_t num_tokens,
                              int32_t num_q_heads, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks_total,
                              double scale, int32_t window, int32_t nthreads)
{
    struct problem P = {q, NULL, NULL, query_start_loc, seq_lens, block_table,
                        block_table_stride, num_reqs, num_tokens, num_q_heads, num_kv_heads,
                        head_dim, block_size, num_blocks_total, scale, window,
                        k_codes, v_codes, k_scale, v_scale};
    return run_rows(&P, out, tokens, heads, count, nthreads);
}

static int run_rows(const struct problem *PP, double *out, const int32_t *tokens, const int32_t *heads,
                    int32_t count, int32_t nthreads)
{
    struct problem P = *PP;
    int32_t num_tokens = P.num_tokens, num_q_heads = P.hq, head_dim = P.d;
    int rc = check_problem(&P);
    if (rc)
        return rc;
    int32_t *owner = rows_to_requests(&P);
    if (!owner)
        return -3;
    int32_t lmax = max_seq(&P);
    int status = 0;
    if (nthreads < 1)
        nthreads = 1;
#pragma omp parallel num_threads(nthreads)
    {
        double *scores = (double *)malloc(sizeof(double) * (size_t)lmax);
        int local = scores ? 0 : -3;
#pragma omp for schedule(dynamic, 1)
        for (int32_t k = 0; k < count; k++) {
            if (local)
                continue;
            if (tokens[k] < 0 || tokens[k] >= num_tokens || heads[k] < 0 || heads[k] >= num_q_heads) {
                local = -2;
                continue;
            }
            int e = attend_row(&P, owner[tokens[k]], tokens[k], heads[k], scores,
                               out + (int64_t)k * head_dim);
            if (e)
                local = e;
        }
        if (local) {
#pragma omp critical
            status = local;
        }
        free(scores);
    }
    free(owner);
    return status;
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Block copies of the block manager.  "vllm-lite README": blocks are
 * reference counted; a write into a block two sequences share is preceded
 * by a copy of that block, which the runner makes before the forward pass.
 * "31. Engine v2", "Preemption: recompute or swap": swap-out copies a
 * preempted request's blocks (every layer's K and V) to host memory, and
 * swap-in copies them back into newly allocated blocks.  A pool is viewed
 * as nb_total blocks of block_bytes bytes (the slot-major layout keeps a
 * block contiguous).  Copies are byte copies applied in list order.
 * Each returns 0, or -1 at the first block id outside the pool.
 */
int oracle_copy_blocks(uint8_t *pool, const int32_t *src, const int32_t *dst, int32_t n, int32_t nb_total,
                       int64_t block_bytes)
{
    for (int32_t i = 0; i < n; i++) {
        if (src[i] < 0 || src[i] >= nb_total || dst[i] < 0 || dst[i] >= nb_total)
            return -1;
        for (int64_t b = 0; b < block_bytes; b++)
            pool[(int64_t)dst[i] * block_bytes + b] = pool[(int64_t)src[i] * block_bytes + b];
    }
    return 0;
}

/* out[i] := block blocks[i] (out is n * block_bytes bytes). */
int oracle_gather_blocks(uint8_t *out, const uint8_t *pool, const int32_t *blocks, int32_t n, int32_t nb_total,
                         int64_t block_bytes)
{
    for (int32_t i = 0; i < n; i++) {
        if (blocks[i] < 0 || blocks[i] >= nb_total)
            return -1;
        for (int64_t b = 0; b < block_bytes; b++)
            out[(int64_t)i * block_bytes + b] = pool[(int64_t)blocks[i] * block_bytes + b];
    }
    return 0;
}

/* block blocks[i] := in[i]. */
int oracle_scatter_blocks(uint8_t *pool, const uint8_t *in, const int32_t *blocks, int32_t n, int32_t nb_total,
                          int64_t block_bytes)
{
    for (int32_t i = 0; i < n; i++) {
        if (blocks[i] < 0 || blocks[i] >= nb_total)
            return -1;
        for (int64_t b = 0; b < block_bytes; b++)
            pool[(int64_t)blocks[i] * block_bytes + b] = in[(int64_t)i * block_bytes + b];
    }
    return 0;
}

/*
 * Quantized pools.  "31. Engine v2", "Attention over the pool": a quantized
 * pool carries its scales next to K and V (cache[2], cache[3]), one per slot
 * and KV head, and the reference backend dequantizes a gathered row as
 * x.float() * scale.  The pages leave the code format and the quantizing
 * write open; this oracle takes the plain reading used with an fp8 KV cache:
 * FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 mantissa bits, no
 * infinities, largest finite 448), per (slot, head) scale = max |x| / 448
 * computed in fp32, code = E4M3(x / scale) with the fp32 quotient rounded to
 * nearest-even and clamped to +-448; a row of zeros gets scale 0 and codes 0.
 */

/* E4M3 code -> value (exact). */
double oracle_e4m3_decode(uint8_t c)
{
    int sign = c >> 7, field = (c >> 3) & 15, man = c & 7;
    double v;
    if (field == 15 && man == 7)
        return NAN;
    if (field == 0)
        v = man * ldexp(1.0, -9);                   /* subnormal: man/8 * 2^-6 */
    else
        v = (1.0 + man / 8.0) * ldexp(1.0, field - 7);
    return sign ? -v : v;
}

/* round half to even of a non-negative double */
static double round_half_even(double y)
{
    double f = floor(y), r = y - f;
    if (r > 0.5 || (r == 0.5 && fmod(f, 2.0) != 0.0))
        return f + 1.0;
    return f;
}

/* fp32 value -> E4M3 code, round to nearest even, saturating at +-448. */
uint8_t oracle_e4m3_encode(float x)
{
    uint8_t sign = signbit(x) ? 0x80 : 0;
    double a = fabs((double)x);
    if (a >= 448.0)
        return sign | 0x7E;                          /* 1111.110 = 448 */
    if (a < ldexp(1.0, -6)) {                        /* subnormal range: k * 2^-9 */
        double k = round_half_even(a / ldexp(1.0, -9));
        return sign | (uint8_t)k;                    /* k == 8 is 0x08, the smallest normal */
    }
    int e;
    frexp(a, &e);                                    /* a = f * 2^e, f in [0.5, 1) */
    e -= 1;                                          /* a = m * 2^e, m in [1, 2) */
    double m3 = round_half_even((a / ldexp(1.0, e) - 1.0) * 8.0);
    if (m3 == 8.0) {
        m3 = 0.0;
        e += 1;
    }
    return sign | (uint8_t)(((e + 7) << 3) | (int)m3);
}

/* the quantizing write: like oracle_paged_kv_write, with codes and scales */
int oracle_paged_kv_write_fp8(uint8_t *k_cache, uint8_t *v_cache, float *k_scale, float *v_scale,
                              const uint16_t *k, const uint16_t *v, const int64_t *slot_mapping,
                              int32_t num_tokens, int32_t num_kv_heads, int32_t head_dim,
                              int32_t block_size, int32_t num_blocks_total)
{
    int64_t scratch = (int64_t)num_blocks_total * block_size - 1;
    for (int32_t i = 0; i < num_tokens; i++) {
        int64_t s = slot_mapping[i] >= 0 ? slot_mapping[i] : scratch;
        if (s > scratch)
            return -1;
        for (int32_t h = 0; h < num_kv_heads; h++) {
            for (int which = 0; which < 2; which++) {
                const uint16_t *src = (which ? v : k) + ((int64_t)i * num_kv_heads + h) * head_dim;
                uint8_t *dst = (which ? v_cache : k_cache) + (s * num_kv_heads + h) * head_dim;
                float amax = 0.0f;
                for (int32_t e = 0; e < head_dim; e++) {
                    float a = fabsf((float)widen(src[e]));
                    if (a > amax)
                        amax = a;
                }
                float scale = amax / 448.0f;             /* fp32 division */
                for (int32_t e = 0; e < head_dim; e++)
                    dst[e] = scale > 0.0f ? oracle_e4m3_encode((float)widen(src[e]) / scale) : 0;
                (which ? v_scale : k_scale)[s * num_kv_heads + h] = scale;
            }
        }
    }
    return 0;
}
