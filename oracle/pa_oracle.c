/*
 * Plain fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library links, loads or
 * calls this file; only the tests, the package's smoke check and the
 * benchmark's CPU-baseline leg do.  It shares no code, header or constant with
 * the CUDA path.
 *
 * Sources (web pages, cited by title and section):
 *   [P1] "LLM推理优化：vLLM PagedAttention深度解析与工程实践" (lpnh.cn/news/754185)
 *        section 二 (attention formula softmax(Q*K^T/sqrt(d))*V),
 *        section 3.1 (block table: logical block -> physical block, 16 slots),
 *        section 4.1 (paged K layout [num_blocks, block_size, num_heads, head_dim]).
 *   [P3] "vLLM 深度拆解：当大模型推理学会「分页注意力」" (chenxutan.com/d/4834.html)
 *        section 1.1 (decode: the new token's query attends to all cached K/V),
 *        section 2.1 (block table maps logical positions to physical blocks).
 *   [P4] "LLM推理优化技术地图：从KV Cache到量化与投机解码" (qwbw.cn/news/280730)
 *        section 2.3 (GQA: query heads split into groups sharing one K/V head).
 *
 * What it computes (the plain definition; paging changes where K/V live, not
 * the arithmetic):
 *   for sequence i with n = context_lens[i] tokens and query head h,
 *     G   = H / Hkv, g = h / G                       (contiguous GQA groups)
 *     K_j = k_cache[tbl[i][j / bs], j % bs, g, :]     (V_j likewise), j < n
 *     s_j = scale * sum_k q[i,h,k] * K_j[k]
 *     w_j = exp(s_j - max s) / sum_l exp(s_l - max s)
 *     out[i,h,:] = sum_j w_j V_j
 *   all in fp64 from exactly converted fp16 / bf16 inputs; n == 0 gives zeros.
 *
 * Threads: sequences are split over POSIX threads; each (i, h) output is
 * computed by one thread with the same loop order as the single-thread run, so
 * the result does not depend on the thread count.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_OK 0
#define ORC_ERR_ARG 1
#define ORC_ERR_TABLE 2

/* IEEE 754 binary16 -> double, exact: sign, 5-bit biased exponent, 10-bit
 * fraction. */
static double orc_half_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(f + 1024), e - 25);     /* (1 + f/1024) * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE 754 binary32 -> exact in double. */
static double orc_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double orc_elem(const uint16_t* p, int64_t idx, int dtype) {
    return dtype == 1 ? orc_bf16_to_double(p[idx]) : orc_half_to_double(p[idx]);
}

typedef struct {
    const uint16_t *q, *k, *v;
    const int32_t *tbl, *lens;
    int32_t max_blocks, B, H, Hkv, d, bs, dtype;
    int64_t num_blocks;
    double scale;
    double* out;
    int32_t seq_begin, seq_end;
    int status;
} orc_job;

/* One query row (q at element offset qoff) of sequence i against its first n
 * cached tokens of KV head g; the result goes to o[0..d). */
static int orc_attend(const orc_job* J, int32_t i, int32_t g, int64_t qoff, int32_t n, double* o,
                      double* s /* [n] scratch */) {
    const int32_t d = J->d;
    for (int32_t k = 0; k < d; ++k) o[k] = 0.0;
    if (n == 0) return ORC_OK;

    /* logits */
    for (int32_t j = 0; j < n; ++j) {
        int32_t lb = j / J->bs;
        if (lb >= J->max_blocks) return ORC_ERR_TABLE;
        int32_t pb = J->tbl[(int64_t)i * J->max_blocks + lb];
        if (pb < 0 || (int64_t)pb >= J->num_blocks) return ORC_ERR_TABLE;
        int64_t row = (((int64_t)pb * J->bs + (j % J->bs)) * J->Hkv + g) * d;
        double acc = 0.0;
        for (int32_t k = 0; k < d; ++k)
            acc += orc_elem(J->q, qoff + k, J->dtype) * orc_elem(J->k, row + k, J->dtype);
        s[j] = J->scale * acc;
    }
    /* softmax, max-subtracted */
    double m = s[0];
    for (int32_t j = 1; j < n; ++j)
        if (s[j] > m) m = s[j];
    double sum = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        s[j] = exp(s[j] - m);
        sum += s[j];
    }
    /* weighted sum of V */
    for (int32_t j = 0; j < n; ++j) {
        int32_t pb = J->tbl[(int64_t)i * J->max_blocks + j / J->bs];
        int64_t row = (((int64_t)pb * J->bs + (j % J->bs)) * J->Hkv + g) * d;
        double w = s[j] / sum;
        for (int32_t k = 0; k < d; ++k) o[k] += w * orc_elem(J->v, row + k, J->dtype);
    }
    return ORC_OK;
}

/* One (sequence, query head) output row of the decode. */
static int orc_row(const orc_job* J, int32_t i, int32_t h, double* s /* [n] scratch */) {
    const int32_t G = J->H / J->Hkv;
    const int64_t off = ((int64_t)i * J->H + h) * J->d;
    return orc_attend(J, i, h / G, off, J->lens[i], J->out + off, s);
}

static void* orc_worker(void* arg) {
    orc_job* J = (orc_job*)arg;
    int32_t nmax = 1;
    for (int32_t i = J->seq_begin; i < J->seq_end; ++i)
        if (J->lens[i] > nmax) nmax = J->lens[i];
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    if (!s) {
        J->status = ORC_ERR_ARG;
        return NULL;
    }
    J->status = ORC_OK;
    for (int32_t i = J->seq_begin; i < J->seq_end && J->status == ORC_OK; ++i)
        for (int32_t h = 0; h < J->H && J->status == ORC_OK; ++h)
            J->status = orc_row(J, i, h, s);
    free(s);
    return NULL;
}

/*
 * q          [B, H, d]             fp16/bf16 bit patterns
 * k_cache    [num_blocks, bs, Hkv, d]
 * v_cache    [num_blocks, bs, Hkv, d]
 * block_tables [B, max_blocks] int32 physical block ids
 * context_lens [B] int32
 * dtype      0 = fp16, 1 = bf16
 * out        [B, H, d] double
 * Returns 0, or 1 for bad arguments, 2 for a table entry outside the pool.
 */
int pa_oracle_decode(const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                     const int32_t* block_tables, int32_t max_blocks, const int32_t* context_lens,
                     int32_t B, int32_t H, int32_t Hkv, int32_t d, int32_t block_size,
                     int64_t num_blocks, double scale, int32_t dtype, double* out,
                     int32_t num_threads) {
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || d <= 0 || block_size <= 0 ||
        max_blocks < 0 || num_blocks < 0 || (dtype != 0 && dtype != 1))
        return ORC_ERR_ARG;
    for (int32_t i = 0; i < B; ++i)
        if (context_lens[i] < 0) return ORC_ERR_ARG;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > B) num_threads = B > 0 ? B : 1;

    orc_job* jobs = (orc_job*)calloc((size_t)num_threads, sizeof(orc_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return ORC_ERR_ARG;
    }
    for (int t = 0; t < num_threads; ++t) {
        orc_job* J = &jobs[t];
        J->q = q; J->k = k_cache; J->v = v_cache;
        J->tbl = block_tables; J->lens = context_lens;
        J->max_blocks = max_blocks; J->B = B; J->H = H; J->Hkv = Hkv; J->d = d;
        J->bs = block_size; J->dtype = dtype; J->num_blocks = num_blocks;
        J->scale = scale; J->out = out;
        /* sequences are dealt out in contiguous ranges */
        J->seq_begin = (int32_t)((int64_t)B * t / num_threads);
        J->seq_end = (int32_t)((int64_t)B * (t + 1) / num_threads);
    }
    int rc = ORC_OK;
    if (num_threads == 1) {
        orc_worker(&jobs[0]);
    } else {
        for (int t = 0; t < num_threads; ++t) pthread_create(&th[t], NULL, orc_worker, &jobs[t]);
        for (int t = 0; t < num_threads; ++t) pthread_join(th[t], NULL);
    }
    for (int t = 0; t < num_threads; ++t)
        if (jobs[t].status != ORC_OK) rc = jobs[t].status;
    free(jobs);
    free(th);
    return rc;
}

/*
 * The softmax weights w_j of one (sequence i, query head h), for the
 * invariant that they sum to one.  w must hold context_lens[i] doubles.
 */
int pa_oracle_weights(const uint16_t* q, const uint16_t* k_cache, const int32_t* block_tables,
                      int32_t max_blocks, const int32_t* context_lens, int32_t B, int32_t H,
                      int32_t Hkv, int32_t d, int32_t block_size, int64_t num_blocks, double scale,
                      int32_t dtype, int32_t i, int32_t h, double* w) {
    if (i < 0 || i >= B || h < 0 || h >= H || H % Hkv != 0) return ORC_ERR_ARG;
    const int32_t n = context_lens[i];
    const int32_t g = h / (H / Hkv);
    const int64_t qoff = ((int64_t)i * H + h) * d;
    for (int32_t j = 0; j < n; ++j) {
        int32_t lb = j / block_size;
        if (lb >= max_blocks) return ORC_ERR_TABLE;
        int32_t pb = block_tables[(int64_t)i * max_blocks + lb];
        if (pb < 0 || (int64_t)pb >= num_blocks) return ORC_ERR_TABLE;
        int64_t row = (((int64_t)pb * block_size + (j % block_size)) * Hkv + g) * d;
        double acc = 0.0;
        for (int32_t k = 0; k < d; ++k)
            acc += orc_elem(q, qoff + k, dtype) * orc_elem(k_cache, row + k, dtype);
        w[j] = scale * acc;
    }
    if (n == 0) return ORC_OK;
    double m = w[0];
    for (int32_t j = 1; j < n; ++j)
        if (w[j] > m) m = w[j];
    double sum = 0.0;
    for (int32_t j = 0; j < n; ++j) {
        w[j] = exp(w[j] - m);
        sum += w[j];
    }
    for (int32_t j = 0; j < n; ++j) w[j] /= sum;
    return ORC_OK;
}

/* Exact conversion of a buffer of fp16 / bf16 bit patterns to double. */
int pa_oracle_to_double(const uint16_t* x, int64_t count, int32_t dtype, double* y) {
    if (dtype != 0 && dtype != 1) return ORC_ERR_ARG;
    for (int64_t t = 0; t < count; ++t) y[t] = orc_elem(x, t, dtype);
    return ORC_OK;
}

/*
 * FP8 KV cache (OCP 8-bit floating point, E4M3: 1 sign bit, 4 exponent bits
 * with bias 7, 3 mantissa bits, no infinities, 0x7F / 0xFF are NaN, largest
 * finite 448).  The cache holds codes [num_blocks][bs][Hkv][d] and one fp32
 * scale per token and KV head, laid out [num_blocks][Hkv][bs]; element j of
 * K is code_value * scale.  Same attention as pa_oracle_decode otherwise.
 */
static double orc_e4m3_to_double(uint8_t b) {
    int sign = (b >> 7) & 1;
    int e = (b >> 3) & 0xf;
    int m = b & 7;
    double v;
    if (e == 15 && m == 7)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)m, -9);          /* (m / 8) * 2^-6 */
    else
        v = ldexp((double)(m + 8), e - 10); /* (1 + m / 8) * 2^(e - 7) */
    return sign ? -v : v;
}

int pa_oracle_e4m3_to_double(const uint8_t* x, int64_t count, double* y) {
    for (int64_t t = 0; t < count; ++t) y[t] = orc_e4m3_to_double(x[t]);
    return ORC_OK;
}

/*
 * INT8 KV cache: a code is a two's-complement byte c in [-127, 127] and the
 * element is c * scale (same layouts and scales as E4M3).
 */
static double orc_code_to_double(uint8_t b, int32_t kind) {
    return kind == 0 ? orc_e4m3_to_double(b) : (double)(int8_t)b;
}

/* Attention over an 8-bit cache: kind 0 = E4M3 codes, 1 = INT8 codes. */
static int orc_decode_q8(const uint16_t* q, int32_t q_dtype, int32_t kind,
                         const uint8_t* k_codes, const uint8_t* v_codes, const float* k_scale,
                         const float* v_scale, const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* context_lens, int32_t B, int32_t H, int32_t Hkv,
                         int32_t d, int32_t block_size, int64_t num_blocks, double scale,
                         double* out) {
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || d <= 0 || block_size <= 0 ||
        (q_dtype != 0 && q_dtype != 1))
        return ORC_ERR_ARG;
    const int32_t G = H / Hkv;
    int32_t nmax = 1;
    for (int32_t i = 0; i < B; ++i) {
        if (context_lens[i] < 0) return ORC_ERR_ARG;
        if (context_lens[i] > nmax) nmax = context_lens[i];
    }
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    if (!s) return ORC_ERR_ARG;
    for (int32_t i = 0; i < B; ++i) {
        const int32_t n = context_lens[i];
        for (int32_t h = 0; h < H; ++h) {
            const int32_t g = h / G;
            double* o = out + ((int64_t)i * H + h) * d;
            for (int32_t k = 0; k < d; ++k) o[k] = 0.0;
            if (n == 0) continue;
            const int64_t qoff = ((int64_t)i * H + h) * d;
            for (int32_t j = 0; j < n; ++j) {
                int32_t lb = j / block_size;
                if (lb >= max_blocks) { free(s); return ORC_ERR_TABLE; }
                int32_t pb = block_tables[(int64_t)i * max_blocks + lb];
                if (pb < 0 || (int64_t)pb >= num_blocks) { free(s); return ORC_ERR_TABLE; }
                int64_t row = (((int64_t)pb * block_size + (j % block_size)) * Hkv + g) * d;
                double ks = (double)k_scale[((int64_t)pb * Hkv + g) * block_size + j % block_size];
                double acc = 0.0;
                for (int32_t k = 0; k < d; ++k)
                    acc += orc_elem(q, qoff + k, q_dtype) * (orc_code_to_double(k_codes[row + k], kind) * ks);
                s[j] = scale * acc;
            }
            double m = s[0];
            for (int32_t j = 1; j < n; ++j)
                if (s[j] > m) m = s[j];
            double sum = 0.0;
            for (int32_t j = 0; j < n; ++j) {
                s[j] = exp(s[j] - m);
                sum += s[j];
            }
            for (int32_t j = 0; j < n; ++j) {
                int32_t pb = block_tables[(int64_t)i * max_blocks + j / block_size];
                int64_t row = (((int64_t)pb * block_size + (j % block_size)) * Hkv + g) * d;
                double vs = (double)v_scale[((int64_t)pb * Hkv + g) * block_size + j % block_size];
                double w = s[j] / sum;
                for (int32_t k = 0; k < d; ++k)
                    o[k] += w * (orc_code_to_double(v_codes[row + k], kind) * vs);
            }
        }
    }
    free(s);
    return ORC_OK;
}

int pa_oracle_decode_fp8(const uint16_t* q, int32_t q_dtype, const uint8_t* k_codes,
                         const uint8_t* v_codes, const float* k_scale, const float* v_scale,
                         const int32_t* block_tables, int32_t max_blocks,
                         const int32_t* context_lens, int32_t B, int32_t H, int32_t Hkv,
                         int32_t d, int32_t block_size, int64_t num_blocks, double scale,
                         double* out) {
    return orc_decode_q8(q, q_dtype, 0, k_codes, v_codes, k_scale, v_scale, block_tables,
                         max_blocks, context_lens, B, H, Hkv, d, block_size, num_blocks, scale, out);
}

int pa_oracle_decode_int8(const uint16_t* q, int32_t q_dtype, const uint8_t* k_codes,
                          const uint8_t* v_codes, const float* k_scale, const float* v_scale,
                          const int32_t* block_tables, int32_t max_blocks,
                          const int32_t* context_lens, int32_t B, int32_t H, int32_t Hkv,
                          int32_t d, int32_t block_size, int64_t num_blocks, double scale,
                          double* out) {
    return orc_decode_q8(q, q_dtype, 1, k_codes, v_codes, k_scale, v_scale, block_tables,
                         max_blocks, context_lens, B, H, Hkv, d, block_size, num_blocks, scale, out);
}

/*
 * Multi-token query over the paged cache (chunked prefill / speculative
 * verification; "vLLM 深度拆解：当大模型推理学会「分页注意力」", section 5: a long
 * prompt's prefill split into chunks, and a draft's N tokens verified by one
 * forward pass).  Reading: sequence i's queries are its LAST qlen_i cached
 * tokens, rows q_start[i] .. q_start[i+1]-1 of q; query r (0-based) attends to
 * the cached tokens 0 .. n_i - qlen_i + r (causal), n_i = context_lens[i].
 * Each output row is the decode's attention over that prefix.
 *
 * q       [T, H, d], T = q_start[B]      out  [T, H, d] double
 * Rows are split over threads (each row computed by one thread).
 */
typedef struct {
    orc_job base;
    const int32_t* q_start;
    int32_t t_begin, t_end;
} orc_mq_job;

static void* orc_mq_worker(void* arg) {
    orc_mq_job* M = (orc_mq_job*)arg;
    const orc_job* J = &M->base;
    int32_t nmax = 1;
    for (int32_t i = 0; i < J->B; ++i)
        if (J->lens[i] > nmax) nmax = J->lens[i];
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    if (!s) {
        M->base.status = ORC_ERR_ARG;
        return NULL;
    }
    M->base.status = ORC_OK;
    const int32_t G = J->H / J->Hkv;
    int32_t i = 0;
    for (int32_t t = M->t_begin; t < M->t_end && M->base.status == ORC_OK; ++t) {
        while (M->q_start[i + 1] <= t) ++i;
        const int32_t qlen = M->q_start[i + 1] - M->q_start[i];
        const int32_t r = t - M->q_start[i];
        const int32_t n = J->lens[i] - qlen + r + 1;
        for (int32_t h = 0; h < J->H && M->base.status == ORC_OK; ++h) {
            const int64_t off = ((int64_t)t * J->H + h) * J->d;
            M->base.status = orc_attend(J, i, h / G, off, n, J->out + off, s);
        }
    }
    free(s);
    return NULL;
}

int pa_oracle_multi_query(const uint16_t* q, const int32_t* q_start, const uint16_t* k_cache,
                          const uint16_t* v_cache, const int32_t* block_tables,
                          int32_t max_blocks, const int32_t* context_lens, int32_t B, int32_t H,
                          int32_t Hkv, int32_t d, int32_t block_size, int64_t num_blocks,
                          double scale, int32_t dtype, double* out, int32_t num_threads) {
    if (B < 0 || H <= 0 || Hkv <= 0 || H % Hkv != 0 || d <= 0 || block_size <= 0 ||
        max_blocks < 0 || num_blocks < 0 || (dtype != 0 && dtype != 1) || !q_start)
        return ORC_ERR_ARG;
    if (q_start[0] != 0) return ORC_ERR_ARG;
    for (int32_t i = 0; i < B; ++i) {
        const int32_t qlen = q_start[i + 1] - q_start[i];
        if (qlen < 0 || qlen > context_lens[i]) return ORC_ERR_ARG;
    }
    const int32_t T = q_start[B];
    if (T == 0) return ORC_OK;
    if (num_threads < 1) num_threads = 1;
    if (num_threads > T) num_threads = T;
    orc_mq_job* jobs = (orc_mq_job*)calloc((size_t)num_threads, sizeof(orc_mq_job));
    pthread_t* th = (pthread_t*)calloc((size_t)num_threads, sizeof(pthread_t));
    if (!jobs || !th) {
        free(jobs);
        free(th);
        return ORC_ERR_ARG;
    }
    for (int t = 0; t < num_threads; ++t) {
        orc_mq_job* M = &jobs[t];
        M->base.q = q;
        M->base.k = k_cache;
        M->base.v = v_cache;
        M->base.tbl = block_tables;
        M->base.lens = context_lens;
        M->base.max_blocks = max_blocks;
        M->base.B = B;
        M->base.H = H;
        M->base.Hkv = Hkv;
        M->base.d = d;
        M->base.bs = block_size;
        M->base.dtype = dtype;
        M->base.num_blocks = num_blocks;
        M->base.scale = scale;
        M->base.out = out;
        M->q_start = q_start;
        M->t_begin = (int32_t)((int64_t)T * t / num_threads);
        M->t_end = (int32_t)((int64_t)T * (t + 1) / num_threads);
    }
    if (num_threads == 1) {
        orc_mq_worker(&jobs[0]);
    } else {
        for (int t = 0; t < num_threads; ++t) pthread_create(&th[t], NULL, orc_mq_worker, &jobs[t]);
        for (int t = 0; t < num_threads; ++t) pthread_join(th[t], NULL);
    }
    int status = ORC_OK;
    for (int t = 0; t < num_threads; ++t)
        if (jobs[t].base.status != ORC_OK) status = jobs[t].base.status;
    free(jobs);
    free(th);
    return status;
}
