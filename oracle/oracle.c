/*
 * Oracle for the paged-KV decode step: plain, slow, fp64 C on the CPU.
 *
 * TEST INFRASTRUCTURE ONLY. Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file. The product library never
 * links, includes or calls it, and it shares no code, header, table or helper
 * with the CUDA path.
 *
 * What it computes, and where the pages define it:
 *  - bf16 <-> double conversion from the IEEE-754 binary16-brain definition
 *    (1 sign, 8 exponent, 7 stored mantissa bits; round to nearest, ties to
 *    even; overflow to infinity).
 *  - RoPE table and rotation: "Rotary Position Embedding (RoPE) construction
 *    and application" in the NJU course brief "端侧大模型推理框架", §2.1
 *    (components to implement). Pairing (i, i+d/2), angle p * theta^(-2i/d).
 *  - Append (write_decode_kv): mini-infer README, "decode_batch 关键步骤",
 *    step 4: the new token's K/V are written back into the block tensor.
 *  - Slot of a token from the block table: mini-infer README, "项目概述"
 *    (Paged KV Cache = BlockTable + free-block pool), and the nxmr.cn article,
 *    §2.1 "KV缓存的内存革命" (logical pages mapped to physical pages).
 *  - Decode attention with GQA: NJU course brief §2.1, "QKV projection and
 *    Grouped-Query Attention" (query head j reads KV head j / G, the
 *    repeat_interleave convention), computed as the plain definition
 *    softmax(scale * q K^T) V over the request's paged history, in double.
 *  - Brute-force contiguous attention: the preallocated contiguous per-layer
 *    KV of the lnwmold.com InferLLM article, §3.4 "KV Cache的优化实现"; used to
 *    pin the paged walk.
 *
 * Every parity function here is pinned by the tests in tests/test_oracle_*.py
 * against closed forms, brute force and invariants that do not reuse this code.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_BLOCK 16

/* ---------------------------------------------------------------- bf16 ---- */

/* bf16 bits -> double. Exact: every bf16 value is a double. */
double or_double_from_bf16(uint16_t h) {
    uint32_t u = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16 bits, one rounding, to nearest with ties to even.
 * The quantum is 2^(E-7) for a value in [2^E, 2^(E+1)), E clamped below at
 * -126 (the subnormal range has the fixed quantum 2^-133). The value is scaled
 * so the quantum becomes 1, rounded to an integer in the default rounding mode
 * (nearest-even), and scaled back; the result is a bf16 value, so converting it
 * to float is exact and its top 16 bits are the answer. NaN gives the quiet NaN
 * 0x7FC0 with the input's sign; values at or beyond 2^128 after rounding give
 * infinity. */
uint16_t or_bf16_from_double(double x) {
    if (isnan(x)) return (uint16_t)(signbit(x) ? 0xFFC0u : 0x7FC0u);
    const uint16_t sgn = (uint16_t)(signbit(x) ? 0x8000u : 0u);
    const double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sgn | 0x7F80u);
    if (a == 0.0) return sgn;
    int e2;
    (void)frexp(a, &e2); /* a = f * 2^e2 with f in [0.5, 1) */
    int E = e2 - 1;      /* a in [2^E, 2^(E+1)) */
    if (E < -126) E = -126;
    const double n = nearbyint(ldexp(a, 7 - E));
    const double r = ldexp(n, E - 7);
    if (r >= 0x1p128) return (uint16_t)(sgn | 0x7F80u);
    const float f = (float)r; /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(sgn | (uint16_t)(u >> 16));
}

void or_bf16_from_double_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_bf16_from_double(x[i]);
}

void or_double_from_bf16_array(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_double_from_bf16(h[i]);
}

/* ---------------------------------------------------------------- RoPE ---- */

/* cos/sin table, layout [max_pos][d/2][2] fp32: entry (p, i) holds
 * cos(p * theta^(-2i/d)) and sin(...) evaluated in double and rounded once to
 * fp32. */
void or_rope_table(double theta, int32_t d, int32_t max_pos, float* out) {
    const int32_t half = d / 2;
    for (int32_t p = 0; p < max_pos; ++p) {
        for (int32_t i = 0; i < half; ++i) {
            const double inv_freq = 1.0 / pow(theta, (2.0 * (double)i) / (double)d);
            const double ang = (double)p * inv_freq;
            out[((int64_t)p * half + i) * 2 + 0] = (float)cos(ang);
            out[((int64_t)p * half + i) * 2 + 1] = (float)sin(ang);
        }
    }
}

/* Rotate one head vector x[d] (bf16 bits) with the table row cs[d/2][2]:
 *   y[i]       = x[i]       * cos_i - x[i+d/2] * sin_i
 *   y[i + d/2] = x[i + d/2] * cos_i + x[i]     * sin_i
 * in double (each product of a bf16 and an fp32 value is exact in double, so
 * the only rounding before the final one is the add), then one rounding to
 * bf16. */
static void rope_rotate_vec(const uint16_t* x, int32_t d, const float* cs, uint16_t* y) {
    const int32_t half = d / 2;
    for (int32_t i = 0; i < half; ++i) {
        const double x1 = or_double_from_bf16(x[i]);
        const double x2 = or_double_from_bf16(x[i + half]);
        const double c = (double)cs[2 * i + 0];
        const double s = (double)cs[2 * i + 1];
        const double p1 = x1 * c;
        const double p2 = x2 * s;
        const double p3 = x2 * c;
        const double p4 = x1 * s;
        y[i] = or_bf16_from_double(p1 - p2);
        y[i + half] = or_bf16_from_double(p3 + p4);
    }
}

/* Rotate n_vec head vectors of length d, all at position pos. */
void or_rope_rotate(const uint16_t* x, int32_t n_vec, int32_t d, const float* table,
                    int32_t pos, uint16_t* y) {
    const float* cs = table + (int64_t)pos * (d / 2) * 2;
    for (int32_t v = 0; v < n_vec; ++v) rope_rotate_vec(x + (int64_t)v * d, d, cs, y + (int64_t)v * d);
}

/* ------------------------------------------------------ slots and append ---- */

/* Slot of token `pos` of request b through its block table row:
 *   slot = table[b][pos / 16] * 16 + pos % 16.
 * Returns 0, or -1 when pos is outside the table row or the block id is < 0. */
int32_t or_slot_mapping(int32_t B, const int32_t* block_tables, int32_t max_blocks_per_seq,
                        const int32_t* pos, int32_t* slot_out) {
    int32_t bad = 0;
    for (int32_t b = 0; b < B; ++b) {
        const int32_t p = pos[b];
        if (p < 0 || p / OR_BLOCK >= max_blocks_per_seq) { slot_out[b] = -1; bad = -1; continue; }
        const int32_t blk = block_tables[(int64_t)b * max_blocks_per_seq + p / OR_BLOCK];
        if (blk < 0) { slot_out[b] = -1; bad = -1; continue; }
        slot_out[b] = blk * OR_BLOCK + p % OR_BLOCK;
    }
    return bad;
}

/* Append one new token per request:
 *   q_out[b][j]   = RoPE(q[b][j], positions[b])            for every query head j
 *   k_cache[slot] = RoPE(k[b][h], positions[b])            for every KV head h
 *   v_cache[slot] = v[b][h]                                (not rotated)
 * with the cache layout [num_blocks][Hkv][16][d], slot = slot_mapping[b]
 * (block slot/16, offset slot%16). No other byte of the caches changes.
 * Returns 0, or -1 if some slot or position is out of range (that request's
 * cache write is skipped, its q_out row is still written when the position is
 * valid). */
int32_t or_append(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_blocks,
                  const uint16_t* q, const uint16_t* k, const uint16_t* v,
                  const int32_t* positions, const int32_t* slot_mapping,
                  const float* table, int32_t max_pos,
                  uint16_t* q_out, uint16_t* k_cache, uint16_t* v_cache) {
    int32_t status = 0;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t p = positions[b];
        if (p < 0 || p >= max_pos) { status = -1; continue; }
        or_rope_rotate(q + (int64_t)b * Hq * d, Hq, d, table, p, q_out + (int64_t)b * Hq * d);
        const int32_t slot = slot_mapping[b];
        if (slot < 0 || slot / OR_BLOCK >= num_blocks) { status = -1; continue; }
        const int64_t blk = slot / OR_BLOCK, off = slot % OR_BLOCK;
        for (int32_t h = 0; h < Hkv; ++h) {
            const int64_t dst = ((blk * Hkv + h) * OR_BLOCK + off) * d;
            or_rope_rotate(k + ((int64_t)b * Hkv + h) * d, 1, d, table, p, tmp);
            memcpy(k_cache + dst, tmp, sizeof(uint16_t) * (size_t)d);
            memcpy(v_cache + dst, v + ((int64_t)b * Hkv + h) * d, sizeof(uint16_t) * (size_t)d);
        }
    }
    free(tmp);
    return status;
}

/* ------------------------------------------------------------ attention ---- */

typedef struct {
    int32_t B, Hq, Hkv, d, max_blocks_per_seq;
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    double scale;
    double* out;
    int64_t row_begin, row_end; /* rows are (b, j) pairs, b-major */
} or_attn_job;

/* One output row: request b, query head j, KV head h = j / G. Walks the block
 * table token by token: K_t and V_t live in block table[b][t/16] at offset
 * t%16. s_t = scale * <q, K_t>; out = sum_t exp(s_t - max s) V_t / sum_t
 * exp(s_t - max s). Context length <= 0 gives a zero row. */
static void attn_row(const or_attn_job* a, int32_t b, int32_t j, double* s) {
    const int32_t d = a->d, G = a->Hq / a->Hkv, h = j / G;
    double* o = a->out + ((int64_t)b * a->Hq + j) * d;
    for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
    const int32_t n = a->context_lens[b];
    if (n <= 0) return;
    const uint16_t* qr = a->q + ((int64_t)b * a->Hq + j) * d;
    double m = -INFINITY;
    for (int32_t t = 0; t < n; ++t) {
        const int64_t blk = a->block_tables[(int64_t)b * a->max_blocks_per_seq + t / OR_BLOCK];
        const uint16_t* kt = a->k_cache + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        double acc = 0.0;
        for (int32_t i = 0; i < d; ++i) acc += or_double_from_bf16(qr[i]) * or_double_from_bf16(kt[i]);
        s[t] = a->scale * acc;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int32_t t = 0; t < n; ++t) {
        const double w = exp(s[t] - m);
        l += w;
        const int64_t blk = a->block_tables[(int64_t)b * a->max_blocks_per_seq + t / OR_BLOCK];
        const uint16_t* vt = a->v_cache + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        for (int32_t i = 0; i < d; ++i) o[i] += w * or_double_from_bf16(vt[i]);
    }
    for (int32_t i = 0; i < d; ++i) o[i] /= l;
}

static void* attn_worker(void* arg) {
    const or_attn_job* a = (const or_attn_job*)arg;
    int32_t nmax = 1;
    for (int32_t b = 0; b < a->B; ++b)
        if (a->context_lens[b] > nmax) nmax = a->context_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    for (int64_t r = a->row_begin; r < a->row_end; ++r)
        attn_row(a, (int32_t)(r / a->Hq), (int32_t)(r % a->Hq), s);
    free(s);
    return NULL;
}

/* Paged decode attention over rows (b, j) for b < B, j < Hq; out is double
 * [B][Hq][d]. Rows are independent; nthreads > 1 splits them into contiguous
 * ranges run on POSIX threads, which leaves every row's arithmetic unchanged.
 * Returns the number of threads used. */
int32_t or_paged_attention(int32_t B, int32_t Hq, int32_t Hkv, int32_t d,
                           const uint16_t* q, const uint16_t* k_cache, const uint16_t* v_cache,
                           const int32_t* block_tables, int32_t max_blocks_per_seq,
                           const int32_t* context_lens, double scale, double* out,
                           int32_t nthreads) {
    const int64_t rows = (int64_t)B * Hq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int32_t)(rows > 0 ? rows : 1);
    or_attn_job* jobs = (or_attn_job*)malloc(sizeof(or_attn_job) * (size_t)nthreads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int32_t t = 0; t < nthreads; ++t) {
        or_attn_job* a = &jobs[t];
        a->B = B; a->Hq = Hq; a->Hkv = Hkv; a->d = d; a->max_blocks_per_seq = max_blocks_per_seq;
        a->q = q; a->k_cache = k_cache; a->v_cache = v_cache;
        a->block_tables = block_tables; a->context_lens = context_lens;
        a->scale = scale; a->out = out;
        a->row_begin = rows * t / nthreads;
        a->row_end = rows * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        attn_worker(&jobs[0]);
    } else {
        for (int32_t t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, attn_worker, &jobs[t]);
        for (int32_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    free(th);
    free(jobs);
    return nthreads;
}

/* Brute force over a contiguous cache: K and V are [B][Hkv][n_max][d] with
 * request b's tokens at positions 0..lens[b]-1 (the non-paged layout). Builds
 * the score vector, subtracts its max, exponentiates, normalises the weights
 * first and then sums weight * V. Used only to pin or_paged_attention. */
void or_contiguous_attention(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t n_max,
                             const uint16_t* q, const uint16_t* K, const uint16_t* V,
                             const int32_t* lens, double scale, double* out) {
    const int32_t G = Hq / Hkv;
    double* w = (double*)malloc(sizeof(double) * (size_t)(n_max > 0 ? n_max : 1));
    for (int32_t b = 0; b < B; ++b) {
        for (int32_t j = 0; j < Hq; ++j) {
            double* o = out + ((int64_t)b * Hq + j) * d;
            memset(o, 0, sizeof(double) * (size_t)d);
            const int32_t n = lens[b];
            if (n <= 0) continue;
            const int32_t h = j / G;
            const uint16_t* qr = q + ((int64_t)b * Hq + j) * d;
            const uint16_t* Kb = K + ((int64_t)b * Hkv + h) * n_max * d;
            const uint16_t* Vb = V + ((int64_t)b * Hkv + h) * n_max * d;
            double mx = -INFINITY;
            for (int32_t t = 0; t < n; ++t) {
                double acc = 0.0;
                for (int32_t i = 0; i < d; ++i)
                    acc += or_double_from_bf16(qr[i]) * or_double_from_bf16(Kb[(int64_t)t * d + i]);
                w[t] = acc * scale;
                mx = w[t] > mx ? w[t] : mx;
            }
            double z = 0.0;
            for (int32_t t = 0; t < n; ++t) { w[t] = exp(w[t] - mx); z += w[t]; }
            for (int32_t t = 0; t < n; ++t) w[t] /= z;
            for (int32_t i = 0; i < d; ++i) {
                double acc = 0.0;
                for (int32_t t = 0; t < n; ++t) acc += w[t] * or_double_from_bf16(Vb[(int64_t)t * d + i]);
                o[i] = acc;
            }
        }
    }
    free(w);
}

/* ------------------------------------------------------ prefill attention -- */

typedef struct {
    int32_t R, Hq, Hkv, d, max_blocks_per_seq;
    const uint16_t* q;
    const uint16_t* k_cache;
    const uint16_t* v_cache;
    const int32_t* block_tables;
    const int32_t* context_lens;
    const int32_t* query_start;
    double scale;
    double* out;
    int64_t row_begin, row_end; /* rows are (query token, head) pairs */
} or_prefill_job;

/* Query token qi (a row of q) of request r is the token at position
 * p = n_r - m_r + i (its i-th new token, n_r = context_lens[r] counting the new
 * tokens, m_r = query_start[r+1] - query_start[r]); it attends causally to the
 * cached tokens t <= p (prefill / chunked prefill of the course brief's
 * prefill + decode loop, §2.1, over mini-infer's paged cache, "项目概述"). */
static void prefill_row(const or_prefill_job* a, int32_t qi, int32_t j, double* s) {
    const int32_t d = a->d, G = a->Hq / a->Hkv, h = j / G;
    double* o = a->out + ((int64_t)qi * a->Hq + j) * d;
    for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
    int32_t r = 0;
    while (r < a->R && a->query_start[r + 1] <= qi) ++r;
    if (r >= a->R) return;
    const int32_t m = a->query_start[r + 1] - a->query_start[r];
    const int32_t n = a->context_lens[r];
    const int32_t pos = n - m + (qi - a->query_start[r]);
    if (pos < 0) return;
    const uint16_t* qr = a->q + ((int64_t)qi * a->Hq + j) * d;
    double mx = -INFINITY;
    for (int32_t t = 0; t <= pos; ++t) {
        const int64_t blk = a->block_tables[(int64_t)r * a->max_blocks_per_seq + t / OR_BLOCK];
        const uint16_t* kt = a->k_cache + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        double acc = 0.0;
        for (int32_t i = 0; i < d; ++i) acc += or_double_from_bf16(qr[i]) * or_double_from_bf16(kt[i]);
        s[t] = a->scale * acc;
        if (s[t] > mx) mx = s[t];
    }
    double l = 0.0;
    for (int32_t t = 0; t <= pos; ++t) {
        const double w = exp(s[t] - mx);
        l += w;
        const int64_t blk = a->block_tables[(int64_t)r * a->max_blocks_per_seq + t / OR_BLOCK];
        const uint16_t* vt = a->v_cache + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        for (int32_t i = 0; i < d; ++i) o[i] += w * or_double_from_bf16(vt[i]);
    }
    for (int32_t i = 0; i < d; ++i) o[i] /= l;
}

static void* prefill_worker(void* arg) {
    const or_prefill_job* a = (const or_prefill_job*)arg;
    int32_t nmax = 1;
    for (int32_t r = 0; r < a->R; ++r)
        if (a->context_lens[r] > nmax) nmax = a->context_lens[r];
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    for (int64_t row = a->row_begin; row < a->row_end; ++row)
        prefill_row(a, (int32_t)(row / a->Hq), (int32_t)(row % a->Hq), s);
    free(s);
    return NULL;
}

/* Causal paged attention for T = query_start[R] new tokens; out is double
 * [T][Hq][d]. Rows are independent; nthreads > 1 runs contiguous row ranges on
 * POSIX threads without changing any row's arithmetic. Returns threads used. */
int32_t or_paged_prefill_attention(int32_t R, int32_t Hq, int32_t Hkv, int32_t d, const uint16_t* q,
                                   const uint16_t* k_cache, const uint16_t* v_cache,
                                   const int32_t* block_tables, int32_t max_blocks_per_seq,
                                   const int32_t* context_lens, const int32_t* query_start,
                                   double scale, double* out, int32_t nthreads) {
    const int64_t rows = (int64_t)query_start[R] * Hq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int32_t)(rows > 0 ? rows : 1);
    or_prefill_job* jobs = (or_prefill_job*)malloc(sizeof(or_prefill_job) * (size_t)nthreads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int32_t t = 0; t < nthreads; ++t) {
        or_prefill_job* a = &jobs[t];
        a->R = R; a->Hq = Hq; a->Hkv = Hkv; a->d = d; a->max_blocks_per_seq = max_blocks_per_seq;
        a->q = q; a->k_cache = k_cache; a->v_cache = v_cache;
        a->block_tables = block_tables; a->context_lens = context_lens; a->query_start = query_start;
        a->scale = scale; a->out = out;
        a->row_begin = rows * t / nthreads;
        a->row_end = rows * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        prefill_worker(&jobs[0]);
    } else {
        for (int32_t t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, prefill_worker, &jobs[t]);
        for (int32_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    free(th);
    free(jobs);
    return nthreads;
}

/* ------------------------------------------------------------- FP8 KV ---- */
/* FP8 KV cache (GitLink project report "mxdyymxgxtlkjdxtjyhysx", section
 * "技术探索：FP8 KV Cache量化效果分析": the KV cache stored as FP8 to cut the
 * bytes moved). The pages name no format or scaling; the reading taken here:
 * the e4m3 format (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
 * exponent field 0 holds subnormals m/8 * 2^-6; the all-ones code S.1111.111
 * is NaN; no infinities; largest finite 448) with one fp32 scale per KV head,
 * symmetric (no zero point, as the nxmr.cn article's §2.2 "量化压缩的实战选择"
 * advises for 8-bit KV): stored code = e4m3(x / scale[h]), value = code value *
 * scale[h]. */

/* e4m3 code -> double, from the format definition. */
double or_double_from_e4m3(uint8_t c) {
    const int s = c >> 7, e = (c >> 3) & 15, m = c & 7;
    double v;
    if (e == 15 && m == 7) return s ? -NAN : NAN;
    if (e == 0)
        v = ldexp((double)m, -9);              /* m/8 * 2^-6 */
    else
        v = ldexp(8.0 + (double)m, e - 10);    /* (1 + m/8) * 2^(e-7) */
    return s ? -v : v;
}

/* double -> e4m3 code, rounding to nearest with ties to even and saturating
 * to +-448 (no code means infinity). The quantum is 2^(E-3) for |x| in
 * [2^E, 2^(E+1)), E clamped below at -6 (the subnormal range has quantum
 * 2^-9); |x| is scaled so the quantum is 1, rounded to an integer in the
 * default rounding mode (nearest-even) and scaled back, then encoded. */
uint8_t or_e4m3_from_double(double x) {
    const uint8_t sgn = signbit(x) ? 0x80 : 0x00;
    if (isnan(x)) return (uint8_t)(sgn | 0x7F);
    double a = fabs(x);
    if (a >= 448.0) return (uint8_t)(sgn | 0x7E);          /* 1.75 * 2^8 */
    if (a == 0.0) return sgn;
    int E;
    (void)frexp(a, &E);                                    /* a = f * 2^E, f in [0.5, 1) */
    E -= 1;                                                /* a in [2^E, 2^(E+1)) */
    if (E < -6) E = -6;
    const double q = nearbyint(ldexp(a, 3 - E));           /* a / 2^(E-3), rounded */
    const double r = ldexp(q, E - 3);                      /* the rounded magnitude */
    if (r >= 448.0) return (uint8_t)(sgn | 0x7E);
    if (r < ldexp(1.0, -6)) return (uint8_t)(sgn | (uint8_t)ldexp(r, 9));   /* subnormal */
    int Er;
    const double fr = frexp(r, &Er);                       /* r = fr * 2^Er */
    const int e = Er - 1 + 7;                              /* biased exponent */
    const int m = (int)(ldexp(fr, 4)) - 8;                 /* fr * 16 = 8 + m */
    return (uint8_t)(sgn | (uint8_t)(e << 3) | (uint8_t)m);
}

void or_e4m3_from_double_array(const double* x, int64_t n, uint8_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_e4m3_from_double(x[i]);
}

void or_double_from_e4m3_array(const uint8_t* c, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = or_double_from_e4m3(c[i]);
}

/* Append into FP8 caches: as or_append, but the cache rows hold
 *   k8 = e4m3(fp32(bf16(RoPE(k)) / k_scale[h])),  v8 = e4m3(fp32(v / v_scale[h]))
 * (the bf16 value the bf16 cache would hold, divided by the head's fp32 scale
 * in IEEE single precision, then rounded to e4m3). q_out is the bf16
 * RoPE(q). */
int32_t or_append_fp8(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_blocks,
                      const uint16_t* q, const uint16_t* k, const uint16_t* v,
                      const int32_t* positions, const int32_t* slot_mapping,
                      const float* table, int32_t max_pos, const float* k_scale, const float* v_scale,
                      uint16_t* q_out, uint8_t* k_cache, uint8_t* v_cache) {
    int32_t status = 0;
    uint16_t* tmp = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)d);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t p = positions[b];
        if (p < 0 || p >= max_pos) { status = -1; continue; }
        or_rope_rotate(q + (int64_t)b * Hq * d, Hq, d, table, p, q_out + (int64_t)b * Hq * d);
        const int32_t slot = slot_mapping[b];
        if (slot < 0 || slot / OR_BLOCK >= num_blocks) { status = -1; continue; }
        const int64_t blk = slot / OR_BLOCK, off = slot % OR_BLOCK;
        for (int32_t h = 0; h < Hkv; ++h) {
            const int64_t dst = ((blk * Hkv + h) * OR_BLOCK + off) * d;
            or_rope_rotate(k + ((int64_t)b * Hkv + h) * d, 1, d, table, p, tmp);
            const uint16_t* vr = v + ((int64_t)b * Hkv + h) * d;
            for (int32_t i = 0; i < d; ++i) {
                const float yk = (float)or_double_from_bf16(tmp[i]) / k_scale[h];
                const float yv = (float)or_double_from_bf16(vr[i]) / v_scale[h];
                k_cache[dst + i] = or_e4m3_from_double((double)yk);
                v_cache[dst + i] = or_e4m3_from_double((double)yv);
            }
        }
    }
    free(tmp);
    return status;
}

typedef struct {
    int32_t B, Hq, Hkv, d, max_blocks_per_seq;
    const uint16_t* q;
    const uint8_t* k_cache;
    const uint8_t* v_cache;
    const float* k_scale;
    const float* v_scale;
    const int32_t* block_tables;
    const int32_t* context_lens;
    double scale;
    double* out;
    int64_t row_begin, row_end;
} or_attn8_job;

/* Decode attention over FP8 caches: the definition of attn_row with
 * K_t = value(k8) * k_scale[h] and V_t = value(v8) * v_scale[h], in double. */
static void attn8_row(const or_attn8_job* a, int32_t b, int32_t j, double* s) {
    const int32_t d = a->d, G = a->Hq / a->Hkv, h = j / G;
    double* o = a->out + ((int64_t)b * a->Hq + j) * d;
    for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
    const int32_t n = a->context_lens[b];
    if (n <= 0) return;
    const uint16_t* qr = a->q + ((int64_t)b * a->Hq + j) * d;
    const double ks = (double)a->k_scale[h], vs = (double)a->v_scale[h];
    double m = -INFINITY;
    for (int32_t t = 0; t < n; ++t) {
        const int64_t blk = a->block_tables[(int64_t)b * a->max_blocks_per_seq + t / OR_BLOCK];
        const uint8_t* kt = a->k_cache + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        double acc = 0.0;
        for (int32_t i = 0; i < d; ++i) acc += or_double_from_bf16(qr[i]) * (or_double_from_e4m3(kt[i]) * ks);
        s[t] = a->scale * acc;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int32_t t = 0; t < n; ++t) {
        const double w = exp(s[t] - m);
        l += w;
        const int64_t blk = a->block_tables[(int64_t)b * a->max_blocks_per_seq + t / OR_BLOCK];
        const uint8_t* vt = a->v_cache + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        for (int32_t i = 0; i < d; ++i) o[i] += w * (or_double_from_e4m3(vt[i]) * vs);
    }
    for (int32_t i = 0; i < d; ++i) o[i] /= l;
}

static void* attn8_worker(void* arg) {
    const or_attn8_job* a = (const or_attn8_job*)arg;
    int32_t nmax = 1;
    for (int32_t b = 0; b < a->B; ++b)
        if (a->context_lens[b] > nmax) nmax = a->context_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    for (int64_t r = a->row_begin; r < a->row_end; ++r)
        attn8_row(a, (int32_t)(r / a->Hq), (int32_t)(r % a->Hq), s);
    free(s);
    return NULL;
}

/* FP8 paged decode attention, rows (b, j) on nthreads POSIX threads as in
 * or_paged_attention. Returns the number of threads used. */
int32_t or_paged_attention_fp8(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, const uint16_t* q,
                               const uint8_t* k_cache, const uint8_t* v_cache, const float* k_scale,
                               const float* v_scale, const int32_t* block_tables,
                               int32_t max_blocks_per_seq, const int32_t* context_lens, double scale,
                               double* out, int32_t nthreads) {
    const int64_t rows = (int64_t)B * Hq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int32_t)(rows > 0 ? rows : 1);
    or_attn8_job* jobs = (or_attn8_job*)malloc(sizeof(or_attn8_job) * (size_t)nthreads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int32_t t = 0; t < nthreads; ++t) {
        or_attn8_job* a = &jobs[t];
        a->B = B; a->Hq = Hq; a->Hkv = Hkv; a->d = d; a->max_blocks_per_seq = max_blocks_per_seq;
        a->q = q; a->k_cache = k_cache; a->v_cache = v_cache; a->k_scale = k_scale; a->v_scale = v_scale;
        a->block_tables = block_tables; a->context_lens = context_lens;
        a->scale = scale; a->out = out;
        a->row_begin = rows * t / nthreads;
        a->row_end = rows * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        attn8_worker(&jobs[0]);
    } else {
        for (int32_t t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, attn8_worker, &jobs[t]);
        for (int32_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    free(th);
    free(jobs);
    return nthreads;
}

/* ------------------------------------------------------------ INT8 KV ---- */
/* INT8 KV cache (nxmr.cn article, §2.2 "量化压缩的实战选择": the KV cache held
 * in 8 bits, quantised in groups of 64 tokens rather than per token,
 * symmetric (no zero point) with scale = 127 / max|x|, the scaled values
 * clamped to [-128, 127] and converted to int8; per head where heads' ranges
 * differ). Readings taken here:
 *  - a group is 64 consecutive tokens (64g .. 64g+63) of one request and one
 *    KV head, over all d dims; K and V are quantised separately;
 *  - x is the bf16 value the bf16 cache would hold (after RoPE for K);
 *  - m = max |x| over the group's tokens; s = 127 / m divided in IEEE single
 *    precision; y = x * s multiplied in single precision; y clamped to
 *    [-128, 127] and converted to int8 toward zero (the article's tensor
 *    cast); m = 0 gives code 0 for every value;
 *  - a code stands for the value code * m / 127;
 *  - a request's last group may hold fewer than 64 tokens; it is quantised
 *    over the tokens it holds, and again over all of them, from their
 *    original values, whenever a token joins it (so a full group ends up
 *    quantised over its 64 tokens, the article's definition).
 * Storage: codes in int8 caches [num_blocks][Hkv][16][d]; m (a bf16 value
 * held as fp32) at amax[blk][h] for every block blk the group's tokens lie
 * in; the original bf16 rows of each request's last group in an open-group
 * buffer [slots][Hkv][64][d] at the request's slot. Inputs are finite. */

#define OR_GROUP 64

/* Codes of one group of `count` bf16 values; returns m. */
float or_int8_quantize(const uint16_t* x, int64_t count, int8_t* codes) {
    double m = 0.0;
    for (int64_t i = 0; i < count; ++i) {
        const double a = fabs(or_double_from_bf16(x[i]));
        if (a > m) m = a;
    }
    if (m == 0.0) {
        memset(codes, 0, (size_t)count);
        return 0.0f;
    }
    const float s = 127.0f / (float)m;  /* m is a bf16 value: exact in float */
    for (int64_t i = 0; i < count; ++i) {
        float y = (float)or_double_from_bf16(x[i]) * s;
        if (y > 127.0f) y = 127.0f;
        if (y < -128.0f) y = -128.0f;
        codes[i] = (int8_t)(int)y;      /* C's float -> int conversion truncates toward zero */
    }
    return (float)m;
}

/* The group holding tokens t0 .. t0+ntok-1 of one request and head h, from
 * its bf16 rows [ntok][d]: codes to the tokens' cache slots through the
 * request's block table row, m to amax of every block those tokens lie in.
 * Returns -1 (and writes nothing) if a block id is out of range. */
static int32_t int8_group(const uint16_t* rows, int32_t ntok, int32_t d, int32_t Hkv, int32_t h,
                          const int32_t* bt_row, int32_t t0, int32_t num_blocks, int8_t* cache, float* amax,
                          int8_t* tmp) {
    for (int32_t t = 0; t < ntok; ++t) {
        const int32_t blk = bt_row[(t0 + t) / OR_BLOCK];
        if (blk < 0 || blk >= num_blocks) return -1;
    }
    const float m = or_int8_quantize(rows, (int64_t)ntok * d, tmp);
    for (int32_t t = 0; t < ntok; ++t) {
        const int64_t blk = bt_row[(t0 + t) / OR_BLOCK], off = (t0 + t) % OR_BLOCK;
        memcpy(cache + ((blk * Hkv + h) * OR_BLOCK + off) * d, tmp + (int64_t)t * d, (size_t)d);
        amax[blk * Hkv + h] = m;
    }
    return 0;
}

/* INT8 caches of B requests whose first context_lens[b] tokens are held in
 * bf16 caches (layout [num_blocks][Hkv][16][d]) at the same slots: every
 * group quantised over the tokens it holds, and each request's last group
 * copied to its open-group slot. Returns 0, or -1 if a block id or a slot is
 * out of range (that request is skipped). */
int32_t or_int8_from_bf16_cache(int32_t B, int32_t Hkv, int32_t d, int32_t num_blocks,
                                const uint16_t* k_cache, const uint16_t* v_cache,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, const int32_t* open_slots, int32_t num_slots,
                                int8_t* k8, int8_t* v8, float* k_amax, float* v_amax,
                                uint16_t* k_open, uint16_t* v_open) {
    int32_t status = 0;
    uint16_t* rk = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)OR_GROUP * d);
    uint16_t* rv = (uint16_t*)malloc(sizeof(uint16_t) * (size_t)OR_GROUP * d);
    int8_t* tmp = (int8_t*)malloc((size_t)OR_GROUP * d);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t n = context_lens[b];
        if (n <= 0) continue;
        const int32_t slot = open_slots[b];
        const int32_t* bt = block_tables + (int64_t)b * max_blocks_per_seq;
        int bad = slot < 0 || slot >= num_slots;
        for (int32_t t = 0; t < n && !bad; t += OR_BLOCK) bad = bt[t / OR_BLOCK] < 0 || bt[t / OR_BLOCK] >= num_blocks;
        if (bad) { status = -1; continue; }
        for (int32_t h = 0; h < Hkv; ++h) {
            for (int32_t t0 = 0; t0 < n; t0 += OR_GROUP) {
                const int32_t ntok = n - t0 < OR_GROUP ? n - t0 : OR_GROUP;
                for (int32_t t = 0; t < ntok; ++t) {
                    const int64_t blk = bt[(t0 + t) / OR_BLOCK], off = (t0 + t) % OR_BLOCK;
                    const int64_t src = ((blk * Hkv + h) * OR_BLOCK + off) * d;
                    memcpy(rk + (int64_t)t * d, k_cache + src, sizeof(uint16_t) * (size_t)d);
                    memcpy(rv + (int64_t)t * d, v_cache + src, sizeof(uint16_t) * (size_t)d);
                }
                (void)int8_group(rk, ntok, d, Hkv, h, bt, t0, num_blocks, k8, k_amax, tmp);
                (void)int8_group(rv, ntok, d, Hkv, h, bt, t0, num_blocks, v8, v_amax, tmp);
                if (t0 + OR_GROUP >= n) {  /* the last group: its rows to the open-group slot */
                    const int64_t o = ((int64_t)slot * Hkv + h) * OR_GROUP * d;
                    memcpy(k_open + o, rk, sizeof(uint16_t) * (size_t)ntok * d);
                    memcpy(v_open + o, rv, sizeof(uint16_t) * (size_t)ntok * d);
                }
            }
        }
    }
    free(rk);
    free(rv);
    free(tmp);
    return status;
}

/* Append one new token per request into INT8 caches: n = context_lens[b]
 * (the length after the append; n <= 0 appends nothing), position p = n - 1,
 * group g = p / 64, offset o = p % 64.
 *   q_out[b][j] = RoPE(q[b][j], p);
 *   open[slot][h][o] = RoPE(k[b][h], p) for K, v[b][h] for V;
 *   the group is quantised over open[slot][h][0 .. o] and its codes and m
 *   written to tokens 64g .. p through the block table.
 * Returns 0, or -1 if some position, slot or block id is out of range (that
 * request's cache writes are skipped; q_out is written when p is valid). */
int32_t or_append_int8(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, int32_t num_blocks,
                       const uint16_t* q, const uint16_t* k, const uint16_t* v,
                       const float* table, int32_t max_pos,
                       const int32_t* block_tables, int32_t max_blocks_per_seq, const int32_t* context_lens,
                       const int32_t* open_slots, int32_t num_slots,
                       uint16_t* q_out, int8_t* k8, int8_t* v8, float* k_amax, float* v_amax,
                       uint16_t* k_open, uint16_t* v_open) {
    int32_t status = 0;
    int8_t* tmp = (int8_t*)malloc((size_t)OR_GROUP * d);
    for (int32_t b = 0; b < B; ++b) {
        const int32_t n = context_lens[b];
        if (n <= 0) continue;
        const int32_t p = n - 1;
        if (p >= max_pos || n > max_blocks_per_seq * OR_BLOCK) { status = -1; continue; }
        or_rope_rotate(q + (int64_t)b * Hq * d, Hq, d, table, p, q_out + (int64_t)b * Hq * d);
        const int32_t slot = open_slots[b];
        if (slot < 0 || slot >= num_slots) { status = -1; continue; }
        const int32_t* bt = block_tables + (int64_t)b * max_blocks_per_seq;
        const int32_t t0 = p / OR_GROUP * OR_GROUP, o = p % OR_GROUP;
        int bad = 0;
        for (int32_t t = t0; t <= p; t += OR_BLOCK) bad |= bt[t / OR_BLOCK] < 0 || bt[t / OR_BLOCK] >= num_blocks;
        if (bad) { status = -1; continue; }
        for (int32_t h = 0; h < Hkv; ++h) {
            uint16_t* ko = k_open + ((int64_t)slot * Hkv + h) * OR_GROUP * d;
            uint16_t* vo = v_open + ((int64_t)slot * Hkv + h) * OR_GROUP * d;
            or_rope_rotate(k + ((int64_t)b * Hkv + h) * d, 1, d, table, p, ko + (int64_t)o * d);
            memcpy(vo + (int64_t)o * d, v + ((int64_t)b * Hkv + h) * d, sizeof(uint16_t) * (size_t)d);
            (void)int8_group(ko, o + 1, d, Hkv, h, bt, t0, num_blocks, k8, k_amax, tmp);
            (void)int8_group(vo, o + 1, d, Hkv, h, bt, t0, num_blocks, v8, v_amax, tmp);
        }
    }
    free(tmp);
    return status;
}

typedef struct {
    int32_t B, Hq, Hkv, d, max_blocks_per_seq;
    const uint16_t* q;
    const int8_t* k8;
    const int8_t* v8;
    const float* k_amax;
    const float* v_amax;
    const int32_t* block_tables;
    const int32_t* context_lens;
    double scale;
    double* out;
    int64_t row_begin, row_end;
} or_attn_i8_job;

/* Decode attention over INT8 caches: the definition of attn_row with
 * K_t = code * amax_k[blk][h] / 127 and V_t = code * amax_v[blk][h] / 127,
 * blk = table[b][t/16], in double. */
static void attn_i8_row(const or_attn_i8_job* a, int32_t b, int32_t j, double* s) {
    const int32_t d = a->d, G = a->Hq / a->Hkv, h = j / G;
    double* o = a->out + ((int64_t)b * a->Hq + j) * d;
    for (int32_t i = 0; i < d; ++i) o[i] = 0.0;
    const int32_t n = a->context_lens[b];
    if (n <= 0) return;
    const uint16_t* qr = a->q + ((int64_t)b * a->Hq + j) * d;
    double m = -INFINITY;
    for (int32_t t = 0; t < n; ++t) {
        const int64_t blk = a->block_tables[(int64_t)b * a->max_blocks_per_seq + t / OR_BLOCK];
        const int8_t* kt = a->k8 + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        const double am = (double)a->k_amax[blk * a->Hkv + h];
        double acc = 0.0;
        for (int32_t i = 0; i < d; ++i) acc += or_double_from_bf16(qr[i]) * ((double)kt[i] * am / 127.0);
        s[t] = a->scale * acc;
        if (s[t] > m) m = s[t];
    }
    double l = 0.0;
    for (int32_t t = 0; t < n; ++t) {
        const double w = exp(s[t] - m);
        l += w;
        const int64_t blk = a->block_tables[(int64_t)b * a->max_blocks_per_seq + t / OR_BLOCK];
        const int8_t* vt = a->v8 + ((blk * a->Hkv + h) * OR_BLOCK + t % OR_BLOCK) * d;
        const double am = (double)a->v_amax[blk * a->Hkv + h];
        for (int32_t i = 0; i < d; ++i) o[i] += w * ((double)vt[i] * am / 127.0);
    }
    for (int32_t i = 0; i < d; ++i) o[i] /= l;
}

static void* attn_i8_worker(void* arg) {
    const or_attn_i8_job* a = (const or_attn_i8_job*)arg;
    int32_t nmax = 1;
    for (int32_t b = 0; b < a->B; ++b)
        if (a->context_lens[b] > nmax) nmax = a->context_lens[b];
    double* s = (double*)malloc(sizeof(double) * (size_t)nmax);
    for (int64_t r = a->row_begin; r < a->row_end; ++r)
        attn_i8_row(a, (int32_t)(r / a->Hq), (int32_t)(r % a->Hq), s);
    free(s);
    return NULL;
}

/* INT8 paged decode attention, rows (b, j) on nthreads POSIX threads as in
 * or_paged_attention. Returns the number of threads used. */
int32_t or_paged_attention_int8(int32_t B, int32_t Hq, int32_t Hkv, int32_t d, const uint16_t* q,
                                const int8_t* k8, const int8_t* v8, const float* k_amax, const float* v_amax,
                                const int32_t* block_tables, int32_t max_blocks_per_seq,
                                const int32_t* context_lens, double scale, double* out, int32_t nthreads) {
    const int64_t rows = (int64_t)B * Hq;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > rows) nthreads = (int32_t)(rows > 0 ? rows : 1);
    or_attn_i8_job* jobs = (or_attn_i8_job*)malloc(sizeof(or_attn_i8_job) * (size_t)nthreads);
    pthread_t* th = (pthread_t*)malloc(sizeof(pthread_t) * (size_t)nthreads);
    for (int32_t t = 0; t < nthreads; ++t) {
        or_attn_i8_job* a = &jobs[t];
        a->B = B; a->Hq = Hq; a->Hkv = Hkv; a->d = d; a->max_blocks_per_seq = max_blocks_per_seq;
        a->q = q; a->k8 = k8; a->v8 = v8; a->k_amax = k_amax; a->v_amax = v_amax;
        a->block_tables = block_tables; a->context_lens = context_lens;
        a->scale = scale; a->out = out;
        a->row_begin = rows * t / nthreads;
        a->row_end = rows * (t + 1) / nthreads;
    }
    if (nthreads == 1) {
        attn_i8_worker(&jobs[0]);
    } else {
        for (int32_t t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, attn_i8_worker, &jobs[t]);
        for (int32_t t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
    }
    free(th);
    free(jobs);
    return nthreads;
}
