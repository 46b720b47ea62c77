/*
 * pa_oracle.c -- plain CPU oracle for attention over a block-paged KV cache.
 *
 * TEST INFRASTRUCTURE ONLY.  This file is the slow, obviously correct
 * definition that the CUDA library is checked against.  Only the tests, the
 * package smoke check and the benchmark's CPU-baseline leg may load it; the
 * product path never calls it and shares no code, header or constant with it.
 *
 * Sources (page title, section):
 *   [P1] "大模型推理入门与 nano-vLLM 源码详解" (duanmeng.github.io)
 *        §1.3 single-head attention, §4.4 KV bytes per position,
 *        §9.2 token position -> physical slot, §9.5 PagedAttention,
 *        §10.2 prefix hit (108 queries over 620 keys), §11.2 Prefill inputs,
 *        §11.4 Decode inputs, §13.1 KV write, §13.5 padded rows,
 *        §19.1 softmax, §19.6 GQA.
 *   [P2] "大模型推理引擎入门：从 Continuous Batching 到 Scheduler，对着日志读懂
 *        nano-vllm" (juejin.cn), §2.7.2-2.7.3 prepare_prefill / prepare_decode.
 *   [P3] "VLLM on Fain的Blog" (Pico-vLLM log), #6 paged decode kernel,
 *        #8 fused RoPE and paged KV store.
 *   [P4] "nano-vllm 技术分析" (deepseek.csdn.net), §4.3 RMSNorm, §4.4 RoPE,
 *        the prefill parameter computation (prepare_prefill).
 *   [P2] also §2.7.2-2.7.3 worked prepare_prefill / prepare_decode values.
 *   [P1] also §12.2 (head norm and RoPE before the KV write), §19.5 RMSNorm,
 *        §19.7 RoPE.
 *
 * What it computes is the plain definition of softmax attention, with K/V
 * rows fetched by walking block_table one key at a time.  There is no
 * blocking, no online softmax and no split: every query row gets all of its
 * scores, one max, one exponent sum and one weighted sum of V, in double
 * precision.  bf16 inputs are widened exactly; outputs are returned as double.
 *
 * Data layouts (all row-major):
 *   q          [T, Hq, d]   bf16 bits, token stride q_stride (elements)
 *   k, v       [T, Hkv, d]  bf16 bits, token stride kv_stride (elements)
 *   k_cache    [num_blocks, block_size, Hkv, d] bf16 bits (one layer)
 *   block_table[num_seqs, max_blocks] int32, -1 padded
 *   cu_seqlens [num_seqs + 1] int32 prefix sums
 *   out        [T, Hq, d]   double
 *
 * Status codes returned: 0 ok, 1 invalid argument, 4 an index out of range.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORC_OK 0
#define ORC_INVALID 1
#define ORC_BOUNDS 4

/* bf16 is the upper half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

void orc_set_num_threads(int n)
{
#ifdef _OPENMP
    if (n > 0) omp_set_num_threads(n);
#else
    (void)n;
#endif
}

/* [P1] §4.4: bytes = 2 (K and V) x layers x KV heads x head_dim x bytes per element. */
int64_t orc_kv_bytes_per_token(int layers, int kv_heads, int head_dim, int elem_bytes)
{
    return (int64_t)2 * layers * kv_heads * head_dim * elem_bytes;
}

/* [P1] §9.2: slot = block_table[pos // block_size] * block_size + pos % block_size.
 * A slot numbers a token row of the pool, not a byte address. */
int64_t orc_slot(const int32_t *block_table_row, int block_size, int64_t pos)
{
    return (int64_t)block_table_row[pos / block_size] * block_size + pos % block_size;
}

/* [P1] §13.1: every token with slot != -1 copies its Hkv*d values of K and of V
 * to row `slot` of the layer's cache; slot == -1 marks a padding row and is
 * skipped.  Any other slot outside [0, num_blocks*block_size) is reported. */
int orc_store_kvcache(const uint16_t *k, int64_t k_stride, const uint16_t *v, int64_t v_stride,
                      int64_t num_tokens, int kv_heads, int head_dim,
                      uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks, int block_size,
                      const int32_t *slot_mapping)
{
    const int64_t row = (int64_t)kv_heads * head_dim;
    const int64_t num_slots = num_blocks * block_size;
    int status = ORC_OK;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) { status = ORC_BOUNDS; continue; }
        for (int64_t e = 0; e < row; ++e) {
            k_cache[slot * row + e] = k[t * k_stride + e];
            v_cache[slot * row + e] = v[t * v_stride + e];
        }
    }
    return status;
}

/* Where the keys of one sequence live: either the paged pool reached through
 * one block_table row, or a contiguous run of the new-token k/v tensors. */
typedef struct {
    const uint16_t *k_cache, *v_cache;
    const int32_t *table_row; /* NULL: contiguous k/v */
    int64_t num_blocks;
    int block_size;
    int max_blocks;
    const uint16_t *k, *v; /* first row of the sequence in k / v */
    int64_t kv_stride;
    int kv_heads, head_dim;
    const uint8_t *k8_cache, *v8_cache; /* fp8 (E4M3) pool instead of k_cache / v_cache, or NULL */
    double k_scale, v_scale;            /* value = E4M3 value * scale */
} key_source;

static double e4m3_to_double(uint8_t code);

/* K_j and V_j of kv head g as doubles (head_dim each); returns 0, or
 * ORC_BOUNDS if the table entry that holds position j is not a block of the
 * pool. */
static int fetch_kv(const key_source *src, int64_t j, int g, double *kj, double *vj)
{
    const int d = src->head_dim;
    if (src->table_row == NULL) {
        const uint16_t *kp = src->k + j * src->kv_stride + (int64_t)g * d;
        const uint16_t *vp = src->v + j * src->kv_stride + (int64_t)g * d;
        for (int e = 0; e < d; ++e) kj[e] = bf16_to_double(kp[e]), vj[e] = bf16_to_double(vp[e]);
        return ORC_OK;
    }
    int64_t logical_block = j / src->block_size;
    if (logical_block >= src->max_blocks) return ORC_BOUNDS;
    int32_t phys = src->table_row[logical_block];
    if (phys < 0 || phys >= src->num_blocks) return ORC_BOUNDS;
    int64_t slot = orc_slot(src->table_row, src->block_size, j);
    int64_t row = (slot * src->kv_heads + g) * d;
    for (int e = 0; e < d; ++e) {
        if (src->k8_cache) {
            kj[e] = e4m3_to_double(src->k8_cache[row + e]) * src->k_scale;
            vj[e] = e4m3_to_double(src->v8_cache[row + e]) * src->v_scale;
        } else {
            kj[e] = bf16_to_double(src->k_cache[row + e]);
            vj[e] = bf16_to_double(src->v_cache[row + e]);
        }
    }
    return ORC_OK;
}

/* One query row against keys 0..n_keys-1 ([P1] §9.5, §19.1):
 *   s_j = scale * sum_e q[e] k_j[e]
 *   w_j = exp(s_j - max_r s_r) / sum_r exp(s_r - max_r s_r)
 *   out = sum_j w_j v_j
 * n_keys == 0 (a padded row, [P1] §13.5) gives out = 0.  `scores` holds
 * n_keys doubles; `weights`, if not NULL, receives w. */
static int attend_row(const uint16_t *qrow, const key_source *src, int g, int64_t n_keys,
                      double scale, double *scores, double *out, double *weights)
{
    const int d = src->head_dim;
    double kj[1024], vj[1024];
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (n_keys <= 0) return ORC_OK;
    if (d > 1024) return ORC_INVALID;

    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        if (fetch_kv(src, j, g, kj, vj) != ORC_OK) return ORC_BOUNDS;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += bf16_to_double(qrow[e]) * kj[e];
        scores[j] = scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) denom += exp(scores[j] - m);
    for (int64_t j = 0; j < n_keys; ++j) {
        fetch_kv(src, j, g, kj, vj);
        double w = exp(scores[j] - m) / denom;
        if (weights) weights[j] = w;
        for (int e = 0; e < d; ++e) out[e] += w * vj[e];
    }
    return ORC_OK;
}

static int check_heads(int num_heads, int kv_heads, int head_dim)
{
    if (num_heads <= 0 || kv_heads <= 0 || head_dim <= 0) return ORC_INVALID;
    if (num_heads % kv_heads != 0) return ORC_INVALID;
    return ORC_OK;
}

/*
 * Causal varlen prefill ([P1] §11.2, §10.2, §13.2; [P2] §2.7.2).
 * Sequence b owns query rows cu_q[b]..cu_q[b+1]-1 and a key context of
 * Lk = cu_k[b+1]-cu_k[b] positions; its Lq new queries are the last Lq
 * positions of that context, so query i sits at absolute position
 * p = Lk - Lq + i and sees keys 0..p (bottom-right causal alignment).
 * Query head h reads kv head h / (Hq/Hkv) ([P1] §19.6).
 * block_table == NULL: keys come from k/v rows cu_k[b]..cu_k[b+1]-1;
 * otherwise from the pool through block_table[b].
 * If `weights_out` is not NULL, the weights of row (wb, wh, wi) are written
 * there (Lk doubles; entries past p are 0).
 */
static int prefill_impl(const uint16_t *q, int64_t q_stride,
                        const uint16_t *k, const uint16_t *v, int64_t kv_stride,
                        const uint16_t *k_cache, const uint16_t *v_cache,
                        int64_t num_blocks, int block_size,
                        const int32_t *block_table, int max_blocks,
                        const int32_t *cu_q, const int32_t *cu_k, int num_seqs,
                        int num_heads, int kv_heads, int head_dim, double scale, double *out,
                        int wb, int wh, int wi, double *weights_out)
{
    if (check_heads(num_heads, kv_heads, head_dim) != ORC_OK) return ORC_INVALID;
    for (int b = 0; b < num_seqs; ++b) {
        int lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
        if (lq < 0 || lk < lq) return ORC_INVALID;
        if (block_table == NULL && lk != lq) return ORC_INVALID;
    }
    const int group = num_heads / kv_heads;
    int status = ORC_OK;
    const int64_t work = (int64_t)num_seqs * num_heads;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < work; ++task) {
        const int b = (int)(task / num_heads), h = (int)(task % num_heads);
        const int lq = cu_q[b + 1] - cu_q[b], lk = cu_k[b + 1] - cu_k[b];
        key_source src = {k_cache, v_cache,
                          block_table ? block_table + (int64_t)b * max_blocks : NULL,
                          num_blocks, block_size, max_blocks,
                          k ? k + (int64_t)cu_k[b] * kv_stride : NULL,
                          v ? v + (int64_t)cu_k[b] * kv_stride : NULL,
                          kv_stride, kv_heads, head_dim, NULL, NULL, 1.0, 1.0};
        double *scores = (double *)malloc(sizeof(double) * (size_t)(lk > 0 ? lk : 1));
        for (int i = 0; i < lq; ++i) {
            const int64_t t = (int64_t)cu_q[b] + i;
            const int64_t p = (int64_t)lk - lq + i;
            double *o = out + (t * num_heads + h) * head_dim;
            double *w = (weights_out && b == wb && h == wh && i == wi) ? weights_out : NULL;
            if (w) for (int64_t j = 0; j < lk; ++j) w[j] = 0.0;
            int rc = attend_row(q + t * q_stride + (int64_t)h * head_dim, &src, h / group, p + 1,
                                scale, scores, o, w);
            if (rc != ORC_OK) {
#pragma omp critical
                status = rc;
            }
        }
        free(scores);
    }
    return status;
}

int orc_prefill(const uint16_t *q, int64_t q_stride,
                const uint16_t *k, const uint16_t *v, int64_t kv_stride,
                const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks, int block_size,
                const int32_t *block_table, int max_blocks,
                const int32_t *cu_q, const int32_t *cu_k, int num_seqs,
                int num_heads, int kv_heads, int head_dim, double scale, double *out)
{
    return prefill_impl(q, q_stride, k, v, kv_stride, k_cache, v_cache, num_blocks, block_size,
                        block_table, max_blocks, cu_q, cu_k, num_seqs, num_heads, kv_heads,
                        head_dim, scale, out, -1, -1, -1, NULL);
}

/* Same as orc_prefill, and also returns the softmax weights of one row. */
int orc_prefill_weights(const uint16_t *q, int64_t q_stride,
                        const uint16_t *k, const uint16_t *v, int64_t kv_stride,
                        const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks,
                        int block_size, const int32_t *block_table, int max_blocks,
                        const int32_t *cu_q, const int32_t *cu_k, int num_seqs,
                        int num_heads, int kv_heads, int head_dim, double scale, double *out,
                        int b, int h, int i, double *weights)
{
    return prefill_impl(q, q_stride, k, v, kv_stride, k_cache, v_cache, num_blocks, block_size,
                        block_table, max_blocks, cu_q, cu_k, num_seqs, num_heads, kv_heads,
                        head_dim, scale, out, b, h, i, weights);
}

/*
 * Paged decode ([P1] §9.5, §11.4; [P3] #6): one query per sequence, q[b]
 * (seq stride q_stride), over context_lens[b] keys read through
 * block_table[b].  context_lens counts the token written this step, so the
 * query sits at position ctx-1 and sees every key.  ctx == 0 is a padded
 * row ([P1] §13.5) and yields zeros.  out is [num_seqs, Hq, d].
 */
static int decode_impl(const uint16_t *q, int64_t q_stride,
                       const uint16_t *k_cache, const uint16_t *v_cache,
                       const uint8_t *k8_cache, const uint8_t *v8_cache, double k_scale, double v_scale,
                       int64_t num_blocks, int block_size,
                       const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                       int num_seqs, int num_heads, int kv_heads, int head_dim, double scale, double *out)
{
    if (check_heads(num_heads, kv_heads, head_dim) != ORC_OK) return ORC_INVALID;
    for (int b = 0; b < num_seqs; ++b)
        if (context_lens[b] < 0) return ORC_INVALID;
    const int group = num_heads / kv_heads;
    int status = ORC_OK;
    const int64_t work = (int64_t)num_seqs * num_heads;

#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t task = 0; task < work; ++task) {
        const int b = (int)(task / num_heads), h = (int)(task % num_heads);
        const int64_t ctx = context_lens[b];
        key_source src = {k_cache, v_cache, block_table + (int64_t)b * max_blocks,
                          num_blocks, block_size, max_blocks, NULL, NULL, 0, kv_heads, head_dim,
                          k8_cache, v8_cache, k_scale, v_scale};
        double *scores = (double *)malloc(sizeof(double) * (size_t)(ctx > 0 ? ctx : 1));
        int rc = attend_row(q + (int64_t)b * q_stride + (int64_t)h * head_dim, &src, h / group, ctx,
                            scale, scores, out + ((int64_t)b * num_heads + h) * head_dim, NULL);
        free(scores);
        if (rc != ORC_OK) {
#pragma omp critical
            status = rc;
        }
    }
    return status;
}


int orc_decode(const uint16_t *q, int64_t q_stride,
               const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks, int block_size,
               const int32_t *block_table, int max_blocks, const int32_t *context_lens,
               int num_seqs, int num_heads, int kv_heads, int head_dim, double scale, double *out)
{
    return decode_impl(q, q_stride, k_cache, v_cache, NULL, NULL, 1.0, 1.0, num_blocks, block_size, block_table,
                       max_blocks, context_lens, num_seqs, num_heads, kv_heads, head_dim, scale, out);
}

/* ------------------------------------------------------------------ fp8 KV cache
 *
 * The pages list the KV precision as a way to fit longer contexts ([P1]
 * §17.3; [P3]'s arithmetic-intensity table counts FP8 as 1 byte per element)
 * but fix no format.  The reading taken here: each cache element is an OCP
 * FP8 E4M3 value (1 sign, 4 exponent bits with bias 7, 3 mantissa bits; no
 * infinities; S.1111.111 is NaN; largest finite 448), and a layer's K and V
 * each carry one float scale: stored code = E4M3(x / scale), with the
 * division in float (the precision of the bf16 inputs' widening) and
 * round-to-nearest-even with saturation to +-448; value = E4M3 value * scale.
 */

/* Value of an E4M3 code. */
static double e4m3_to_double(uint8_t code)
{
    const int s = code >> 7, e = (code >> 3) & 15, m = code & 7;
    if (e == 15 && m == 7) return NAN;
    const double mag = e == 0 ? ldexp(m / 8.0, -6) : ldexp(1.0 + m / 8.0, e - 7);
    return s ? -mag : mag;
}

double orc_e4m3_value(int code) { return e4m3_to_double((uint8_t)code); }

/* Nearest E4M3 code of a float (ties to even), saturating to +-448; NaN -> 0x7f. */
int orc_e4m3_encode(float x)
{
    if (isnan(x)) return 0x7f;
    const int s = signbit(x) ? 0x80 : 0;
    const double a = fabs((double)x);
    if (a >= 448.0) return s | 0x7e;
    int e2;
    frexp(a, &e2);                         /* a = f * 2^e2, f in [0.5, 1): leading bit 2^(e2-1) */
    if (a == 0.0 || e2 - 1 < -6) {         /* subnormal range: multiples of 2^-9 (code = k) */
        const int k = (int)nearbyint(ldexp(a, 9));
        return s | k;                      /* k == 8 is 2^-6, the first normal code */
    }
    int ex = e2 - 1;                       /* value = q * 2^(ex - 3), q in [8, 16] */
    int q = (int)nearbyint(ldexp(a, 3 - ex));
    if (q == 16) {
        q = 8;
        ++ex;
    }
    return s | ((ex + 7) << 3) | (q - 8);
}

/* KV write into an fp8 pool: code of float(bf16 value) / scale per element. */
int orc_store_kvcache_fp8(const uint16_t *k, int64_t k_stride, const uint16_t *v, int64_t v_stride,
                          int64_t num_tokens, int kv_heads, int head_dim, float k_scale, float v_scale,
                          uint8_t *k_cache, uint8_t *v_cache, int64_t num_blocks, int block_size,
                          const int32_t *slot_mapping)
{
    const int64_t row = (int64_t)kv_heads * head_dim;
    const int64_t num_slots = num_blocks * block_size;
    int status = ORC_OK;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t slot = slot_mapping[t];
        const int padding_row = slot == -1;
        if (padding_row) continue;
        if (slot < 0 || slot >= num_slots) { status = ORC_BOUNDS; continue; }
        for (int64_t e = 0; e < row; ++e) {
            const float kx = (float)bf16_to_double(k[t * k_stride + e]);
            const float vx = (float)bf16_to_double(v[t * v_stride + e]);
            k_cache[slot * row + e] = (uint8_t)orc_e4m3_encode(kx / k_scale);
            v_cache[slot * row + e] = (uint8_t)orc_e4m3_encode(vx / v_scale);
        }
    }
    return status;
}

/* Paged decode over an fp8 pool: as orc_decode, with K_j = E4M3 value *
 * k_scale and V_j = E4M3 value * v_scale. */
int orc_decode_fp8(const uint16_t *q, int64_t q_stride, const uint8_t *k_cache, const uint8_t *v_cache,
                   double k_scale, double v_scale, int64_t num_blocks, int block_size,
                   const int32_t *block_table, int max_blocks, const int32_t *context_lens,
                   int num_seqs, int num_heads, int kv_heads, int head_dim, double scale, double *out)
{
    return decode_impl(q, q_stride, NULL, NULL, k_cache, v_cache, k_scale, v_scale, num_blocks, block_size,
                       block_table, max_blocks, context_lens, num_seqs, num_heads, kv_heads, head_dim, scale, out);
}

/* ------------------------------------------------------------------ head norm, RoPE, KV write
 *
 * [P1] §12.2 and §19.7: after the fused QKV projection, every Q head and every
 * K head (not V) is RMS-normalised over its own d features, then rotated by
 * its token's position; the cache receives the rotated K and the plain V.
 */

/* Round a double to the nearest bf16 (ties to even), returned as its bits.
 * Direct rounding to 8 significant bits, so no intermediate float rounding. */
static uint16_t double_to_bf16(double x)
{
    float f;
    uint32_t u;
    if (isnan(x)) return 0x7fc0u;
    if (x == 0.0 || isinf(x)) {
        f = (float)x;
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    int e;
    const double m = frexp(x, &e);            /* x = m * 2^e, 0.5 <= |m| < 1 */
    double r = ldexp(nearbyint(ldexp(m, 8)), e - 8);  /* 8 significant bits, ties to even */
    if (fabs(x) < 1.1754943508222875e-38)     /* below 2^-126: bf16's subnormal grid is 2^-133 */
        r = ldexp(nearbyint(ldexp(x, 133)), -133);
    if (fabs(r) > 3.3895313892515355e38) r = x > 0 ? INFINITY : -INFINITY;  /* past bf16's largest */
    f = (float)r;                             /* exact: r has 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/* [P1] §19.5; [P4] §4.3 RMSNorm.rms_forward: r = 1 / sqrt(mean(x^2) + eps),
 * y = x * r, then (when w is given) y * w.  In double, no rounding. */
void orc_rmsnorm(const double *x, int n, const double *w, double eps, double *y)
{
    double ss = 0.0;
    for (int i = 0; i < n; ++i) ss += x[i] * x[i];
    const double r = 1.0 / sqrt(ss / n + eps);
    for (int i = 0; i < n; ++i) y[i] = x[i] * r * (w ? w[i] : 1.0);
}

/* [P4] §4.4 RotaryEmbedding: inv_freq[i] = 1 / base^(2i / d) for i < d/2; the
 * table row of position p is cos(p * inv_freq) followed by sin(p * inv_freq)
 * (d values).  Computed in double and stored as float, the precision in
 * which the table is held. */
void orc_rope_cos_sin(double base, int d, int64_t max_positions, float *table)
{
    const int half = d / 2;
    for (int64_t p = 0; p < max_positions; ++p)
        for (int i = 0; i < half; ++i) {
            const double inv_freq = 1.0 / pow(base, (2.0 * i) / d);
            const double phi = (double)p * inv_freq;
            table[p * d + i] = (float)cos(phi);
            table[p * d + half + i] = (float)sin(phi);
        }
}

/* [P1] §19.7: feature i is paired with feature i + d/2 (the two halves, not
 * neighbours); the pair (a, b) turns by phi: a' = a cos - b sin,
 * b' = a sin + b cos.  cs is one table row (cos half, then sin half). */
void orc_rope_apply(const double *x, int d, const float *cs, double *y)
{
    const int half = d / 2;
    for (int i = 0; i < half; ++i) {
        const double a = x[i], b = x[i + half];
        const double c = cs[i], s = cs[half + i];
        y[i] = a * c - b * s;
        y[i + half] = a * s + b * c;
    }
}

/* One head row, as the pages order it ([P1] §19.5 and §12.2): statistics and
 * normalisation in float precision (here double), the result rounded to the
 * activation dtype (bf16), multiplied by the bf16 weight and rounded again
 * (w == NULL: no head norm); then RoPE on those values, rounded once to bf16. */
static void norm_rope_row(const uint16_t *x_bits, int d, const uint16_t *w_bits, double eps, const float *cs,
                          uint16_t *out_bits)
{
    double x[1024], y[1024];
    for (int i = 0; i < d; ++i) x[i] = bf16_to_double(x_bits[i]);
    if (w_bits) {
        orc_rmsnorm(x, d, NULL, eps, y);
        for (int i = 0; i < d; ++i) {
            const double yn = bf16_to_double(double_to_bf16(y[i]));
            x[i] = bf16_to_double(double_to_bf16(yn * bf16_to_double(w_bits[i])));
        }
    }
    orc_rope_apply(x, d, cs, y);
    for (int i = 0; i < d; ++i) out_bits[i] = double_to_bf16(y[i]);
}

/* [P3] #8 fused RoPE and paged KV store, with [P1] §12.2's head norm:
 *   qkv       [T, (Hq + 2 Hkv) * d] bf16 bits, token stride qkv_stride; the
 *             Q heads, then the K heads, then the V heads ([P4] qkv.split)
 *   positions [T] int32, each in [0, max_positions)
 *   cos_sin   [max_positions, d] float (orc_rope_cos_sin's layout)
 *   q_weight, k_weight  [d] bf16 bits, or NULL for no head norm
 *   q_out     [T, Hq, d] bf16 bits, token stride q_out_stride: rotated Q
 *   k_cache, v_cache   pool rows `slot_mapping[t]` receive the rotated K and
 *             the unchanged V; slot -1 skips the write (q_out is still written).
 * A position outside the table or a slot outside the pool is reported
 * (status 4) and that token is skipped. */
int orc_norm_rope_store(const uint16_t *qkv, int64_t qkv_stride, int64_t num_tokens, int num_heads, int kv_heads,
                        int d, const int32_t *positions, const float *cos_sin, int64_t max_positions,
                        const uint16_t *q_weight, const uint16_t *k_weight, double eps,
                        uint16_t *q_out, int64_t q_out_stride,
                        uint16_t *k_cache, uint16_t *v_cache, int64_t num_blocks, int block_size,
                        const int32_t *slot_mapping)
{
    if (d <= 0 || d > 1024 || d % 2 || num_heads <= 0 || kv_heads <= 0) return ORC_INVALID;
    const int64_t row = (int64_t)kv_heads * d;
    const int64_t num_slots = num_blocks * block_size;
    int status = ORC_OK;
    for (int64_t t = 0; t < num_tokens; ++t) {
        const int64_t p = positions[t], slot = slot_mapping[t];
        if (p < 0 || p >= max_positions || (slot != -1 && (slot < 0 || slot >= num_slots))) {
            status = ORC_BOUNDS;
            continue;
        }
        const uint16_t *tok = qkv + t * qkv_stride;
        const float *cs = cos_sin + p * d;
        for (int h = 0; h < num_heads; ++h)
            norm_rope_row(tok + (int64_t)h * d, d, q_weight, eps, cs, q_out + t * q_out_stride + (int64_t)h * d);
        const int padding_row = slot == -1;  /* q is still rotated; nothing is stored */
        for (int g = 0; g < kv_heads && !padding_row; ++g) {
            norm_rope_row(tok + ((int64_t)num_heads + g) * d, d, k_weight, eps, cs, k_cache + slot * row + (int64_t)g * d);
            for (int i = 0; i < d; ++i)
                v_cache[slot * row + (int64_t)g * d + i] = tok[((int64_t)num_heads + kv_heads + g) * d + i];
        }
    }
    return status;
}


/* ------------------------------------------------------------------ step metadata
 *
 * [P4] prepare_prefill, step by step, for sequence b of the batch:
 *   seqlen = seq_lens[b] (cached + uncached tokens); start = min(num_cached,
 *   seqlen - 1) (a fully cached prompt still computes its last token);
 *   seqlen_q = num_scheduled; end = start + seqlen_q; positions start..end-1;
 *   cu_seqlens_q += seqlen_q; cu_seqlens_k += seqlen_k; slots block by block
 *   from start_block = start / bs to end_block = ceil(end / bs), the first
 *   block starting at start % bs and the last one ending at end.
 * seqlen_k is taken as `end`: the page writes `seqlen`, which is the same
 * whenever the rest of the prompt is scheduled at once; for a chunk, the keys
 * its last query may read end at `end` ([P1] §8.2, §11.2's key lengths).
 * A table entry that is not a block of the pool gives slot -1 and status 4;
 * end > seqlen or seqlen_q < 1 gives status 1.
 */
int orc_prepare_prefill(const int32_t *seq_lens, const int32_t *num_cached, const int32_t *num_scheduled,
                        int num_seqs, const int32_t *block_table, int max_blocks, int block_size, int64_t num_blocks,
                        int32_t *cu_seqlens_q, int32_t *cu_seqlens_k, int32_t *positions, int32_t *slot_mapping,
                        int32_t *max_seqlen_q, int32_t *max_seqlen_k)
{
    int status = ORC_OK;
    int64_t nq = 0;
    cu_seqlens_q[0] = 0;
    cu_seqlens_k[0] = 0;
    *max_seqlen_q = 0;
    *max_seqlen_k = 0;
    for (int b = 0; b < num_seqs; ++b) {
        const int seqlen = seq_lens[b];
        const int start = num_cached[b] < seqlen - 1 ? num_cached[b] : seqlen - 1;
        const int seqlen_q = num_scheduled[b];
        const int end = start + seqlen_q;
        if (seqlen_q < 1 || start < 0 || end > seqlen) status = ORC_INVALID;
        const int seqlen_k = end;
        for (int p = start; p < end; ++p) positions[nq + p - start] = p;
        cu_seqlens_q[b + 1] = cu_seqlens_q[b] + seqlen_q;
        cu_seqlens_k[b + 1] = cu_seqlens_k[b] + seqlen_k;
        if (seqlen_q > *max_seqlen_q) *max_seqlen_q = seqlen_q;
        if (seqlen_k > *max_seqlen_k) *max_seqlen_k = seqlen_k;
        const int32_t *table = block_table + (int64_t)b * max_blocks;
        const int start_block = start / block_size;
        const int end_block = (end + block_size - 1) / block_size;
        int64_t k = nq;
        for (int i = start_block; i < end_block; ++i) {
            const int ok = i < max_blocks && table[i] >= 0 && table[i] < num_blocks;
            if (!ok) status = ORC_BOUNDS;
            const int64_t base = ok ? (int64_t)table[i] * block_size : 0;
            int64_t slot_start = base, slot_end = base + block_size;
            if (i == start_block) slot_start += start % block_size;
            if (i == end_block - 1) slot_end = base + end - (int64_t)i * block_size;
            for (int64_t sl = slot_start; sl < slot_end; ++sl) slot_mapping[k++] = ok ? (int32_t)sl : -1;
        }
        nq += seqlen_q;
    }
    return status;
}

/* [P2] §2.7.3 and [P1] §11.4 prepare_decode: every sequence adds its last
 * token: position = seqlen - 1, context_lens = seqlen, slot = the table's
 * last block used (block (seqlen - 1) / bs) * bs + last_block_num_tokens - 1.
 * seqlen 0 is a padding row ([P1] §13.5): position 0, context 0, slot -1. */
int orc_prepare_decode(const int32_t *seq_lens, int num_seqs, const int32_t *block_table, int max_blocks,
                       int block_size, int64_t num_blocks, int32_t *positions, int32_t *context_lens,
                       int32_t *slot_mapping)
{
    int status = ORC_OK;
    for (int b = 0; b < num_seqs; ++b) {
        const int seqlen = seq_lens[b];
        if (seqlen < 0) status = ORC_INVALID;
        if (seqlen <= 0) {
            positions[b] = 0;
            context_lens[b] = 0;
            slot_mapping[b] = -1;
            continue;
        }
        const int num_blocks_seq = (seqlen + block_size - 1) / block_size;
        const int last_block_num_tokens = seqlen - (num_blocks_seq - 1) * block_size;
        positions[b] = seqlen - 1;
        context_lens[b] = seqlen;
        const int last = num_blocks_seq - 1;
        const int32_t id = last < max_blocks ? block_table[(int64_t)b * max_blocks + last] : -1;
        if (id < 0 || id >= num_blocks) {
            status = ORC_BOUNDS;
            slot_mapping[b] = -1;
        } else {
            slot_mapping[b] = (int32_t)((int64_t)id * block_size + last_block_num_tokens - 1);
        }
    }
    return status;
}
