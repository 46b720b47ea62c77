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
 *   [P3] "VLLM on Fain的Blog" (Pico-vLLM log), #6 paged decode kernel.
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
} key_source;

/* Pointers to K_j and V_j for kv head g; returns 0, or ORC_BOUNDS if the table
 * entry that holds position j is not a block of the pool. */
static int fetch_kv(const key_source *src, int64_t j, int g, const uint16_t **kj, const uint16_t **vj)
{
    if (src->table_row == NULL) {
        *kj = src->k + j * src->kv_stride + (int64_t)g * src->head_dim;
        *vj = src->v + j * src->kv_stride + (int64_t)g * src->head_dim;
        return ORC_OK;
    }
    int64_t logical_block = j / src->block_size;
    if (logical_block >= src->max_blocks) return ORC_BOUNDS;
    int32_t phys = src->table_row[logical_block];
    if (phys < 0 || phys >= src->num_blocks) return ORC_BOUNDS;
    int64_t slot = orc_slot(src->table_row, src->block_size, j);
    int64_t row = (slot * src->kv_heads + g) * src->head_dim;
    *kj = src->k_cache + row;
    *vj = src->v_cache + row;
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
    for (int e = 0; e < d; ++e) out[e] = 0.0;
    if (n_keys <= 0) return ORC_OK;

    double m = -INFINITY;
    for (int64_t j = 0; j < n_keys; ++j) {
        const uint16_t *kj, *vj;
        if (fetch_kv(src, j, g, &kj, &vj) != ORC_OK) return ORC_BOUNDS;
        double dot = 0.0;
        for (int e = 0; e < d; ++e) dot += bf16_to_double(qrow[e]) * bf16_to_double(kj[e]);
        scores[j] = scale * dot;
        if (scores[j] > m) m = scores[j];
    }
    double denom = 0.0;
    for (int64_t j = 0; j < n_keys; ++j) denom += exp(scores[j] - m);
    for (int64_t j = 0; j < n_keys; ++j) {
        const uint16_t *kj, *vj;
        fetch_kv(src, j, g, &kj, &vj);
        double w = exp(scores[j] - m) / denom;
        if (weights) weights[j] = w;
        for (int e = 0; e < d; ++e) out[e] += w * bf16_to_double(vj[e]);
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
                          kv_stride, kv_heads, head_dim};
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
int orc_decode(const uint16_t *q, int64_t q_stride,
               const uint16_t *k_cache, const uint16_t *v_cache, int64_t num_blocks, int block_size,
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
                          num_blocks, block_size, max_blocks, NULL, NULL, 0, kv_heads, head_dim};
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
