/*
 * pa.h -- C ABI of libpa: attention over a block-paged KV cache on one GB300
 * (sm_103a).
 *
 * The three calls are the three GPU steps of one attention layer in a
 * nano-vLLM style engine ("大模型推理入门与 nano-vLLM 源码详解" §13.1-13.2 and
 * §20.5.2; "nano-vllm 技术分析" §4.1 Attention): write the new tokens' K/V
 * into the cache by slot_mapping, then either causal varlen prefill over
 * cu_seqlens (reading cached prefix blocks through block_table) or decode of
 * one query per sequence over context_lens keys.
 *
 * Conventions for every call:
 *   - All tensor pointers are DEVICE pointers owned by the caller.  The
 *     library allocates no device memory; scratch space is passed in.
 *   - bf16 data (IEEE binary16 "brain float", 2 bytes), int32 metadata.
 *   - head_dim must be 128; Hq / Hkv (the query heads per KV head) must be
 *     1, 2, 4 or 8; Hkv must be 1, 2, 4 or 8; block_size must be a multiple
 *     of 16 in [16, 1024].  Other shapes return PA_ERR_UNSUPPORTED.
 *   - The per-layer cache layout is [num_blocks, block_size, Hkv, head_dim],
 *     row-major: pool row `slot` starts at element slot * Hkv * head_dim
 *     ("大模型推理入门与 nano-vLLM 源码详解" §11.5, the per-layer slice of the
 *     [2, layers, num_blocks, block_size, Hkv, head_dim] pool).
 *   - Calls are asynchronous on `stream` (a cudaStream_t; NULL = the legacy
 *     default stream).  They never synchronise, never allocate, and launch
 *     a grid whose shape depends only on the host arguments, so they can be
 *     captured in a CUDA graph.
 *   - Errors the host can see (null pointers, unsupported shapes, negative
 *     sizes) are returned synchronously and nothing is launched.  A launch
 *     failure returns PA_ERR_CUDA.  Errors only the device can see (a slot
 *     or block id outside the pool, a -1 table entry inside a live context,
 *     a context longer than the table or the stated maximum) are written to
 *     *dev_status (if dev_status is not NULL) as the first nonzero pa_status
 *     code; the offending row is skipped and the kernel still completes.
 *     Kernels never trap.  The caller zeroes *dev_status before the call and
 *     reads it after synchronising.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = 1, /* null pointer, negative size, inconsistent arguments */
    PA_ERR_UNSUPPORTED = 2, /* shape outside what the kernels are built for */
    PA_ERR_CUDA = 3,        /* a CUDA runtime call or a launch failed */
    PA_ERR_BOUNDS = 4,      /* (device) an index outside the pool or the table */
    PA_ERR_TIMEOUT = 5      /* (device) a bounded wait gave up */
} pa_status;

/* Static English text for a status code; never NULL. */
const char *pa_status_string(int status);

/* Version of this ABI, major * 100 + minor. */
int pa_abi_version(void);

/*
 * KV-cache bytes per token position across a whole model:
 * 2 (K and V) x layers x kv_heads x head_dim x elem_bytes
 * ("大模型推理入门与 nano-vLLM 源码详解" §4.4; 114,688 for Qwen3-0.6B bf16).
 * Returns 0 if any argument is not positive.
 */
size_t pa_kv_bytes_per_token(int layers, int kv_heads, int head_dim, int elem_bytes);

/*
 * KV write ("大模型推理入门与 nano-vLLM 源码详解" §13.1; "nano-vllm 技术分析"
 * §4.1 store_kvcache).  For every token t < num_tokens with
 * s = slot_mapping[t] != -1, copy the num_kv_heads * head_dim bf16 values of
 * k[t] to pool row s of k_cache, and those of v[t] to row s of v_cache.
 *
 *   k, v          [num_tokens, num_kv_heads, head_dim] bf16; head rows are
 *                 packed, consecutive tokens are k_stride_tok / v_stride_tok
 *                 ELEMENTS apart (k and v may be column views of a fused
 *                 QKV buffer).  Strides must be >= num_kv_heads * head_dim.
 *   k_cache,      [num_blocks, block_size, num_kv_heads, head_dim] bf16,
 *   v_cache       written in place.
 *   slot_mapping  [num_tokens] int32; -1 marks a padding row (skipped).
 *                 Any other value outside [0, num_blocks * block_size) sets
 *                 PA_ERR_BOUNDS in *dev_status and that row is skipped.
 *                 Live slots must be distinct (not checked).
 * num_tokens == 0 is valid and launches nothing.  The copy is bit-exact.
 */
pa_status pa_store_kvcache(const void *k, int64_t k_stride_tok, const void *v, int64_t v_stride_tok,
                           int64_t num_tokens, int num_kv_heads, int head_dim,
                           void *k_cache, void *v_cache, int64_t num_blocks, int block_size,
                           const int32_t *slot_mapping, int32_t *dev_status, void *stream);

/*
 * Head RMSNorm, rotary position embedding and KV write in one pass
 * ("大模型推理入门与 nano-vLLM 源码详解" §12.2, §19.3 RMSNorm, §19.7 RoPE;
 * "nano-vllm 技术分析" §4.3-4.4; "VLLM on Fain的Blog" #8 fused RoPE and paged
 * KV store).  For every token t:
 *   - each Q head and each K head of qkv[t] is RMS-normalised over its
 *     head_dim features (fp32 statistics, 1 / sqrt(mean(x^2) + eps), result
 *     rounded to bf16, times the bf16 weight, rounded again), unless that
 *     weight pointer is NULL;
 *   - then rotated by position positions[t]: feature i pairs with feature
 *     i + head_dim / 2 and (a, b) -> (a cos - b sin, a sin + b cos), with
 *     cos / sin from row positions[t] of cos_sin (fp32 math, bf16 result);
 *   - rotated Q goes to q_out[t]; rotated K and the unchanged V go to pool row
 *     slot_mapping[t] of k_cache / v_cache.  slot -1 stores nothing (q_out[t]
 *     is still written).
 *
 *   qkv           [num_tokens, (num_heads + 2 num_kv_heads) * head_dim] bf16,
 *                 the Q heads, then the K heads, then the V heads of a token
 *                 (the fused QKV projection's output); token stride
 *                 qkv_stride_tok elements (a multiple of 8).
 *   positions     [num_tokens] int32, each in [0, max_positions).
 *   cos_sin       [max_positions, head_dim] fp32: cos(p * f_i) for the
 *                 head_dim / 2 pairs, then sin(p * f_i), f_i = base^(-2i / head_dim)
 *                 (the caller builds it once per model).
 *   q_norm_weight, k_norm_weight   [head_dim] bf16 or NULL.
 *   eps           added to mean(x^2), >= 0.
 *   q_out         [num_tokens, num_heads, head_dim] bf16, token stride
 *                 q_out_stride_tok (a multiple of 8).  It may be the Q part of
 *                 qkv itself (same stride): each row is read before it is
 *                 written.
 *   k_cache, v_cache, num_blocks, block_size, slot_mapping   as for
 *                 pa_store_kvcache.
 * A position outside the table or a slot outside the pool sets PA_ERR_BOUNDS
 * and that token is skipped.  Pointers must be 16-byte aligned.  The V copy
 * is bit-exact; Q and K agree with an fp64 evaluation of the same steps up to
 * the bf16 rounding of each step.
 */
/*
 * Fill the rotary table pa_norm_rope_store_kvcache reads ("nano-vllm 技术分析"
 * §4.4 RotaryEmbedding; "大模型推理入门与 nano-vLLM 源码详解" §19.7, rope_theta):
 * row p of table [max_positions, head_dim] fp32 (device) holds cos(p * f_i)
 * for i < head_dim / 2, then sin(p * f_i), with f_i = base^(-2i / head_dim),
 * evaluated in double precision and rounded to float.  base > 1, head_dim even
 * and at most 1024; max_positions == 0 launches nothing.
 */
pa_status pa_rope_cos_sin_table(double base, int head_dim, int64_t max_positions, float *table, void *stream);

pa_status pa_norm_rope_store_kvcache(const void *qkv, int64_t qkv_stride_tok, int64_t num_tokens,
                                     int num_heads, int num_kv_heads, int head_dim,
                                     const int32_t *positions, const float *cos_sin, int64_t max_positions,
                                     const void *q_norm_weight, const void *k_norm_weight, float eps,
                                     void *q_out, int64_t q_out_stride_tok,
                                     void *k_cache, void *v_cache, int64_t num_blocks, int block_size,
                                     const int32_t *slot_mapping, int32_t *dev_status, void *stream);

/*
 * Step metadata of a prefill batch, built on the device ("nano-vllm 技术分析",
 * prepare_prefill; "大模型推理引擎入门 ... 对着日志读懂 nano-vllm" §2.7.2;
 * "大模型推理入门与 nano-vLLM 源码详解" §11.2-11.3).  For sequence b with
 * seq_lens[b] tokens of which num_cached[b] are in the cache, and
 * num_scheduled[b] scheduled this step:
 *   start = min(num_cached, seq_len - 1), end = start + num_scheduled;
 *   positions of its tokens: start .. end-1 (concatenated in sequence order);
 *   cu_seqlens_q: prefix sums of num_scheduled; cu_seqlens_k: of end (the
 *   keys its last query reads: the whole prompt once the rest is scheduled);
 *   max_seqlens[0] / [1]: the largest num_scheduled / end;
 *   slot_mapping[token] = block_table[b][pos / block_size] * block_size +
 *   pos % block_size.
 *   seq_lens, num_cached, num_scheduled   [num_seqs] int32 (device)
 *   block_table   [num_seqs, max_blocks] int32 (device)
 *   cu_seqlens_q, cu_seqlens_k   [num_seqs + 1] int32 out
 *   positions, slot_mapping      [max_tokens] int32 out (capacity)
 *   max_seqlens   [2] int32 out
 * A sequence with num_scheduled < 1 or end > seq_len sets PA_ERR_INVALID_ARG
 * and contributes no tokens; a table entry outside the pool gives slot -1 and
 * PA_ERR_BOUNDS; tokens past max_tokens set PA_ERR_BOUNDS and are not written.
 * Two launches on `stream`; graph-capturable.
 */
pa_status pa_prepare_prefill(const int32_t *seq_lens, const int32_t *num_cached, const int32_t *num_scheduled,
                             int num_seqs, const int32_t *block_table, int max_blocks, int block_size,
                             int64_t num_blocks, int32_t *cu_seqlens_q, int32_t *cu_seqlens_k, int32_t *positions,
                             int32_t *slot_mapping, int64_t max_tokens, int32_t *max_seqlens, int32_t *dev_status,
                             void *stream);

/*
 * Step metadata of a decode batch, built on the device
 * ("大模型推理引擎入门 ... 对着日志读懂 nano-vllm" §2.7.3; "大模型推理入门与
 * nano-vLLM 源码详解" §11.4, §13.5): sequence b adds its last token:
 * positions[b] = seq_lens[b] - 1, context_lens[b] = seq_lens[b], slot_mapping[b]
 * = the slot of that position.  seq_lens[b] == 0 marks a padding row (a CUDA
 * graph's spare batch entry): position 0, context 0, slot -1.  All arrays are
 * [num_seqs] int32 on the device.  A table entry outside the pool gives slot
 * -1 and PA_ERR_BOUNDS; a negative length sets PA_ERR_INVALID_ARG.
 */
pa_status pa_prepare_decode(const int32_t *seq_lens, int num_seqs, const int32_t *block_table, int max_blocks,
                            int block_size, int64_t num_blocks, int32_t *positions, int32_t *context_lens,
                            int32_t *slot_mapping, int32_t *dev_status, void *stream);

/*
 * Causal varlen prefill ("大模型推理入门与 nano-vLLM 源码详解" §11.2, §13.2-13.3,
 * §10.2; flash_attn_varlen_func as nano-vLLM calls it, §20.5.2.2).
 * Sequence b owns query rows cu_seqlens_q[b] .. cu_seqlens_q[b+1]-1 and a key
 * context of Lk_b = cu_seqlens_k[b+1] - cu_seqlens_k[b] positions; its
 * Lq_b queries are the LAST Lq_b positions of that context, so query i may
 * read keys 0 .. Lk_b - Lq_b + i (bottom-right causal alignment).  Query
 * head h reads KV head h / (num_heads / num_kv_heads).
 *
 *   q             [Tq, num_heads, head_dim] bf16, token stride q_stride_tok
 *                 elements (a multiple of 8); Tq = cu_seqlens_q[num_seqs].
 *   num_tokens    rows q holds (and, without a table, k and v hold): at
 *                 least Tq.  The kernel reads no row at or past it; a
 *                 sequence whose rows would pass it sets PA_ERR_INVALID_ARG
 *                 and is skipped.  0 launches nothing.
 *   block_table   NULL: keys come from k / v rows cu_seqlens_k[b] ..
 *                 (token stride kv_stride_tok), which requires
 *                 cu_seqlens_k == cu_seqlens_q (checked on the device:
 *                 PA_ERR_INVALID_ARG in *dev_status) and max_seqlen_k ==
 *                 max_seqlen_q (checked on the host).  k_cache/v_cache are
 *                 then ignored and may be NULL.
 *                 Otherwise [num_seqs, max_blocks_per_seq] int32: key j of
 *                 sequence b is pool row block_table[b][j / block_size] *
 *                 block_size + j % block_size of k_cache / v_cache (the
 *                 caller ran pa_store_kvcache for this call's tokens first);
 *                 k / v are ignored and may be NULL.
 *   max_seqlen_q, max_seqlen_k   host-side upper bounds of Lq_b and Lk_b;
 *                 they size the grid.  A sequence that exceeds them sets
 *                 PA_ERR_BOUNDS and its rows beyond the bound are not computed.
 *   scale         softmax scale applied to q.k (1/sqrt(head_dim) usually).
 *   out           [Tq, num_heads, head_dim] bf16, packed.
 *   workspace     device scratch of pa_prefill_workspace_bytes(num_seqs,
 *                 max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads) bytes,
 *                 256-byte aligned (NULL when that is 0); its contents on entry
 *                 do not matter.  A call with fewer (query tile pair, KV head)
 *                 items than fill the GPU twice splits each item's keys into
 *                 ranges computed by different CTAs and merges their softmax
 *                 statistics exactly (§9.5); the workspace holds the shares.
 *                 Calls that overlap on the GPU must not share a workspace.
 * Sequences with Lq_b == 0 are skipped.  Lk_b < Lq_b sets PA_ERR_INVALID_ARG.
 */
size_t pa_prefill_workspace_bytes(int num_seqs, int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads);

pa_status pa_prefill_paged(const void *q, int64_t q_stride_tok, int64_t num_tokens,
                           const void *k, const void *v, int64_t kv_stride_tok,
                           const void *k_cache, const void *v_cache, int64_t num_blocks, int block_size,
                           const int32_t *block_table, int max_blocks_per_seq,
                           const int32_t *cu_seqlens_q, const int32_t *cu_seqlens_k, int num_seqs,
                           int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads,
                           int head_dim, float scale, void *out, void *workspace, size_t workspace_bytes,
                           int32_t *dev_status, void *stream);

/*
 * Test hook, not part of the computation: makes the bounded waits of
 * pa_prefill_paged and pa_norm_rope_store_kvcache run out, for the calls
 * launched after this one (process-wide).  With cycles > 0, one wait of every
 * CTA of those kernels (the prefill's MMA issuer, the fused write's compute
 * warps) is on a barrier that nothing arrives on, and every pipeline wait
 * gives up after `cycles` SM clock cycles instead of the default 2^31 (about a
 * second).  0 restores normal operation.  A call whose wait gives up writes
 * PA_ERR_TIMEOUT to *dev_status; its CTAs then wait for their own copies and
 * MMAs in flight (those waits keep the default limit), free their tensor
 * memory and return, leaving the output incomplete and the stream usable.
 */
void pa_test_stall_pipelines(long long cycles);

/*
 * Bytes of scratch pa_decode_paged needs for these host-side sizes on the
 * current device (it depends on the device's SM count).  pa_decode_paged_fp8
 * cuts contexts into no more splits than pa_decode_paged (its splits are
 * longer: its tokens carry half the bytes), so the same size serves it.
 * Returns 0 when the arguments are invalid.
 */
size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len);

/*
 * Paged decode of one query per sequence ("大模型推理入门与 nano-vLLM 源码详解"
 * §9.5, §11.4, §13.5; flash_attn_with_kvcache as nano-vLLM calls it).
 * Sequence b attends with q[b] to keys 0 .. context_lens[b]-1 read through
 * block_table[b] (context_lens counts the token written this step).
 * Softmax statistics of key ranges ("splits") are merged exactly as in §9.5
 * (maximum, exponent sum, weighted numerator), never per page: through the
 * workspace and a merge kernel, or, for long contexts in a large batch (the
 * bf16 calls whose split plan would exceed eight splits, with
 * max_context_len <= 8192 and at least four cluster CTAs per SM), inside one
 * thread-block cluster per sequence (eight equal splits, merged in
 * distributed shared memory), which leaves the workspace untouched.  Either
 * way the caller passes a workspace of the size below.  Arithmetic: scores,
 * softmax statistics and the weighted sums in fp32; with 4 or 8 query heads
 * per KV head the dot products and P.V run on tensor cores (bf16 operands,
 * fp32 accumulation, P rounded to bf16), otherwise on CUDA cores in fp32.
 *
 *   q             [num_seqs, num_heads, head_dim] bf16, seq stride
 *                 q_stride_seq elements.
 *   block_table   [num_seqs, max_blocks_per_seq] int32 (-1 padded; only the
 *                 first ceil(ctx / block_size) entries are read).
 *   context_lens  [num_seqs] int32.  0 marks a padded row: its output is 0
 *                 and nothing is read.  A value above max_context_len or
 *                 max_blocks_per_seq * block_size sets PA_ERR_BOUNDS and the
 *                 row's output is 0.
 *   max_context_len  host-side upper bound of context_lens (sizes the grid).
 *   out           [num_seqs, num_heads, head_dim] bf16, packed.
 *   workspace     device scratch of at least
 *                 pa_decode_workspace_bytes(num_seqs, num_heads, head_dim,
 *                 max_context_len) bytes, 256-byte aligned; its contents on
 *                 entry do not matter.  Calls that overlap on the GPU must
 *                 not share a workspace.
 */
pa_status pa_decode_paged(const void *q, int64_t q_stride_seq,
                          const void *k_cache, const void *v_cache, int64_t num_blocks, int block_size,
                          const int32_t *block_table, int max_blocks_per_seq,
                          const int32_t *context_lens, int num_seqs, int max_context_len,
                          int num_heads, int num_kv_heads, int head_dim, float scale, void *out,
                          void *workspace, size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * The decode step's KV write and paged decode in one launch ("大模型推理入门与
 * nano-vLLM 源码详解" §13.1 and §13.5: store_kvcache then attention over the
 * cache).  For every sequence b with context_lens[b] > 0, k_new[b] and
 * v_new[b] (the token at position p = context_lens[b] - 1) are written to pool
 * row block_table[b][p / block_size] * block_size + p % block_size, and q[b]
 * attends to keys 0 .. p as in pa_decode_paged.  The result (out and the pool)
 * is the same as pa_store_kvcache with that row as slot_mapping[b], followed
 * by pa_decode_paged with the same arguments.
 *
 *   k_new, v_new  [num_seqs, num_kv_heads, head_dim] bf16, sequence stride
 *                 kv_new_stride_seq elements (a multiple of 8, at least
 *                 num_kv_heads * head_dim); 16-byte aligned.
 *   k_cache, v_cache  bf16 pools, written.
 *   Every other argument, the workspace and the errors as pa_decode_paged;
 *   an invalid block id of the new token's row sets PA_ERR_BOUNDS and that
 *   row is neither written nor read.  Rows of padded sequences (context 0)
 *   are not written.
 */
pa_status pa_store_decode_paged(const void *q, int64_t q_stride_seq, const void *k_new, const void *v_new,
                                int64_t kv_new_stride_seq, void *k_cache, void *v_cache, int64_t num_blocks,
                                int block_size, const int32_t *block_table, int max_blocks_per_seq,
                                const int32_t *context_lens, int num_seqs, int max_context_len, int num_heads,
                                int num_kv_heads, int head_dim, float scale, void *out, void *workspace,
                                size_t workspace_bytes, int32_t *dev_status, void *stream);

/*
 * The attention decode step of one layer from the fused QKV projection's
 * output, in one launch (plus the split merge): the per-head RMSNorm and RoPE
 * of the new token ("nano-vllm 技术分析" §4.3-4.4; "大模型推理入门与 nano-vLLM
 * 源码详解" §19.3, §19.7, §12.2), its KV write and the paged decode.  For every
 * sequence b with context_lens[b] > 0, at position p = context_lens[b] - 1:
 *   - each query head and key head of qkv[b] is normalised and rotated as in
 *     pa_norm_rope_store_kvcache (norm skipped without its weight; cos / sin
 *     from row p of cos_sin);
 *   - the rotated key heads and the unchanged value heads go to the pool row
 *     of position p (through block_table), as pa_store_decode_paged writes;
 *   - the rotated query attends to keys 0 .. p as in pa_decode_paged.
 * The result equals pa_norm_rope_store_kvcache (positions p, slots the rows
 * of p) followed by pa_decode_paged over its q_out, up to the bf16 rounding
 * of the normalised values (the sum of squares is added in another order).
 *
 *   qkv           [num_seqs, (num_heads + 2 num_kv_heads) * head_dim] bf16:
 *                 query heads, key heads, value heads; sequence stride
 *                 qkv_stride_seq elements (a multiple of 8); 16-byte aligned.
 *   cos_sin, max_positions, q_norm_weight, k_norm_weight, eps   as for
 *                 pa_norm_rope_store_kvcache; a position at or past
 *                 max_positions sets PA_ERR_BOUNDS and that sequence's output
 *                 is zero and its row is not written.
 *   Every other argument, the workspace and the errors as
 *   pa_store_decode_paged.
 */
pa_status pa_norm_rope_store_decode_paged(const void *qkv, int64_t qkv_stride_seq, const float *cos_sin,
                                          int64_t max_positions, const void *q_norm_weight,
                                          const void *k_norm_weight, float eps, void *k_cache, void *v_cache,
                                          int64_t num_blocks, int block_size, const int32_t *block_table,
                                          int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                          int max_context_len, int num_heads, int num_kv_heads, int head_dim,
                                          float scale, void *out, void *workspace, size_t workspace_bytes,
                                          int32_t *dev_status, void *stream);

/*
 * fp8 KV cache ("大模型推理入门与 nano-vLLM 源码详解" §17.3 names the KV
 * precision as the lever for longer contexts; "VLLM on Fain的Blog" counts FP8
 * at one byte per element.  The pages fix no format; this library's is the
 * OCP FP8 E4M3 format with one float scale per layer for K and one for V).
 *
 * pa_store_kvcache_fp8: as pa_store_kvcache, but pool element e receives the
 * E4M3 code of float(x) / scale (division in fp32, round to nearest even,
 * saturating to +-448; NaN stays NaN).  k_cache / v_cache are
 * [num_blocks, block_size, num_kv_heads, head_dim] bytes.  Scales must be
 * positive and finite.  k, v and the caches must be 16-byte aligned and the
 * token strides multiples of 8.  The codes are deterministic (bit-exact).
 */
pa_status pa_store_kvcache_fp8(const void *k, int64_t k_stride_tok, const void *v, int64_t v_stride_tok,
                               int64_t num_tokens, int num_kv_heads, int head_dim, float k_scale, float v_scale,
                               void *k_cache, void *v_cache, int64_t num_blocks, int block_size,
                               const int32_t *slot_mapping, int32_t *dev_status, void *stream);

/*
 * pa_decode_paged_fp8: pa_decode_paged over fp8 pools written by
 * pa_store_kvcache_fp8, with K_j = E4M3 value * k_scale and V_j = E4M3 value *
 * v_scale.  Same arguments, workspace (pa_decode_workspace_bytes) and errors
 * as pa_decode_paged; half the bytes per context token.  The codes are
 * converted to f16 exactly and multiplied on tensor cores with fp32
 * accumulation: q enters as an f16 value (each head scaled by a power of two,
 * undone on the score, so any normal bf16 query is exact), P is rounded to
 * f16 for P.V.
 */
pa_status pa_decode_paged_fp8(const void *q, int64_t q_stride_seq, const void *k_cache, const void *v_cache,
                              float k_scale, float v_scale, int64_t num_blocks, int block_size,
                              const int32_t *block_table, int max_blocks_per_seq, const int32_t *context_lens,
                              int num_seqs, int max_context_len, int num_heads, int num_kv_heads, int head_dim,
                              float scale, void *out, void *workspace, size_t workspace_bytes,
                              int32_t *dev_status, void *stream);

/*
 * Paged decode for callers that cannot allocate device memory.  (The pages
 * describe no counterpart: this is a calling convention of this library.)
 *
 * Who needs it: code embedded in a host framework that owns the whole device
 * memory pool and forbids foreign cudaMalloc calls, services that must not
 * allocate once they serve requests, and plain C callers with no
 * device-memory manager.  Such callers cannot provide the workspace that
 * pa_decode_paged asks for.
 *
 * Same arguments and result as pa_decode_paged, without the workspace: the
 * split partials live in a fixed device array inside this library, of
 * PA_DECODE_NOALLOC_SCRATCH_BYTES bytes, that every GPU which loads the
 * library holds until the process exits.  The call allocates nothing.
 *   - If pa_decode_workspace_bytes(num_seqs, num_heads, head_dim,
 *     max_context_len) exceeds PA_DECODE_NOALLOC_SCRATCH_BYTES, it returns
 *     PA_ERR_UNSUPPORTED and launches nothing; use pa_decode_paged then.
 *   - The first call on each device looks up the array's device address
 *     (with that device current) and keeps it for the life of the process;
 *     make that first call before any stream capture begins.  After
 *     cudaDeviceReset (or any reset of the device's primary context) the
 *     library's module is loaded again at another address and the kept one
 *     is stale: do not call this entry point after such a reset.
 *   - All calls share the one array: calls that overlap on the GPU (on
 *     different streams, or from different threads) race and give wrong
 *     results.  Calls on one stream are ordered and safe.  The array keeps
 *     the last call's contents; nothing in it needs to start at zero.
 */
#define PA_DECODE_NOALLOC_SCRATCH_BYTES ((size_t)32 << 20)

pa_status pa_decode_paged_noalloc(const void *q, int64_t q_stride_seq,
                                  const void *k_cache, const void *v_cache, int64_t num_blocks, int block_size,
                                  const int32_t *block_table, int max_blocks_per_seq,
                                  const int32_t *context_lens, int num_seqs, int max_context_len,
                                  int num_heads, int num_kv_heads, int head_dim, float scale, void *out,
                                  int32_t *dev_status, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
