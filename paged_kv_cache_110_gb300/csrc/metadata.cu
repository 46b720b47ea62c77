// metadata.cu -- the per-step attention metadata, built on the device from
// per-sequence counts and the device-resident block tables.
//
// What it computes ("nano-vllm 技术分析", the prefill parameter computation
// prepare_prefill; "大模型推理引擎入门 ... 对着日志读懂 nano-vllm" §2.7.2-2.7.3;
// "大模型推理入门与 nano-vLLM 源码详解" §11.2-11.4):
//   prefill, for sequence b: start = min(num_cached, seq_len - 1), the
//     scheduled tokens are positions start .. end-1 (end = start +
//     num_scheduled); cu_seqlens_q / cu_seqlens_k are the prefix sums of
//     num_scheduled and of end (the keys the last query reads); max_seqlen_q /
//     max_seqlen_k their maxima; every token's slot is
//     table[b][pos / bs] * bs + pos % bs;
//   decode: every sequence adds its last token: position seq_len - 1,
//     context_lens seq_len, slot of that position; seq_len 0 is a padding row
//     (position 0, context 0, slot -1).
// A host scheduler thus uploads three int32 per sequence (or nothing, when the
// counts are already on the device) instead of per-token arrays.
//
// Design: prefill takes two launches -- one CTA of 1024 threads scans the
// per-sequence counts (cu_seqlens and maxima), then a grid over sequences
// expands each sequence's tokens (positions and slots, coalesced writes).
// Decode is one thread per sequence.
#include "pa_common.cuh"

namespace {

constexpr int SCAN_THREADS = 1024;

struct SeqCounts {
    int start, q, k;  // first scheduled position, scheduled tokens, keys (end)
    bool ok;
};

__device__ __forceinline__ SeqCounts counts(const int32_t *seq_lens, const int32_t *num_cached,
                                            const int32_t *num_scheduled, int b)
{
    SeqCounts c;
    const int len = seq_lens[b], cached = num_cached[b], sched = num_scheduled[b];
    c.start = cached < len - 1 ? cached : len - 1;
    c.ok = sched >= 1 && c.start >= 0 && int64_t(c.start) + sched <= len;
    c.q = c.ok ? sched : 0;
    c.k = c.ok ? c.start + sched : 0;
    return c;
}

// Block-wide inclusive scan of one value per thread (1024 threads).
__device__ __forceinline__ int64_t block_scan(int64_t v, int64_t *warp_sums)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int64_t n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v += n;
    }
    if (lane == 31) warp_sums[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int64_t w = warp_sums[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int64_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_sums[lane] = w;
    }
    __syncthreads();
    const int64_t r = v + (warp > 0 ? warp_sums[warp - 1] : 0);
    __syncthreads();  // warp_sums is reused by the next call
    return r;
}

__device__ __forceinline__ int block_max(int v, int *warp_max)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int o = 16; o >= 1; o >>= 1) v = max(v, __shfl_xor_sync(0xffffffffu, v, o));
    if (lane == 0) warp_max[warp] = v;
    __syncthreads();
    int r = warp_max[0];
    for (int w = 1; w < SCAN_THREADS / 32; ++w) r = max(r, warp_max[w]);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(SCAN_THREADS) prefill_scan_kernel(const int32_t *seq_lens, const int32_t *num_cached,
                                                                    const int32_t *num_scheduled, int num_seqs,
                                                                    int32_t *cu_q, int32_t *cu_k, int32_t *max_seqlens,
                                                                    int32_t *status)
{
    pa::grid_dependency_wait();  // launched programmatically: the counts may come from the kernel before
    pa::grid_dependents_launch();
    __shared__ int64_t sums[32];
    __shared__ int maxes[32];
    __shared__ int64_t last[2];
    int64_t carry_q = 0, carry_k = 0;
    int mq = 0, mk = 0;
    if (threadIdx.x == 0) cu_q[0] = cu_k[0] = 0;
    for (int base = 0; base < num_seqs; base += SCAN_THREADS) {
        const int b = base + int(threadIdx.x);
        SeqCounts c{0, 0, 0, true};
        if (b < num_seqs) {
            c = counts(seq_lens, num_cached, num_scheduled, b);
            if (!c.ok) pa::report(status, PA_ERR_INVALID_ARG);
        }
        const int64_t sq = block_scan(c.q, sums) + carry_q;
        const int64_t sk = block_scan(c.k, sums) + carry_k;
        if (b < num_seqs) {
            if (sk > 0x7fffffff) pa::report(status, PA_ERR_BOUNDS);
            cu_q[b + 1] = int32_t(sq);
            cu_k[b + 1] = int32_t(sk);
        }
        mq = max(mq, block_max(c.q, maxes));
        mk = max(mk, block_max(c.k, maxes));
        // the last thread's inclusive sums are the carries of the next chunk
        if (threadIdx.x == SCAN_THREADS - 1) last[0] = sq, last[1] = sk;
        __syncthreads();
        carry_q = last[0];
        carry_k = last[1];
        __syncthreads();
    }
    if (threadIdx.x == 0) max_seqlens[0] = mq, max_seqlens[1] = mk;
}

__global__ void __launch_bounds__(256) prefill_expand_kernel(const int32_t *seq_lens, const int32_t *num_cached,
                                                             const int32_t *num_scheduled, int num_seqs,
                                                             const int32_t *block_table, int max_blocks,
                                                             int block_size, int64_t num_blocks, const int32_t *cu_q,
                                                             int32_t *positions, int32_t *slot_mapping,
                                                             int64_t max_tokens, int32_t *status)
{
    pa::grid_dependency_wait();  // cu_seqlens_q from the scan
    for (int b = blockIdx.x; b < num_seqs; b += gridDim.x) {
        const SeqCounts c = counts(seq_lens, num_cached, num_scheduled, b);
        const int64_t offset = cu_q[b];
        const int32_t *table = block_table + int64_t(b) * max_blocks;
        for (int i = threadIdx.x; i < c.q; i += blockDim.x) {
            const int64_t tok = offset + i;
            if (tok >= max_tokens) {
                pa::report(status, PA_ERR_BOUNDS);
                break;
            }
            const int pos = c.start + i;
            const int blk = pos / block_size;
            const int32_t id = blk < max_blocks ? table[blk] : -1;
            const bool ok = id >= 0 && id < num_blocks;
            if (!ok) pa::report(status, PA_ERR_BOUNDS);
            positions[tok] = pos;
            slot_mapping[tok] = ok ? int32_t(int64_t(id) * block_size + pos % block_size) : -1;
        }
    }
}

__global__ void __launch_bounds__(256) decode_meta_kernel(const int32_t *seq_lens, int num_seqs,
                                                          const int32_t *block_table, int max_blocks, int block_size,
                                                          int64_t num_blocks, int32_t *positions, int32_t *context_lens,
                                                          int32_t *slot_mapping, int32_t *status)
{
    pa::grid_dependency_wait();  // launched programmatically
    for (int b = blockIdx.x * blockDim.x + threadIdx.x; b < num_seqs; b += gridDim.x * blockDim.x) {
        const int len = seq_lens[b];
        if (len <= 0) {  // padding row
            if (len < 0) pa::report(status, PA_ERR_INVALID_ARG);
            positions[b] = 0;
            context_lens[b] = 0;
            slot_mapping[b] = -1;
            continue;
        }
        const int pos = len - 1, blk = pos / block_size;
        const int32_t id = blk < max_blocks ? block_table[int64_t(b) * max_blocks + blk] : -1;
        const bool ok = id >= 0 && id < num_blocks;
        if (!ok) pa::report(status, PA_ERR_BOUNDS);
        positions[b] = pos;
        context_lens[b] = len;
        slot_mapping[b] = ok ? int32_t(int64_t(id) * block_size + pos % block_size) : -1;
    }
}

bool metadata_shape_ok(int max_blocks, int block_size, int64_t num_blocks)
{
    return max_blocks >= 1 && block_size >= 1 && num_blocks >= 1 && num_blocks * block_size < (int64_t(1) << 31);
}

}  // namespace

extern "C" pa_status pa_prepare_prefill(const int32_t *seq_lens, const int32_t *num_cached,
                                        const int32_t *num_scheduled, int num_seqs, const int32_t *block_table,
                                        int max_blocks, int block_size, int64_t num_blocks, int32_t *cu_seqlens_q,
                                        int32_t *cu_seqlens_k, int32_t *positions, int32_t *slot_mapping,
                                        int64_t max_tokens, int32_t *max_seqlens, int32_t *dev_status, void *stream)
{
    if (num_seqs < 0 || max_tokens < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!seq_lens || !num_cached || !num_scheduled || !block_table || !cu_seqlens_q || !cu_seqlens_k ||
        !max_seqlens || (max_tokens > 0 && (!positions || !slot_mapping)))
        return PA_ERR_INVALID_ARG;
    if (!metadata_shape_ok(max_blocks, block_size, num_blocks)) return PA_ERR_INVALID_ARG;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    pa::launch_pdl(prefill_scan_kernel, dim3(1), dim3(SCAN_THREADS), 0, s, seq_lens, num_cached, num_scheduled,
                   num_seqs, cu_seqlens_q, cu_seqlens_k, max_seqlens, dev_status);
    const int sms = pa::num_sms() > 0 ? pa::num_sms() : 148;
    const int grid = num_seqs < sms * 8 ? num_seqs : sms * 8;
    pa::launch_pdl(prefill_expand_kernel, dim3(grid), dim3(256), 0, s, seq_lens, num_cached, num_scheduled, num_seqs,
                   block_table, max_blocks, block_size, num_blocks, static_cast<const int32_t *>(cu_seqlens_q),
                   positions, slot_mapping, max_tokens, dev_status);
    return pa::launch_status();
}

extern "C" pa_status pa_prepare_decode(const int32_t *seq_lens, int num_seqs, const int32_t *block_table,
                                       int max_blocks, int block_size, int64_t num_blocks, int32_t *positions,
                                       int32_t *context_lens, int32_t *slot_mapping, int32_t *dev_status,
                                       void *stream)
{
    if (num_seqs < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!seq_lens || !block_table || !positions || !context_lens || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (!metadata_shape_ok(max_blocks, block_size, num_blocks)) return PA_ERR_INVALID_ARG;
    const int grid = (num_seqs + 255) / 256;
    pa::launch_pdl(decode_meta_kernel, dim3(grid < 1024 ? grid : 1024), dim3(256), 0, static_cast<cudaStream_t>(stream),
                   seq_lens, num_seqs, block_table, max_blocks, block_size, num_blocks, positions, context_lens,
                   slot_mapping, dev_status);
    return pa::launch_status();
}
