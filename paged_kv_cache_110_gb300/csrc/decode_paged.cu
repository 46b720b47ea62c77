// decode_paged.cu -- split-KV paged decode: one query token per sequence over
// its paged history, grouped by KV head.
//
// What it computes ("大模型推理入门与 nano-vLLM 源码详解" §9.5, §11.4, §19.6):
// for sequence b with ctx = context_lens[b] keys and query head h reading
// KV head g = h / G (G = Hq / Hkv),
//     s_j = scale * q_h . k_j,  out_h = sum_j softmax(s)_j v_j,  j < ctx,
// where key j lives in pool row block_table[b][j / bs] * bs + j % bs.
// The keys are cut into "splits"; each split keeps (max, exponent sum,
// unnormalised numerator) and the splits are merged with the same
// statistics, never normalised page by page (§9.5, the 2-and-6 example).
//
// Layout of the work (GB300 design, not the pages'):
//  * CTA = (sequence, split), 8 warps.  Warp w serves KV head w % Hkv and
//    every (8 / Hkv)-th 16-token chunk of the split, so each K/V byte of the
//    split is read from HBM exactly once and all G query heads of the group
//    use it (the pages' Triton kernel re-read K/V once per query head).
//  * Within a warp, lanes 0-15 and 16-31 each take one token row of 256 B
//    per 16-byte load (lane c holds dims 8c..8c+7), so one warp load moves
//    two full 256-byte rows.
//  * Scores: each lane forms 8 tokens x G heads partial dot products over
//    its 8 dims, then a transposing butterfly over the 16 lanes of its half
//    (shuffle masks 8, 4, 2, 1 that halve the live values each step) leaves
//    each lane with whole dot products, 8G values for the cost of about 8G
//    shuffles instead of 32G.
//  * Online softmax in base 2 (scale folded with log2 e), per chunk.
//  * Splits with more than one part write fp32 partials to the workspace and
//    a small merge kernel combines them; a single-split sequence is
//    finalised in place.
#include <cuda_fp16.h>
#include <cuda_fp8.h>

#include <mutex>

#include "pa_common.cuh"
#include "sm100_ptx.cuh"

namespace {

constexpr int D = pa::kHeadDim;
constexpr int NW = 8;          // warps per CTA
constexpr int CHUNK = 16;      // tokens per warp iteration (8 per half-warp)
constexpr int PREFETCH_CHUNKS = 1;  // how many of a warp's chunks ahead to prefetch into L2
constexpr int PREFETCH_CHUNKS_FP8 = 1;  // the same for fp8 pools (half the bytes per chunk)
constexpr unsigned FULL = 0xffffffffu;
constexpr float LOG2E = 1.4426950408889634f;

struct DecodeParams {
    const uint16_t *q;
    int64_t q_stride;
    const void *k_cache;  // bf16, or E4M3 codes (fp8 pools)
    const void *v_cache;
    int64_t num_blocks;
    int block_size;
    const int32_t *block_table;
    int max_blocks;
    const int32_t *context_lens;
    int num_seqs;
    int max_ctx;
    int num_heads;
    int kv_heads;
    float scale_log2;   // scale * log2(e) (times the K scale for fp8 pools)
    float out_scale;    // 1, or the V scale times 2^8 for fp8 pools (their values enter the MMAs times 2^-8)
    uint16_t *out;
    const uint16_t *k_new;  // fused KV write: the step's new K / V rows [num_seqs][kv_heads][D], or null
    const uint16_t *v_new;
    int64_t kv_new_stride;  // elements between sequences' rows of k_new / v_new
    // head norm + RoPE of the step's new token (q, and k_new before it is stored), or cos_sin == null
    const float *cos_sin;   // [max_positions][D]: cos of the 64 pairs, then sin
    int64_t max_positions;
    const uint16_t *q_weight, *k_weight;  // [D] bf16, or null: no norm
    float eps;
    float *ws_o;      // [num_seqs][max_splits][num_heads][D]
    float2 *ws_ml;    // [num_seqs][max_splits][num_heads] (max, sum), base-2
    int split_len;
    int max_splits;
    int32_t *status;
    // 128, the factor that moves a permuted E4M3 code into f16 position (a
    // multiply read from the parameters issues on the FMA pipe; a shift by a
    // constant would load the ALU pipe, the busiest of the fp8 decode)
    uint32_t code_mul;
};

struct Plan {
    int split_len;
    int max_splits;
};

// CTAs per SM the split plan aims at: bf16 pools, and fp8 pools, whose tokens
// carry half the bytes, so that a split's fixed work (its query, its partial
// and its share of the merge) weighs twice as much (measured on 512 x U[1k,
// 4k] contexts: 470 us per fp8 call at 16, 473 at 32, 487 at 64).  Fewer CTAs
// per SM never give more splits, so the workspace size pa_decode_workspace_bytes
// returns (the bf16 plan) covers the fp8 plan too.
constexpr int PLAN_CTAS_PER_SM = 64;
constexpr int PLAN_CTAS_PER_SM_FP8 = 16;

Plan make_plan(int num_seqs, int max_ctx, int num_heads, int ctas_per_sm = PLAN_CTAS_PER_SM)
{
    Plan p{CHUNK, 0};
    if (num_seqs <= 0 || max_ctx <= 0) return p;
    // Many CTAs keep enough loads in flight (about 64 per SM measured best for
    // long contexts over bf16 pools), but a split shorter than 128 tokens costs
    // more in fixed work and partials than it gains (measured on 1k contexts),
    // and shorter than 256 from 32 query heads on, whose partials and merge
    // grow with the head count (measured: 64 q heads over 8 KV heads 5%
    // faster).  The plan depends only on the call's arguments and the device's
    // SM count.
    const int sms = pa::num_sms() > 0 ? pa::num_sms() : 152;
    const long long target_ctas = (long long)ctas_per_sm * sms;
    long long per_seq = (target_ctas + num_seqs - 1) / num_seqs;
    if (per_seq < 1) per_seq = 1;
    long long len = (max_ctx + per_seq - 1) / per_seq;
    len = (len + 63) / 64 * 64;
    const int min_split = num_heads >= 32 ? 256 : 128;
    int split = int(len < min_split ? min_split : len);
    split = (split + CHUNK - 1) / CHUNK * CHUNK;
    p.split_len = split;
    p.max_splits = (max_ctx + split - 1) / split;
    return p;
}

size_t workspace_bytes(int num_seqs, int num_heads, const Plan &p)
{
    if (p.max_splits <= 1) return 0;
    const size_t n = size_t(num_seqs) * p.max_splits * num_heads;
    const size_t o_bytes = (n * D * sizeof(float) + 255) / 256 * 256;
    return o_bytes + n * sizeof(float2);
}

__device__ __forceinline__ void unpack8(const uint4 &u, float (&f)[8])
{
    f[0] = pa::bf16_lo(u.x); f[1] = pa::bf16_hi(u.x);
    f[2] = pa::bf16_lo(u.y); f[3] = pa::bf16_hi(u.y);
    f[4] = pa::bf16_lo(u.z); f[5] = pa::bf16_hi(u.z);
    f[6] = pa::bf16_lo(u.w); f[7] = pa::bf16_hi(u.w);
}

// A bf16 pool row piece: 8 elements (16 bytes) per lane load.
struct KvRow {
    using Raw = uint4;
    using Elem = uint16_t;
    static __device__ __forceinline__ Raw load(const Elem *p) { return pa::ld_stream16(p); }
    static __device__ __forceinline__ Raw load_l2(const Elem *p) { return __ldcg(reinterpret_cast<const uint4 *>(p)); }
    static __device__ __forceinline__ Raw zero() { return make_uint4(0, 0, 0, 0); }
};

// RMSNorm (when `norm`: v = bf16(bf16(v / rms) * w), w = 1 without a weight)
// and RoPE of one head row of the step's new token, held as 8 features per
// lane by the 16 lanes of a half-warp (lane c: features 8c .. 8c+7).  Feature
// i pairs with feature i + 64, which sits in lane c ^ 8: (a, b) ->
// (a cos - b sin, a sin + b cos) in fp32, rounded to bf16 ("nano-vllm 技术分析"
// §4.3-4.4; "大模型推理入门与 nano-vLLM 源码详解" §19.3, §19.7).  The steps
// and their roundings are those of the fused norm + RoPE + KV write.  Every
// lane of the warp calls this with the same `norm` (the sum of squares is
// reduced over the half-warp and the partners exchanged by shuffles).
__device__ __forceinline__ void norm_rope_row8(float (&x)[8], int c, bool norm, const float (&wv)[8], float eps,
                                               const float (&cv)[8], const float (&sv)[8])
{
    if (norm) {
        float ss = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) ss = fmaf(x[e], x[e], ss);
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
        const float r = 1.0f / sqrtf(ss * (1.0f / D) + eps);
#pragma unroll
        for (int e = 0; e < 8; e += 2) {
            const uint32_t t = pa::pack_bf16x2(x[e] * r, x[e + 1] * r);
            const uint32_t u = pa::pack_bf16x2(pa::bf16_lo(t) * wv[e], pa::bf16_hi(t) * wv[e + 1]);
            x[e] = pa::bf16_lo(u);
            x[e + 1] = pa::bf16_hi(u);
        }
    }
    float y[8];
#pragma unroll
    for (int e = 0; e < 8; ++e) y[e] = __shfl_xor_sync(FULL, x[e], 8);
    float out[8];
#pragma unroll
    for (int e = 0; e < 8; ++e)
        out[e] = (c < 8) ? fmaf(x[e], cv[e], -y[e] * sv[e])   // a' = a cos - b sin (x = a, y = b)
                         : fmaf(y[e], sv[e], x[e] * cv[e]);   // b' = a sin + b cos (y = a, x = b)
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const uint32_t u = pa::pack_bf16x2(out[e], out[e + 1]);
        x[e] = pa::bf16_lo(u);
        x[e + 1] = pa::bf16_hi(u);
    }
}

// The norm weight (8 features of lane c, 1 without a weight) and the cos / sin
// of lane c's 8 pairs at one position (row cs of the table).
struct RopeLane {
    float w[8], c[8], s[8];
};
__device__ __forceinline__ RopeLane rope_lane(const uint16_t *w, const float *cs, int c)
{
    RopeLane r;
    if (w != nullptr) {
        unpack8(*reinterpret_cast<const uint4 *>(w + 8 * c), r.w);
    } else {
#pragma unroll
        for (int e = 0; e < 8; ++e) r.w[e] = 1.f;
    }
    const float4 *cp = reinterpret_cast<const float4 *>(cs + 8 * (c & 7));
    const float4 *sp = reinterpret_cast<const float4 *>(cs + D / 2 + 8 * (c & 7));
    const float4 c0 = cp[0], c1 = cp[1], s0 = sp[0], s1 = sp[1];
    r.c[0] = c0.x; r.c[1] = c0.y; r.c[2] = c0.z; r.c[3] = c0.w; r.c[4] = c1.x; r.c[5] = c1.y; r.c[6] = c1.z; r.c[7] = c1.w;
    r.s[0] = s0.x; r.s[1] = s0.y; r.s[2] = s0.z; r.s[3] = s0.w; r.s[4] = s1.x; r.s[5] = s1.y; r.s[6] = s1.z; r.s[7] = s1.w;
    return r;
}

__device__ __forceinline__ uint4 pack8(const float (&f)[8])
{
    return make_uint4(pa::pack_bf16x2(f[0], f[1]), pa::pack_bf16x2(f[2], f[3]), pa::pack_bf16x2(f[4], f[5]),
                      pa::pack_bf16x2(f[6], f[7]));
}

// One transposing butterfly step over the 16 lanes of a half-warp: lanes
// whose bit M is set keep the upper half of x, the others the lower half,
// and each adds its partner's copy of the half it keeps.  With N == 1 it is
// a plain butterfly sum.
template <int N, int M>
__device__ __forceinline__ void xpose_step(float (&x)[8 * 8], int c)
{
    if constexpr (N >= 2) {
        const bool upper = (c & M) != 0;
#pragma unroll
        for (int j = 0; j < N / 2; ++j) {
            const float send = upper ? x[j] : x[j + N / 2];
            const float keep = upper ? x[j + N / 2] : x[j];
            x[j] = keep + __shfl_xor_sync(FULL, send, M);
        }
    } else {
        x[0] += __shfl_xor_sync(FULL, x[0], M);
    }
}

// Max / sum over the 16 lanes that share lane bit 0 (xor 2, 4, 8, 16).
__device__ __forceinline__ float group_max(float v)
{
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) v = fmaxf(v, __shfl_xor_sync(FULL, v, m));
    return v;
}
__device__ __forceinline__ float group_sum(float v)
{
#pragma unroll
    for (int m = 2; m <= 16; m <<= 1) v += __shfl_xor_sync(FULL, v, m);
    return v;
}

// Before a decode CTA waits on the previous kernel: bring the first chunk
// (16 rows of every KV head) of each of its warp groups into L2, so that the
// first loads after the wait find them there.  The context length and the
// block id read here may still be written by the previous kernel (the kernel
// reads both again after the wait); validated, they serve only as the address
// of an L2 prefetch, which changes no result.  cluster_parts > 0: the
// sequence is cut into that many equal parts, else into the call's splits.
__device__ __forceinline__ void prefetch_first_chunks(const DecodeParams &p, int elem_bytes, int cluster_parts)
{
    const int warp = threadIdx.x >> 5;
    if ((threadIdx.x & 31) != 0 || warp % p.kv_heads != 0) return;
    const int b = blockIdx.x, s = blockIdx.y;
    const int ctx = p.context_lens[b];
    if (ctx <= 0 || ctx > p.max_ctx || int64_t(ctx) > int64_t(p.max_blocks) * p.block_size) return;
    const int split_len = cluster_parts > 0
                              ? ((ctx + cluster_parts - 1) / cluster_parts + CHUNK - 1) / CHUNK * CHUNK
                              : p.split_len;
    const int t0 = s * split_len, t1 = min(ctx, t0 + split_len);
    const int cf = t0 + (warp / p.kv_heads) * CHUNK;
    if (cf >= t1) return;
    const int32_t pf = p.block_table[int64_t(b) * p.max_blocks + cf / p.block_size];
    if (pf < 0 || int64_t(pf) >= p.num_blocks) return;
    const int64_t row_bytes = int64_t(p.kv_heads) * D * elem_bytes;
    const int64_t off = (int64_t(pf) * p.block_size + cf % p.block_size) * row_bytes;
    const uint32_t bytes = uint32_t(min(CHUNK, t1 - cf) * row_bytes);  // (a multiple of 128)
    pa::sm100::prefetch_l2_bulk(static_cast<const char *>(p.k_cache) + off, bytes);
    pa::sm100::prefetch_l2_bulk(static_cast<const char *>(p.v_cache) + off, bytes);
}

template <int G, bool ROPE, bool CLUSTER>
__global__ void __launch_bounds__(NW * 32, 2) decode_split_kernel(const DecodeParams p)
{
    using KV = KvRow;
    constexpr int V = 8 * G;                 // partial dot products per lane per chunk
    constexpr int R = V >= 16 ? V / 16 : 1;  // whole dot products per lane after the butterfly
    const int b = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int half = lane >> 4, c = lane & 15;
    if constexpr (!CLUSTER) prefetch_first_chunks(p, int(sizeof(typename KV::Elem)), 0);
    // launched programmatically: everything below may depend on the previous
    // kernel (the KV write of this step's token)
    pa::grid_dependency_wait();

    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_ctx || int64_t(ctx) > int64_t(p.max_blocks) * p.block_size ||
        (ROPE && int64_t(ctx) > p.max_positions)) {
        if (s == 0 && threadIdx.x == 0) pa::report(p.status, PA_ERR_BOUNDS);
        ctx = 0;
    }
    if (ctx == 0) {  // padded row: output zeros, read nothing
        if (s == 0) {
            uint4 *o = reinterpret_cast<uint4 *>(p.out + int64_t(b) * p.num_heads * D);
            for (int i = threadIdx.x; i < p.num_heads * D / 8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    // In a cluster the sequence's keys are cut into as many equal splits (whole
    // 16-token chunks) as the cluster has CTAs, so that its CTAs finish
    // together; otherwise every sequence uses the call's split length.
    const int split_len = CLUSTER ? ((ctx + int(gridDim.y) - 1) / int(gridDim.y) + CHUNK - 1) / CHUNK * CHUNK
                                  : p.split_len;
    const int nsplit = (ctx + split_len - 1) / split_len;
    // (in a cluster every CTA stays to the end: it takes part in the merge's
    // barriers; a CTA past the sequence's splits reads nothing)
    if (!CLUSTER && s >= nsplit) return;

    const int g = warp % p.kv_heads;
    const int sub = warp / p.kv_heads;
    const int wph = NW / p.kv_heads;
    const int t0 = s * split_len;
    const int t1 = min(ctx, t0 + split_len);
    const int64_t row_elems = int64_t(p.kv_heads) * D;
    const int32_t *table = p.block_table + int64_t(b) * p.max_blocks;

    // Fused KV write (bf16 pools): the sequence's last split stores the step's new
    // token, position ctx - 1, at its pool row (warp g: head g, lanes 0-15 K,
    // 16-31 V) before any of its warps reads.  Only this CTA reads that row in
    // this launch, after the barrier below, and the chunk that holds it is read
    // through L2 (ld.global.cg), not the read-only path the other chunks use.
    int new_tok = -1;  // position written by this launch, or -1
    {
        if (p.k_new != nullptr && s == nsplit - 1) {  // the same for the whole CTA
            new_tok = ctx - 1;
            if (sub == 0) {
                const int32_t phys = table[new_tok / p.block_size];
                const uint16_t *src = (half ? p.v_new : p.k_new) + int64_t(b) * p.kv_new_stride + g * D + 8 * c;
                uint4 u = *reinterpret_cast<const uint4 *>(src);
                if constexpr (ROPE) {
                    // K (lanes 0-15) normalised and rotated before it is stored; the V
                    // lanes take part in the shuffles and store their row unchanged
                    const RopeLane rl = rope_lane(p.k_weight, p.cos_sin + int64_t(new_tok) * D, c);
                    float x[8];
                    unpack8(u, x);
                    norm_rope_row8(x, c, p.k_weight != nullptr, rl.w, p.eps, rl.c, rl.s);
                    if (!half) u = pack8(x);
                }
                if (phys >= 0 && int64_t(phys) < p.num_blocks) {
                    const int64_t row = int64_t(phys) * p.block_size + new_tok % p.block_size;
                    uint16_t *dst = static_cast<uint16_t *>(const_cast<void *>(half ? p.v_cache : p.k_cache)) +
                                    row * row_elems + g * D + 8 * c;
                    *reinterpret_cast<uint4 *>(dst) = u;
                }
                // an invalid block id is reported by the loop below, which skips that chunk
            }
            __syncthreads();
        }
    }

    // (a cluster's CTAs prefetch after the wait: measured 0.4% faster on long contexts)
    if constexpr (CLUSTER) prefetch_first_chunks(p, int(sizeof(typename KV::Elem)), int(gridDim.y));
    float qf[G][8];
    {
        uint4 qr[G];
#pragma unroll
        for (int h = 0; h < G; ++h)
            qr[h] = *reinterpret_cast<const uint4 *>(p.q + int64_t(b) * p.q_stride + (g * G + h) * D + 8 * c);
        RopeLane rl;
        // every split rotates the query itself (a few hundred flops); its weight
        // and cos / sin are loaded together with the row: one round trip
        if constexpr (ROPE) rl = rope_lane(p.q_weight, p.cos_sin + int64_t(ctx - 1) * D, c);
#pragma unroll
        for (int h = 0; h < G; ++h) {
            unpack8(qr[h], qf[h]);
            if constexpr (ROPE) norm_rope_row8(qf[h], c, p.q_weight != nullptr, rl.w, p.eps, rl.c, rl.s);
#pragma unroll
            for (int e = 0; e < 8; ++e) qf[h][e] *= p.scale_log2;
        }
    }
    float o[G][8];
    float m[G], l[G];
#pragma unroll
    for (int h = 0; h < G; ++h) {
        m[h] = -INFINITY;
        l[h] = 0.f;
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] = 0.f;
    }

    for (int cb = t0 + sub * CHUNK; cb < t1; cb += wph * CHUNK) {
        const int32_t phys = table[cb / p.block_size];
        if (phys < 0 || int64_t(phys) >= p.num_blocks) {
            if (lane == 0) pa::report(p.status, PA_ERR_BOUNDS);
            continue;
        }
        // a chunk never crosses a block: cb and block_size are multiples of 16
        const int64_t row0 = int64_t(phys) * p.block_size + (cb % p.block_size) + half * 8;
        const typename KV::Elem *kp = static_cast<const typename KV::Elem *>(p.k_cache) + row0 * row_elems + g * D + 8 * c;
        const typename KV::Elem *vp = static_cast<const typename KV::Elem *>(p.v_cache) + row0 * row_elems + g * D + 8 * c;
        const int nvalid = t1 - (cb + half * 8);  // tokens of this half inside the split
        if (PREFETCH_CHUNKS > 0 && g == 0 && lane == 0) {
            // bring a later chunk of this warp's sequence of chunks into L2: its
            // 16 token rows of all KV heads are one contiguous run of one block
            const int cn = cb + PREFETCH_CHUNKS * wph * CHUNK;
            if (cn < t1) {
                const int32_t pn = table[cn / p.block_size];
                if (pn >= 0 && int64_t(pn) < p.num_blocks) {
                    const int64_t r = (int64_t(pn) * p.block_size + cn % p.block_size) * row_elems;
                    const uint32_t bytes = uint32_t(min(CHUNK, t1 - cn) * row_elems * sizeof(typename KV::Elem));
                    const uint32_t b16 = (bytes + 15u) & ~15u;
                    pa::sm100::prefetch_l2_bulk(static_cast<const typename KV::Elem *>(p.k_cache) + r, b16);
                    pa::sm100::prefetch_l2_bulk(static_cast<const typename KV::Elem *>(p.v_cache) + r, b16);
                }
            }
        }

        typename KV::Raw kr[8], vr[8];
        if (unsigned(new_tok - cb) < unsigned(CHUNK)) {
            // the chunk holding the row this launch wrote: coherent loads through L2
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < nvalid) {
                    kr[i] = KV::load_l2(kp + i * row_elems);
                    vr[i] = KV::load_l2(vp + i * row_elems);
                } else {
                    kr[i] = KV::zero();
                    vr[i] = KV::zero();
                }
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (i < nvalid) {
                    kr[i] = KV::load(kp + i * row_elems);
                    vr[i] = KV::load(vp + i * row_elems);
                } else {
                    kr[i] = KV::zero();
                    vr[i] = KV::zero();
                }
            }
        }

        // partial dot products over this lane's 8 dims: x[i * G + h]
        float x[8 * 8];
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float kf[8];
            unpack8(kr[i], kf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 8; ++e) acc = fmaf(qf[h][e], kf[e], acc);
                x[i * G + h] = acc;
            }
        }
        xpose_step<V, 8>(x, c);
        xpose_step<V / 2, 4>(x, c);
        xpose_step<V / 4, 2>(x, c);
        xpose_step<V / 8, 1>(x, c);
        // lane c now holds token i = c >> 1 of its half; register r is head
        // (c & 1) * R + r (G >= 2) or head 0 (G == 1).
        const bool tok_ok = (c >> 1) < nvalid;
        float sc[R], mx[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            sc[r] = tok_ok ? x[r] : -INFINITY;
            mx[r] = group_max(sc[r]);
        }
        float m_new[G], alpha[G];
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float mc = (G == 1) ? mx[0] : __shfl_sync(FULL, mx[h % R], h / R);
            m_new[h] = fmaxf(m[h], mc);
            alpha[h] = exp2f(m[h] - m_new[h]);
        }
        float pr[R], ps[R];
#pragma unroll
        for (int r = 0; r < R; ++r) {
            const float mh = (G == 1) ? m_new[0] : ((c & 1) ? m_new[(R + r) % G] : m_new[r % G]);
            pr[r] = exp2f(sc[r] - mh);
            ps[r] = group_sum(pr[r]);
        }
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float sum = (G == 1) ? ps[0] : __shfl_sync(FULL, ps[h % R], h / R);
            l[h] = alpha[h] * l[h] + sum;
            m[h] = m_new[h];
#pragma unroll
            for (int e = 0; e < 8; ++e) o[h][e] *= alpha[h];
        }
#pragma unroll
        for (int i = 0; i < 8; ++i) {
            float vf[8];
            unpack8(vr[i], vf);
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const int idx = i * G + h;
                const int src_c = (G == 1) ? 2 * i : idx / R;
                const float pv = __shfl_sync(FULL, pr[(G == 1) ? 0 : idx % R], src_c, 16);
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] = fmaf(pv, vf[e], o[h][e]);
            }
        }
    }

    // this CTA's loads are done: the next kernel (the merge) may start launching
    pa::grid_dependents_launch();

    // the two halves saw different tokens of the same chunks: add them
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
        for (int e = 0; e < 8; ++e) o[h][e] += __shfl_xor_sync(FULL, o[h][e], 16);

    // warps that shared one KV head (Hkv < 8) merge through shared memory
    __shared__ __align__(16) float red_o[NW][G][D];
    __shared__ __align__(16) float red_ml[NW][G][2];
    if (wph > 1) {
        if (lane < 16) {
#pragma unroll
            for (int h = 0; h < G; ++h)
#pragma unroll
                for (int e = 0; e < 8; ++e) red_o[warp][h][8 * c + e] = o[h][e];
        }
        if (lane == 0) {
#pragma unroll
            for (int h = 0; h < G; ++h) {
                red_ml[warp][h][0] = m[h];
                red_ml[warp][h][1] = l[h];
            }
        }
        __syncthreads();
        if (!CLUSTER && sub != 0) return;
#pragma unroll
        for (int h = 0; h < G; ++h) {
            if (sub != 0) break;
            float mm = m[h];
            for (int w = 1; w < wph; ++w) mm = fmaxf(mm, red_ml[g + w * p.kv_heads][h][0]);
            const float a0 = exp2f(m[h] - mm);
            float ll = l[h] * a0;
#pragma unroll
            for (int e = 0; e < 8; ++e) o[h][e] *= a0;
            for (int w = 1; w < wph; ++w) {
                const int ww = g + w * p.kv_heads;
                const float mw = red_ml[ww][h][0];
                const float aw = (mw == -INFINITY) ? 0.f : exp2f(mw - mm);
                ll += red_ml[ww][h][1] * aw;
#pragma unroll
                for (int e = 0; e < 8; ++e) o[h][e] = fmaf(red_o[ww][h][8 * c + e], aw, o[h][e]);
            }
            m[h] = mm;
            l[h] = ll;
        }
    }

    if constexpr (CLUSTER) {
        // The splits of this sequence are the CTAs of one cluster (its rank = s).
        // Each leaves its partial (max, sum, unnormalised O of every head of the
        // sequence) in its own shared memory, in red_o / red_ml's space: head row
        // g * G + h is the row warp g's own partial occupied, and the other
        // warps' rows it read lie past num_heads, so no warp overwrites a row
        // another still reads.  After a cluster barrier, CTA s merges heads
        // s, s + nsplit, ... reading every split's partial through distributed
        // shared memory (the same rule as the merge kernel), and a second
        // barrier keeps every CTA's shared memory alive until all have read it.
        // Every thread of every CTA reaches both barriers.
        float *xo = &red_o[0][0][0];                                  // [num_heads][D]
        float2 *xm = reinterpret_cast<float2 *>(&red_ml[0][0][0]);   // [num_heads]
        const bool lead = sub == 0 && lane < 16;
        __syncwarp();  // (the merge above read this warp's rows of red_ml)
        if (lead && s < nsplit) {  // (a CTA past the sequence's splits holds no partial)
#pragma unroll
            for (int h = 0; h < G; ++h) {
                const int hr = g * G + h;
                if (nsplit == 1) {
                    const float inv = p.out_scale / l[h];
                    uint4 u;
                    u.x = pa::pack_bf16x2(o[h][0] * inv, o[h][1] * inv);
                    u.y = pa::pack_bf16x2(o[h][2] * inv, o[h][3] * inv);
                    u.z = pa::pack_bf16x2(o[h][4] * inv, o[h][5] * inv);
                    u.w = pa::pack_bf16x2(o[h][6] * inv, o[h][7] * inv);
                    *reinterpret_cast<uint4 *>(p.out + (int64_t(b) * p.num_heads + hr) * D + 8 * c) = u;
                } else {
                    float4 *dst = reinterpret_cast<float4 *>(xo + hr * D + 8 * c);
                    dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
                    dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
                    if (c == 0) xm[hr] = make_float2(m[h], l[h]);
                }
            }
        }
        pa::sm100::cluster_sync();
        if (nsplit > 1 && s < nsplit) {
            const int mine = (p.num_heads - s + nsplit - 1) / nsplit;  // heads s, s + nsplit, ...
            for (int it = threadIdx.x; it < mine * 16; it += NW * 32) {
                const int h = s + (it >> 4) * nsplit, c8 = (it & 15) * 8;
                const uint32_t ao = pa::sm100::smem_u32(xo + h * D + c8), am = pa::sm100::smem_u32(xm + h);
                float2 ml[NW];
                float4 x0[NW], x1[NW];
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    if (j < nsplit) {
                        ml[j] = pa::sm100::ld_shared_cluster_v2(pa::sm100::mapa_shared(am, j));
                        x0[j] = pa::sm100::ld_shared_cluster_v4(pa::sm100::mapa_shared(ao, j));
                        x1[j] = pa::sm100::ld_shared_cluster_v4(pa::sm100::mapa_shared(ao + 16, j));
                    } else {
                        ml[j] = make_float2(-INFINITY, 0.f);
                        x0[j] = x1[j] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
                float mm = -INFINITY;
#pragma unroll
                for (int j = 0; j < NW; ++j) mm = fmaxf(mm, ml[j].x);
                float ll = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int j = 0; j < NW; ++j) {
                    const float w = (ml[j].x == -INFINITY) ? 0.f : exp2f(ml[j].x - mm);
                    ll += ml[j].y * w;
                    acc[0] += x0[j].x * w; acc[1] += x0[j].y * w; acc[2] += x0[j].z * w; acc[3] += x0[j].w * w;
                    acc[4] += x1[j].x * w; acc[5] += x1[j].y * w; acc[6] += x1[j].z * w; acc[7] += x1[j].w * w;
                }
                const float inv = p.out_scale / ll;
                uint4 u;
                u.x = pa::pack_bf16x2(acc[0] * inv, acc[1] * inv);
                u.y = pa::pack_bf16x2(acc[2] * inv, acc[3] * inv);
                u.z = pa::pack_bf16x2(acc[4] * inv, acc[5] * inv);
                u.w = pa::pack_bf16x2(acc[6] * inv, acc[7] * inv);
                *reinterpret_cast<uint4 *>(p.out + (int64_t(b) * p.num_heads + h) * D + c8) = u;
            }
        }
        pa::sm100::cluster_sync();
        return;
    }

    if (lane >= 16) return;
    if (nsplit == 1) {
#pragma unroll
        for (int h = 0; h < G; ++h) {
            const float inv = p.out_scale / l[h];
            uint4 u;
            u.x = pa::pack_bf16x2(o[h][0] * inv, o[h][1] * inv);
            u.y = pa::pack_bf16x2(o[h][2] * inv, o[h][3] * inv);
            u.z = pa::pack_bf16x2(o[h][4] * inv, o[h][5] * inv);
            u.w = pa::pack_bf16x2(o[h][6] * inv, o[h][7] * inv);
            *reinterpret_cast<uint4 *>(p.out + (int64_t(b) * p.num_heads + g * G + h) * D + 8 * c) = u;
        }
        return;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
        const int64_t row = (int64_t(b) * p.max_splits + s) * p.num_heads + g * G + h;
        float4 *dst = reinterpret_cast<float4 *>(p.ws_o + row * D + 8 * c);
        dst[0] = make_float4(o[h][0], o[h][1], o[h][2], o[h][3]);
        dst[1] = make_float4(o[h][4], o[h][5], o[h][6], o[h][7]);
        if (c == 0) p.ws_ml[row] = make_float2(m[h], l[h]);
    }
}

// ---------------------------------------------------------------------------
// Decode over E4M3 pools on the warp-level tensor-core MMA (mma.sync
// m16n8k16: f16 operands, f32 accumulators).
//
// An fp8 pool halves the bytes but not the work per element: every code must
// become an MMA operand, and converting every code to f32 for CUDA-core FMAs
// is the costliest way.  Here the codes become f16 exactly (every E4M3 value
// times 2^-8 is an f16 value), two at a time by a byte permute, a shift and a
// mask, and the dot products and the P.V sums run as MMAs.  The 2^-8 and the
// K scale are folded into the score scale, the 2^-8 and the V scale into the
// output scale.  The work split is the bf16 kernel's: CTA = (sequence, split),
// warp = (KV head, every wph-th 16-token chunk).
// Lane (gq, tq) = (lane / 4, lane % 4).  Per chunk:
//   S^T = K Q^T   A = the keys of the chunk's 16 tokens (f16), 8 steps of 16
//               dims: lane (gq, tq) supplies tokens gq and gq + 8, dims
//               16 tq .. + 15 and 64 + 16 tq .. + 15 (each step takes four of
//               them, one word per token), and the four lanes of a token read
//               adjacent 16-byte pieces; B = the group's G query heads as
//               columns 0..G-1 of 8 (f16, the same dims; each head multiplied
//               by the power of two that puts its largest magnitude in
//               [2^13, 2^14), undone on the fp32 score).  One MMA per step.
//   softmax     the accumulator holds the scores of tokens gq and gq + 8 for
//               heads 2tq and 2tq + 1 (columns past G are zero and unused).
//               The running max of a head, the same in its 8 lanes, moves only
//               when a score passes it by more than 2^8 (log2 units): only
//               then are the 8 lanes' maxima reduced by shuffles and O
//               rescaled; each lane keeps its share of the sum, added up over
//               the 8 lanes at the end.  O / l uses the same max, so the result
//               does not depend on when it moved.
//   O^T += V^T P^T   A = V^T (16 dims x the 16 tokens): lane gq supplies dims
//               16 gq .. 16 gq + 15 of tokens 2tq, 2tq+1, 2tq+8, 2tq+9, two
//               tokens' codes paired by the conversion's byte permute; B = P^T
//               (f16): each 8 x 8 tile of P as the S^T accumulator holds it,
//               transposed by movmatrix; C = O^T, 8 blocks of 16 dims x 8 head
//               columns, heads 2tq and 2tq + 1 in lane (gq, tq) as in S^T.
// Rounding: the products of f16 operands are exact in the f32 accumulators
// (q is a bf16 value times a power of two, exactly an f16 value in the range
// the prescale gives); P (below 2^8) is rounded to f16 (relative 2^-11) for
// the P.V MMA.

// Two E4M3 codes as an f16 pair, each value times 2^-8, exactly.  One byte
// permute takes the two codes (bytes `sel` picks from a and b) into the low
// bytes of the two 16-bit lanes and fills each lane's high byte with copies of
// that code's sign bit (the permute's sign-replicate selectors, bit 3 of a
// selector nibble); a shift left by 7 then puts eeee mmm where an f16 keeps
// the low four exponent bits and the top three mantissa bits, and one copy of
// the sign at bit 15.  The mask clears what else the shift moved in: the code's
// own sign at bit 14 (the top exponent bit, which stays 0) and the low lane's
// other sign copies at the high lane's bits 0-6.  The f16 exponent bias, 15,
// exceeds E4M3's, 7, by 8: the 2^-8; E4M3 subnormals land on f16 subnormals.
// sel: 0x9180 for bytes 0, 1 of a; 0xB3A2 for bytes 2, 3 of a; 0xC480 + 0x1111 i
// for byte i of a and byte i of b.
// mul: 128 (the shift by 7), passed in so that it stays a multiply.
template <uint32_t SEL>
__device__ __forceinline__ uint32_t e4m3x2_to_f16x2(uint32_t a, uint32_t b, uint32_t mul)
{
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "n"(SEL));
    return (r * mul) & 0xbf80bf80u;
}

// Byte k of a and byte k of b as an f16 pair, for k = 2hb and 2hb + 1.
__device__ __forceinline__ void e4m3_byte_pairs(uint32_t a, uint32_t b, int hb, uint32_t (&f)[2], uint32_t mul)
{
    if (hb == 0) {
        f[0] = e4m3x2_to_f16x2<0xC480u>(a, b, mul);
        f[1] = e4m3x2_to_f16x2<0xD591u>(a, b, mul);
    } else {
        f[0] = e4m3x2_to_f16x2<0xE6A2u>(a, b, mul);
        f[1] = e4m3x2_to_f16x2<0xF7B3u>(a, b, mul);
    }
}

// The four E4M3 codes of w as two f16 pairs (codes 0, 1 and codes 2, 3).
__device__ __forceinline__ void e4m3x4_to_f16x2x2(uint32_t w, uint32_t &lo, uint32_t &hi, uint32_t mul)
{
    lo = e4m3x2_to_f16x2<0x9180u>(w, 0u, mul);
    hi = e4m3x2_to_f16x2<0xB3A2u>(w, 0u, mul);
}

__device__ __forceinline__ uint32_t f16x2_of(float lo, float hi)
{
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const uint32_t *>(&h);
}

// d += A (16 x 16, row) * B (16 x 8, col), f16 in, f32 accumulate
__device__ __forceinline__ void mma_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                          uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// The transpose of an 8 x 8 matrix of 16-bit values held as the warp holds an
// MMA fragment (lane 4r + c: row r, columns 2c, 2c + 1).
__device__ __forceinline__ uint32_t movmatrix_trans(uint32_t a)
{
    uint32_t d;
    asm("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;" : "=r"(d) : "r"(a));
    return d;
}

constexpr float FP8_RESCALE_THRESHOLD = 8.0f;  // log2 units

template <int G>
__global__ void __launch_bounds__(NW * 32, 2) decode_fp8_mma_kernel(const DecodeParams p)
{
    const int b = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    pa::grid_dependency_wait();

    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_ctx || int64_t(ctx) > int64_t(p.max_blocks) * p.block_size) {
        if (s == 0 && threadIdx.x == 0) pa::report(p.status, PA_ERR_BOUNDS);
        ctx = 0;
    }
    if (ctx == 0) {  // padded row: output zeros, read nothing
        if (s == 0) {
            uint4 *o = reinterpret_cast<uint4 *>(p.out + int64_t(b) * p.num_heads * D);
            for (int i = threadIdx.x; i < p.num_heads * D / 8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int nsplit = (ctx + p.split_len - 1) / p.split_len;
    if (s >= nsplit) return;

    const int g = warp % p.kv_heads;
    const int sub = warp / p.kv_heads;
    const int wph = NW / p.kv_heads;
    const int t0 = s * p.split_len;
    const int t1 = min(ctx, t0 + p.split_len);
    const int row_elems = p.kv_heads * D;
    const int32_t *table = p.block_table + int64_t(b) * p.max_blocks;
    const uint8_t *kc = static_cast<const uint8_t *>(p.k_cache);
    const uint8_t *vc = static_cast<const uint8_t *>(p.v_cache);

    auto prefetch_chunk = [&](int cf) {  // a chunk's 16 rows of all KV heads: one contiguous run of one block
        if (cf >= t1) return;
        const int32_t pf = table[cf / p.block_size];
        if (pf < 0 || int64_t(pf) >= p.num_blocks) return;
        const int64_t r = (int64_t(pf) * p.block_size + cf % p.block_size) * row_elems;
        const uint32_t bytes = uint32_t(min(CHUNK, t1 - cf) * row_elems);
        const uint32_t b16 = (bytes + 15u) & ~15u;
        pa::sm100::prefetch_l2_bulk(kc + r, b16);
        pa::sm100::prefetch_l2_bulk(vc + r, b16);
    };
    if (g == 0 && lane == 0) prefetch_chunk(t0 + sub * CHUNK);

    // the query: head gq of the group (rows gq >= G stay zero), the lane's key
    // dims 16 tq .. + 15 (x[0..15]) and 64 + 16 tq .. + 15 (x[16..31])
    uint32_t qa[8][2];
    float sscale;  // score scale of head gq in log2 units, the prescale undone
    {
        float x[32];
        if (gq < G) {
            const uint16_t *qrow = p.q + int64_t(b) * p.q_stride + (g * G + gq) * D + 16 * tq;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float f[8];
                unpack8(*reinterpret_cast<const uint4 *>(qrow + 64 * (i >> 1) + 8 * (i & 1)), f);
#pragma unroll
                for (int e = 0; e < 8; ++e) x[8 * i + e] = f[e];
            }
        } else {
#pragma unroll
            for (int e = 0; e < 32; ++e) x[e] = 0.f;
        }
        float mx = 0.f;
#pragma unroll
        for (int e = 0; e < 32; ++e) mx = fmaxf(mx, fabsf(x[e]));
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(FULL, mx, 2));
        int k = 0;
        if (mx > 0.f) k = min(126, max(-126, 13 - (int((__float_as_uint(mx) >> 23) & 0xffu) - 127)));
        const float up = __uint_as_float(uint32_t(127 + k) << 23);    // 2^k
        const float down = __uint_as_float(uint32_t(127 - k) << 23);  // 2^-k
        sscale = p.scale_log2 * down * 256.f;  // (the keys enter the MMA times 2^-8)
#pragma unroll
        for (int st = 0; st < 8; ++st) {
            qa[st][0] = f16x2_of(x[4 * st] * up, x[4 * st + 1] * up);
            qa[st][1] = f16x2_of(x[4 * st + 2] * up, x[4 * st + 3] * up);
        }
    }
    // the score scales of this lane's S^T columns, heads 2tq and 2tq + 1
    const float ss0 = __shfl_sync(FULL, sscale, 8 * tq), ss1 = __shfl_sync(FULL, sscale, 8 * tq + 4);

    // this lane's byte offsets within a chunk's first row of head g: its two
    // 16-byte pieces of a key row lie 64 bytes apart and the four lanes of a
    // token hold adjacent pieces, so each load instruction reads whole 64-byte runs
    const int offk0 = gq * row_elems + g * D + 16 * tq, offk1 = offk0 + 8 * row_elems;
    const int offv = g * D + 16 * gq;

    float o[8][4];  // O^T: block mb holds dims 16 gq + mb (o[mb][0..1]) and 16 gq + 8 + mb (o[mb][2..3])
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;
    // heads 2tq, 2tq + 1: running max (the same in the 8 lanes of a tq) and this
    // lane's share of the sum (its tokens), added up over the 8 lanes at the end
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int cb = t0 + sub * CHUNK; cb < t1; cb += wph * CHUNK) {
        const int32_t phys = table[cb / p.block_size];
        if (phys < 0 || int64_t(phys) >= p.num_blocks) {
            if (lane == 0) pa::report(p.status, PA_ERR_BOUNDS);
            continue;
        }
        // a chunk never crosses a block: cb and block_size are multiples of 16
        const int64_t base = (int64_t(phys) * p.block_size + (cb % p.block_size)) * row_elems;
        const int nvalid = t1 - cb;
        if (PREFETCH_CHUNKS_FP8 > 0 && g == 0 && lane == 0) prefetch_chunk(cb + PREFETCH_CHUNKS_FP8 * wph * CHUNK);

        uint4 kr[2][2], vr[4];
        {
            const uint8_t *k0 = kc + base + offk0, *k1 = kc + base + offk1;
            const bool v0 = gq < nvalid, v1 = 8 + gq < nvalid;
            kr[0][0] = v0 ? pa::ld_stream16(k0) : make_uint4(0, 0, 0, 0);
            kr[0][1] = v0 ? pa::ld_stream16(k0 + 64) : make_uint4(0, 0, 0, 0);
            kr[1][0] = v1 ? pa::ld_stream16(k1) : make_uint4(0, 0, 0, 0);
            kr[1][1] = v1 ? pa::ld_stream16(k1 + 64) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 2 * tq + (i & 1) + 8 * (i >> 1);
            vr[i] = tok < nvalid ? pa::ld_stream16(vc + base + tok * row_elems + offv) : make_uint4(0, 0, 0, 0);
        }

        // S^T = K Q^T: one MMA per 16-dim step covers the chunk's 16 tokens
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint32_t w0[8] = {kr[0][0].x, kr[0][0].y, kr[0][0].z, kr[0][0].w,
                                    kr[0][1].x, kr[0][1].y, kr[0][1].z, kr[0][1].w};
            const uint32_t w1[8] = {kr[1][0].x, kr[1][0].y, kr[1][0].z, kr[1][0].w,
                                    kr[1][1].x, kr[1][1].y, kr[1][1].z, kr[1][1].w};
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                uint32_t a0, a1, a2, a3;  // tokens gq (a0, a2) and gq + 8 (a1, a3)
                e4m3x4_to_f16x2x2(w0[st], a0, a2, p.code_mul);
                e4m3x4_to_f16x2x2(w1[st], a1, a3, p.code_mul);
                mma_16816(sc, a0, a1, a2, a3, qa[st][0], qa[st][1]);
            }
        }

        // sc: tokens gq (0, 1) and gq + 8 (2, 3), heads 2tq (0, 2) and 2tq + 1 (1, 3)
        float x[4];
        x[0] = gq < nvalid ? sc[0] * ss0 : -INFINITY;
        x[1] = gq < nvalid ? sc[1] * ss1 : -INFINITY;
        x[2] = gq + 8 < nvalid ? sc[2] * ss0 : -INFINITY;
        x[3] = gq + 8 < nvalid ? sc[3] * ss1 : -INFINITY;
        float cm0 = fmaxf(x[0], x[2]), cm1 = fmaxf(x[1], x[3]);
        if (__any_sync(FULL, cm0 > m0 + FP8_RESCALE_THRESHOLD || cm1 > m1 + FP8_RESCALE_THRESHOLD)) {
            // the chunk's max of each head over its 8 lanes (finite: token 0 of a
            // chunk is always in the split)
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                cm0 = fmaxf(cm0, __shfl_xor_sync(FULL, cm0, off));
                cm1 = fmaxf(cm1, __shfl_xor_sync(FULL, cm1, off));
            }
            const float n0 = cm0 > m0 + FP8_RESCALE_THRESHOLD ? cm0 : m0;
            const float n1 = cm1 > m1 + FP8_RESCALE_THRESHOLD ? cm1 : m1;
            const float a0 = pa::sm100::ex2_approx(m0 - n0), a1 = pa::sm100::ex2_approx(m1 - n1);  // 0 at first
            l0 *= a0;
            l1 *= a1;
            m0 = n0;
            m1 = n1;
            // the O^T columns of this lane are the same heads
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
                o[mb][0] *= a0;
                o[mb][1] *= a1;
                o[mb][2] *= a0;
                o[mb][3] *= a1;
            }
        }
        float pr[4];
        pr[0] = pa::sm100::ex2_approx(x[0] - m0);
        pr[1] = pa::sm100::ex2_approx(x[1] - m1);
        pr[2] = pa::sm100::ex2_approx(x[2] - m0);
        pr[3] = pa::sm100::ex2_approx(x[3] - m1);
        l0 += pr[0] + pr[2];
        l1 += pr[1] + pr[3];
        // P^T as the B operand of the P.V MMA wants tokens 2tq, 2tq + 1 of head gq
        // in a lane: the transpose of each 8 x 8 tile of P as the lanes hold it
        const uint32_t pb0 = movmatrix_trans(f16x2_of(pr[0], pr[1]));
        const uint32_t pb1 = movmatrix_trans(f16x2_of(pr[2], pr[3]));
        const uint32_t va[4] = {vr[0].x, vr[0].y, vr[0].z, vr[0].w}, vb[4] = {vr[1].x, vr[1].y, vr[1].z, vr[1].w};
        const uint32_t vcw[4] = {vr[2].x, vr[2].y, vr[2].z, vr[2].w}, vd[4] = {vr[3].x, vr[3].y, vr[3].z, vr[3].w};
#pragma unroll
        for (int i = 0; i < 2; ++i) {
#pragma unroll
            for (int hb = 0; hb < 2; ++hb) {
                // [jj]: byte 2hb + jj of word i (dim 4i + 2hb + jj of the lane's 16) of
                // two tokens as an f16 pair; f0: dim slot gq, tokens 2tq, 2tq+1; f1:
                // slot gq + 8; f2, f3: the same for tokens 2tq+8, 2tq+9
                uint32_t f0[2], f1[2], f2[2], f3[2];
                e4m3_byte_pairs(va[i], vb[i], hb, f0, p.code_mul);
                e4m3_byte_pairs(va[i + 2], vb[i + 2], hb, f1, p.code_mul);
                e4m3_byte_pairs(vcw[i], vd[i], hb, f2, p.code_mul);
                e4m3_byte_pairs(vcw[i + 2], vd[i + 2], hb, f3, p.code_mul);
#pragma unroll
                for (int jj = 0; jj < 2; ++jj)
                    mma_16816(o[4 * i + 2 * hb + jj], f0[jj], f1[jj], f2[jj], f3[jj], pb0, pb1);
            }
        }
    }

    // this CTA's loads are done: the next kernel (the merge) may start launching
    pa::grid_dependents_launch();

    // every warp's partial through shared memory; warp g (sub 0) combines the
    // warps of KV head g
    __shared__ float red_o[NW][G][D];
    __shared__ float red_ml[NW][G][2];
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int h = 2 * tq + (cc & 1);
            if (h < G) red_o[warp][h][16 * gq + 8 * (cc >> 1) + mb] = o[mb][cc];
        }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        l0 += __shfl_xor_sync(FULL, l0, off);
        l1 += __shfl_xor_sync(FULL, l1, off);
    }
    if (gq == 0 && 2 * tq < G) {
        red_ml[warp][2 * tq][0] = m0;
        red_ml[warp][2 * tq][1] = l0;
    }
    if (gq == 0 && 2 * tq + 1 < G) {
        red_ml[warp][2 * tq + 1][0] = m1;
        red_ml[warp][2 * tq + 1][1] = l1;
    }
    __syncthreads();
    if (sub != 0 || lane >= 16) return;
    const int c = lane;  // dims 8c .. 8c + 7 of every head of the group
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mm = -INFINITY;
        for (int w = 0; w < wph; ++w) mm = fmaxf(mm, red_ml[g + w * p.kv_heads][h][0]);
        float ll = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < wph; ++w) {
            const int ww = g + w * p.kv_heads;
            const float mw = red_ml[ww][h][0];
            const float aw = (mw == -INFINITY) ? 0.f : exp2f(mw - mm);
            ll += red_ml[ww][h][1] * aw;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(red_o[ww][h][8 * c + e], aw, acc[e]);
        }
        if (nsplit == 1) {
            const float inv = p.out_scale / ll;
            uint4 u;
            u.x = pa::pack_bf16x2(acc[0] * inv, acc[1] * inv);
            u.y = pa::pack_bf16x2(acc[2] * inv, acc[3] * inv);
            u.z = pa::pack_bf16x2(acc[4] * inv, acc[5] * inv);
            u.w = pa::pack_bf16x2(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4 *>(p.out + (int64_t(b) * p.num_heads + g * G + h) * D + 8 * c) = u;
        } else {
            const int64_t row = (int64_t(b) * p.max_splits + s) * p.num_heads + g * G + h;
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + row * D + 8 * c);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (c == 0) p.ws_ml[row] = make_float2(mm, ll);
        }
    }
}

// ---------------------------------------------------------------------------
// bf16 decode for four or more query heads per KV head on the warp-level
// tensor-core MMA (mma.sync m16n8k16, bf16 operands, f32 accumulators).
//
// The CUDA-core kernel keeps G x 8 partial dot products, G x 8 query values
// and G x 8 outputs per lane; from G = 4 on they no longer fit its register
// budget and spill.  Here S^T = K Q^T and O^T += V^T P^T run as MMAs laid
// out as the fp8 kernel's (see there): lane (gq, tq) = (lane / 4, lane % 4)
// supplies tokens gq and gq + 8 of a 16-token chunk, dims 32 j + 8 tq .. + 7
// for j < 4 (the pool's bf16 words are the A registers as they are, the query,
// the B operand, taken in the same dim order; the four lanes of a token read
// adjacent 16-byte pieces), and dims 8 gq .. + 7 and 64 + 8 gq .. + 7 of
// tokens 2tq, 2tq+1, 2tq+8, 2tq+9 for P.V (two tokens' values of one dim
// paired by a byte permute).  The softmax is the fp8 kernel's (heads 2tq and
// 2tq + 1 per lane, P^T by movmatrix).  The query (with the head norm and RoPE
// when fused) is formed in the half-warp layout of the CUDA-core kernel and
// staged through shared memory, from which the B fragments are read at every
// chunk.  P is rounded to bf16 for the P.V MMA.
// The fused KV write, the split partials and the output are the CUDA-core
// kernel's.

// d += A (16 x 16, row) * B (16 x 8, col), bf16 in, f32 accumulate
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2, uint32_t a3,
                                               uint32_t b0, uint32_t b1)
{
    asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

template <int G, bool ROPE>
__global__ void __launch_bounds__(NW * 32, 2) decode_bf16_mma_kernel(const DecodeParams p)
{
    const int b = blockIdx.x, s = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int gq = lane >> 2, tq = lane & 3;
    const int half = lane >> 4, c = lane & 15;
    prefetch_first_chunks(p, 2, 0);
    // launched programmatically: everything below may depend on the previous
    // kernel (the KV write of this step's token)
    pa::grid_dependency_wait();

    int ctx = p.context_lens[b];
    if (ctx < 0 || ctx > p.max_ctx || int64_t(ctx) > int64_t(p.max_blocks) * p.block_size ||
        (ROPE && int64_t(ctx) > p.max_positions)) {
        if (s == 0 && threadIdx.x == 0) pa::report(p.status, PA_ERR_BOUNDS);
        ctx = 0;
    }
    if (ctx == 0) {  // padded row: output zeros, read nothing
        if (s == 0) {
            uint4 *o = reinterpret_cast<uint4 *>(p.out + int64_t(b) * p.num_heads * D);
            for (int i = threadIdx.x; i < p.num_heads * D / 8; i += blockDim.x) o[i] = make_uint4(0, 0, 0, 0);
        }
        return;
    }
    const int nsplit = (ctx + p.split_len - 1) / p.split_len;
    if (s >= nsplit) return;

    const int g = warp % p.kv_heads;
    const int sub = warp / p.kv_heads;
    const int wph = NW / p.kv_heads;
    const int t0 = s * p.split_len;
    const int t1 = min(ctx, t0 + p.split_len);
    const int row_elems = p.kv_heads * D;
    const int32_t *table = p.block_table + int64_t(b) * p.max_blocks;
    const uint16_t *kc = static_cast<const uint16_t *>(p.k_cache);
    const uint16_t *vc = static_cast<const uint16_t *>(p.v_cache);

    // Fused KV write, as in the CUDA-core kernel: the sequence's last split
    // stores the step's new token (position ctx - 1) before any warp reads, and
    // the chunk holding it is read through L2.
    int new_tok = -1;
    if (p.k_new != nullptr && s == nsplit - 1) {  // the same for the whole CTA
        new_tok = ctx - 1;
        if (sub == 0) {
            const int32_t phys = table[new_tok / p.block_size];
            const uint16_t *src = (half ? p.v_new : p.k_new) + int64_t(b) * p.kv_new_stride + g * D + 8 * c;
            uint4 u = *reinterpret_cast<const uint4 *>(src);
            if constexpr (ROPE) {
                const RopeLane rl = rope_lane(p.k_weight, p.cos_sin + int64_t(new_tok) * D, c);
                float x[8];
                unpack8(u, x);
                norm_rope_row8(x, c, p.k_weight != nullptr, rl.w, p.eps, rl.c, rl.s);
                if (!half) u = pack8(x);
            }
            if (phys >= 0 && int64_t(phys) < p.num_blocks) {
                const int64_t row = int64_t(phys) * p.block_size + new_tok % p.block_size;
                uint16_t *dst = static_cast<uint16_t *>(const_cast<void *>(half ? p.v_cache : p.k_cache)) +
                                row * row_elems + g * D + 8 * c;
                *reinterpret_cast<uint4 *>(dst) = u;
            }
        }
        __syncthreads();
    }

    auto prefetch_chunk = [&](int cf) {  // a chunk's 16 rows of all KV heads: one contiguous run of one block
        if (cf >= t1) return;
        const int32_t pf = table[cf / p.block_size];
        if (pf < 0 || int64_t(pf) >= p.num_blocks) return;
        const int64_t r = (int64_t(pf) * p.block_size + cf % p.block_size) * row_elems;
        const uint32_t bytes = uint32_t(min(CHUNK, t1 - cf) * row_elems * 2);
        const uint32_t b16 = (bytes + 15u) & ~15u;
        pa::sm100::prefetch_l2_bulk(kc + r, b16);
        pa::sm100::prefetch_l2_bulk(vc + r, b16);
    };

    // the group's query heads, this warp's slice of the merge buffer as staging
    __shared__ __align__(16) float red_o[NW][G][D];
    __shared__ __align__(16) float red_ml[NW][G][2];
    // (the A fragments are read from the staging at every chunk: per 16-dim step,
    // head gq's dims 32 tq + 4 st + {0, 1} and + {2, 3}, one 8-byte load)
    uint16_t *qs = reinterpret_cast<uint16_t *>(&red_o[warp][0][0]);  // [G][D] bf16
    {
        RopeLane rl;
        if constexpr (ROPE) rl = rope_lane(p.q_weight, p.cos_sin + int64_t(ctx - 1) * D, c);
#pragma unroll
        for (int i = 0; i < (G + 1) / 2; ++i) {  // half-warp `half` takes heads half, half + 2, ...
            const int h = 2 * i + half;
            const bool hv = h < G;
            uint4 u = hv ? *reinterpret_cast<const uint4 *>(p.q + int64_t(b) * p.q_stride + (g * G + h) * D + 8 * c)
                         : make_uint4(0, 0, 0, 0);
            if constexpr (ROPE) {
                float x[8];
                unpack8(u, x);
                norm_rope_row8(x, c, p.q_weight != nullptr, rl.w, p.eps, rl.c, rl.s);
                u = pack8(x);
            }
            if (hv) *reinterpret_cast<uint4 *>(qs + h * D + 8 * c) = u;
        }
        __syncwarp();
    }
    const uint16_t *qrow = qs + (gq < G ? gq : 0) * D + 8 * tq;

    // this lane's element offsets within a chunk's first row: its four 8-dim
    // pieces of a key row are 32 dims apart and the four lanes of a token hold
    // adjacent pieces, so that each load instruction reads whole 64-byte runs
    // (K); its two pieces of a value row, 64 dims apart, likewise (V)
    const int offk0 = gq * row_elems + g * D + 8 * tq, offk1 = offk0 + 8 * row_elems;
    const int offv = g * D + 8 * gq;

    float o[8][4];  // O^T: block mb holds dims 8 gq + mb (o[mb][0..1]) and 64 + 8 gq + mb (o[mb][2..3])
#pragma unroll
    for (int mb = 0; mb < 8; ++mb) o[mb][0] = o[mb][1] = o[mb][2] = o[mb][3] = 0.f;
    // heads 2tq, 2tq + 1: running max (the same in the 8 lanes of a tq) and this
    // lane's share of the sum (its tokens), added up over the 8 lanes at the end
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    const float sscale = p.scale_log2;

    for (int cb = t0 + sub * CHUNK; cb < t1; cb += wph * CHUNK) {
        const int32_t phys = table[cb / p.block_size];
        if (phys < 0 || int64_t(phys) >= p.num_blocks) {
            if (lane == 0) pa::report(p.status, PA_ERR_BOUNDS);
            continue;
        }
        // a chunk never crosses a block: cb and block_size are multiples of 16
        const int64_t base = (int64_t(phys) * p.block_size + (cb % p.block_size)) * row_elems;
        const int nvalid = t1 - cb;
        if (PREFETCH_CHUNKS > 0 && g == 0 && lane == 0) prefetch_chunk(cb + PREFETCH_CHUNKS * wph * CHUNK);
        // the chunk holding the row this launch wrote: coherent loads through L2
        const bool coherent = unsigned(new_tok - cb) < unsigned(CHUNK);
        auto ld = [&](const uint16_t *ptr, bool v) {
            return !v ? make_uint4(0, 0, 0, 0) : coherent ? __ldcg(reinterpret_cast<const uint4 *>(ptr))
                                                          : pa::ld_stream16(ptr);
        };
        uint4 kr[2][4], vr[4][2];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            kr[0][j] = ld(kc + base + offk0 + 32 * j, gq < nvalid);
            kr[1][j] = ld(kc + base + offk1 + 32 * j, 8 + gq < nvalid);
        }
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const int tok = 2 * tq + (i & 1) + 8 * (i >> 1);
            const uint16_t *vp = vc + base + tok * row_elems + offv;
            vr[i][0] = ld(vp, tok < nvalid);
            vr[i][1] = ld(vp + 64, tok < nvalid);
        }

        // S^T = K Q^T: one MMA per 16-dim step covers the chunk's 16 tokens
        float sc[4] = {0.f, 0.f, 0.f, 0.f};
        {
            const uint32_t w0[16] = {kr[0][0].x, kr[0][0].y, kr[0][0].z, kr[0][0].w,
                                     kr[0][1].x, kr[0][1].y, kr[0][1].z, kr[0][1].w,
                                     kr[0][2].x, kr[0][2].y, kr[0][2].z, kr[0][2].w,
                                     kr[0][3].x, kr[0][3].y, kr[0][3].z, kr[0][3].w};
            const uint32_t w1[16] = {kr[1][0].x, kr[1][0].y, kr[1][0].z, kr[1][0].w,
                                     kr[1][1].x, kr[1][1].y, kr[1][1].z, kr[1][1].w,
                                     kr[1][2].x, kr[1][2].y, kr[1][2].z, kr[1][2].w,
                                     kr[1][3].x, kr[1][3].y, kr[1][3].z, kr[1][3].w};
#pragma unroll
            for (int st = 0; st < 8; ++st) {
                const uint2 qq = gq < G ? *reinterpret_cast<const uint2 *>(qrow + 32 * (st >> 1) + 4 * (st & 1))
                                        : make_uint2(0u, 0u);
                // A: tokens gq (words 2st, 2st + 1) and gq + 8; B: head gq's query
                mma_bf16_16816(sc, w0[2 * st], w1[2 * st], w0[2 * st + 1], w1[2 * st + 1], qq.x, qq.y);
            }
        }

        // sc: tokens gq (0, 1) and gq + 8 (2, 3), heads 2tq (0, 2) and 2tq + 1 (1, 3)
        float x[4];
        x[0] = gq < nvalid ? sc[0] * sscale : -INFINITY;
        x[1] = gq < nvalid ? sc[1] * sscale : -INFINITY;
        x[2] = gq + 8 < nvalid ? sc[2] * sscale : -INFINITY;
        x[3] = gq + 8 < nvalid ? sc[3] * sscale : -INFINITY;
        float cm0 = fmaxf(x[0], x[2]), cm1 = fmaxf(x[1], x[3]);
        if (__any_sync(FULL, cm0 > m0 + FP8_RESCALE_THRESHOLD || cm1 > m1 + FP8_RESCALE_THRESHOLD)) {
            // the chunk's max of each head over its 8 lanes (finite: token 0 of a
            // chunk is always in the split)
#pragma unroll
            for (int off = 4; off <= 16; off <<= 1) {
                cm0 = fmaxf(cm0, __shfl_xor_sync(FULL, cm0, off));
                cm1 = fmaxf(cm1, __shfl_xor_sync(FULL, cm1, off));
            }
            const float n0 = cm0 > m0 + FP8_RESCALE_THRESHOLD ? cm0 : m0;
            const float n1 = cm1 > m1 + FP8_RESCALE_THRESHOLD ? cm1 : m1;
            const float a0 = pa::sm100::ex2_approx(m0 - n0), a1 = pa::sm100::ex2_approx(m1 - n1);  // 0 at first
            l0 *= a0;
            l1 *= a1;
            m0 = n0;
            m1 = n1;
            // the O^T columns of this lane are the same heads
#pragma unroll
            for (int mb = 0; mb < 8; ++mb) {
                o[mb][0] *= a0;
                o[mb][1] *= a1;
                o[mb][2] *= a0;
                o[mb][3] *= a1;
            }
        }
        float pr[4];
        pr[0] = pa::sm100::ex2_approx(x[0] - m0);
        pr[1] = pa::sm100::ex2_approx(x[1] - m1);
        pr[2] = pa::sm100::ex2_approx(x[2] - m0);
        pr[3] = pa::sm100::ex2_approx(x[3] - m1);
        l0 += pr[0] + pr[2];
        l1 += pr[1] + pr[3];
        // P^T as the B operand of the P.V MMA: the transpose of each 8 x 8 tile
        const uint32_t pb0 = movmatrix_trans(pa::pack_bf16x2(pr[0], pr[1]));
        const uint32_t pb1 = movmatrix_trans(pa::pack_bf16x2(pr[2], pr[3]));
        // the words of tokens 2tq (a), 2tq+1 (b), 2tq+8 (c), 2tq+9 (d): word k < 4 holds dims
        // 8 gq + 2k, 2k+1, word 4 + k dims 64 + 8 gq + 2k, 2k+1
        auto words = [&](int t, uint32_t (&w8)[8]) {
            w8[0] = vr[t][0].x; w8[1] = vr[t][0].y; w8[2] = vr[t][0].z; w8[3] = vr[t][0].w;
            w8[4] = vr[t][1].x; w8[5] = vr[t][1].y; w8[6] = vr[t][1].z; w8[7] = vr[t][1].w;
        };
        uint32_t wa[8], wb[8], wc[8], wd[8];
        words(0, wa);
        words(1, wb);
        words(2, wc);
        words(3, wd);
#pragma unroll
        for (int mb = 0; mb < 8; ++mb) {
            // dim slot gq: dim 8 gq + mb; slot gq + 8: dim 64 + 8 gq + mb
            const uint32_t sel = (mb & 1) ? 0x7632u : 0x5410u;
            const int w0 = mb >> 1, w1 = 4 + (mb >> 1);
            mma_bf16_16816(o[mb], __byte_perm(wa[w0], wb[w0], sel), __byte_perm(wa[w1], wb[w1], sel),
                           __byte_perm(wc[w0], wd[w0], sel), __byte_perm(wc[w1], wd[w1], sel), pb0, pb1);
        }
    }

    // this CTA's loads are done: the next kernel (the merge) may start launching
    pa::grid_dependents_launch();

    // every warp's partial through shared memory, over its query staging once
    // every lane of the warp is done with it; warp g (sub 0) combines the warps
    // of KV head g
    __syncwarp();
#pragma unroll
    for (int mb = 0; mb < 8; ++mb)
#pragma unroll
        for (int cc = 0; cc < 4; ++cc) {
            const int h = 2 * tq + (cc & 1);
            if (h < G) red_o[warp][h][8 * gq + 64 * (cc >> 1) + mb] = o[mb][cc];
        }
#pragma unroll
    for (int off = 4; off <= 16; off <<= 1) {
        l0 += __shfl_xor_sync(FULL, l0, off);
        l1 += __shfl_xor_sync(FULL, l1, off);
    }
    if (gq == 0 && 2 * tq < G) {
        red_ml[warp][2 * tq][0] = m0;
        red_ml[warp][2 * tq][1] = l0;
    }
    if (gq == 0 && 2 * tq + 1 < G) {
        red_ml[warp][2 * tq + 1][0] = m1;
        red_ml[warp][2 * tq + 1][1] = l1;
    }
    __syncthreads();
    if (sub != 0 || lane >= 16) return;
#pragma unroll
    for (int h = 0; h < G; ++h) {
        float mm = -INFINITY;
        for (int w = 0; w < wph; ++w) mm = fmaxf(mm, red_ml[g + w * p.kv_heads][h][0]);
        float ll = 0.f, acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        for (int w = 0; w < wph; ++w) {
            const int ww = g + w * p.kv_heads;
            const float mw = red_ml[ww][h][0];
            const float aw = (mw == -INFINITY) ? 0.f : exp2f(mw - mm);
            ll += red_ml[ww][h][1] * aw;
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[e] = fmaf(red_o[ww][h][8 * c + e], aw, acc[e]);
        }
        if (nsplit == 1) {
            const float inv = p.out_scale / ll;
            uint4 u;
            u.x = pa::pack_bf16x2(acc[0] * inv, acc[1] * inv);
            u.y = pa::pack_bf16x2(acc[2] * inv, acc[3] * inv);
            u.z = pa::pack_bf16x2(acc[4] * inv, acc[5] * inv);
            u.w = pa::pack_bf16x2(acc[6] * inv, acc[7] * inv);
            *reinterpret_cast<uint4 *>(p.out + (int64_t(b) * p.num_heads + g * G + h) * D + 8 * c) = u;
        } else {
            const int64_t row = (int64_t(b) * p.max_splits + s) * p.num_heads + g * G + h;
            float4 *dst = reinterpret_cast<float4 *>(p.ws_o + row * D + 8 * c);
            dst[0] = make_float4(acc[0], acc[1], acc[2], acc[3]);
            dst[1] = make_float4(acc[4], acc[5], acc[6], acc[7]);
            if (c == 0) p.ws_ml[row] = make_float2(mm, ll);
        }
    }
}

// Merge the split partials of every sequence that has more than one split
// ("大模型推理入门与 nano-vLLM 源码详解" §9.5): M = max_s m_s,
// L = sum_s l_s 2^(m_s - M), out = sum_s o_s 2^(m_s - M) / L.  A thread per
// (head, 8 columns), 256 threads per CTA and (heads x 16 / 256) CTAs per
// sequence, so the 16 threads of a head are one half-warp.  Per window of 16
// splits each of them loads one split's (max, sum); M and L are reduced over
// the half-warp by shuffles, and each split's weight 2^(m_s - M) is handed to
// the 16 threads by a shuffle as they add that split's 8 columns of o_s.  The
// statistics and the partials of the window's first eight splits are loaded
// together (up to eight splits cost one round trip to L2); a later window
// rescales the running (M, L, out) as M grows.
__global__ void __launch_bounds__(256) decode_merge_kernel(const DecodeParams p)
{
    pa::grid_dependency_wait();  // the split kernel's partials
    pa::grid_dependents_launch();
    const int b = blockIdx.x;
    int ctx = p.context_lens[b];
    if (ctx <= 0 || ctx > p.max_ctx || int64_t(ctx) > int64_t(p.max_blocks) * p.block_size ||
        (p.cos_sin != nullptr && int64_t(ctx) > p.max_positions))
        return;
    const int nsplit = (ctx + p.split_len - 1) / p.split_len;
    if (nsplit <= 1) return;
    const int item = int(blockIdx.y * blockDim.x + threadIdx.x);
    // (heads x 16 items: whole half-warps leave here, never part of one)
    if (item >= p.num_heads * (D / 8)) return;
    const int h = item / (D / 8), c = item % (D / 8);
    const int lane = int(threadIdx.x & 31), half0 = lane & 16;
    const unsigned hmask = 0xffffu << half0;  // this head's half-warp
    const int64_t base = int64_t(b) * p.max_splits * p.num_heads + h;
    constexpr int MS = 8;
    float mm = -INFINITY, ll = 0.f;
    float acc[8] = {0, 0, 0, 0, 0, 0, 0, 0};
    for (int t0 = 0; t0 < nsplit; t0 += 16) {
        const int nw = min(16, nsplit - t0);
        const float2 ml = c < nw ? p.ws_ml[base + int64_t(t0 + c) * p.num_heads] : make_float2(-INFINITY, 0.f);
        float4 x0[MS], x1[MS];
#pragma unroll
        for (int u = 0; u < MS; ++u) {
            if (u < nw) {
                const float4 *src =
                    reinterpret_cast<const float4 *>(p.ws_o + (base + int64_t(t0 + u) * p.num_heads) * D + 8 * c);
                x0[u] = src[0];
                x1[u] = src[1];
            } else {
                x0[u] = x1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
            }
        }
        float gm = ml.x;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) gm = fmaxf(gm, __shfl_xor_sync(hmask, gm, o));
        gm = fmaxf(gm, mm);
        const float a = (mm == -INFINITY) ? 0.f : exp2f(mm - gm);
        ll *= a;
#pragma unroll
        for (int e = 0; e < 8; ++e) acc[e] *= a;
        mm = gm;
        const float w = (ml.x == -INFINITY) ? 0.f : exp2f(ml.x - mm);  // split t0 + c's weight
        float lw = ml.y * w;
#pragma unroll
        for (int o = 8; o >= 1; o >>= 1) lw += __shfl_xor_sync(hmask, lw, o);
        ll += lw;
        for (int v0 = 0; v0 < nw; v0 += MS) {
            if (v0 > 0) {  // splits 8 .. 15 of the window
#pragma unroll
                for (int u = 0; u < MS; ++u) {
                    if (v0 + u < nw) {
                        const float4 *src = reinterpret_cast<const float4 *>(
                            p.ws_o + (base + int64_t(t0 + v0 + u) * p.num_heads) * D + 8 * c);
                        x0[u] = src[0];
                        x1[u] = src[1];
                    } else {
                        x0[u] = x1[u] = make_float4(0.f, 0.f, 0.f, 0.f);
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < MS; ++u) {
                const float wu = __shfl_sync(hmask, w, half0 | (v0 + u));  // 0 past the window's splits
                acc[0] += x0[u].x * wu; acc[1] += x0[u].y * wu; acc[2] += x0[u].z * wu; acc[3] += x0[u].w * wu;
                acc[4] += x1[u].x * wu; acc[5] += x1[u].y * wu; acc[6] += x1[u].z * wu; acc[7] += x1[u].w * wu;
            }
        }
    }
    const float inv = p.out_scale / ll;
    uint4 u;
    u.x = pa::pack_bf16x2(acc[0] * inv, acc[1] * inv);
    u.y = pa::pack_bf16x2(acc[2] * inv, acc[3] * inv);
    u.z = pa::pack_bf16x2(acc[4] * inv, acc[5] * inv);
    u.w = pa::pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4 *>(p.out + (int64_t(b) * p.num_heads + h) * D + 8 * c) = u;
}

// Long contexts in a large batch: every sequence is split into CLUSTER_SPLITS
// equal parts, launched as one thread-block cluster that merges them in
// distributed shared memory (the workspace and the merge kernel go unused).
// Taken where the split plan would cut sequences into more parts than that,
// the batch has at least four such CTAs per SM and no part exceeds
// CLUSTER_MAX_SPLIT tokens (measured: a 512 x U[1k, 4k] batch 3% faster than
// 256-token splits and the merge kernel; shorter contexts, where the plan's
// 128-token splits leave many sequences with fewer parts than a cluster has
// CTAs, were slower in clusters).
constexpr int CLUSTER_SPLITS = 8;
// bf16 calls with at least this many query heads per KV head run the MMA kernel
constexpr int MMA_GROUP_MIN = 4;
constexpr int CLUSTER_MAX_SPLIT = 1024;
inline bool use_cluster(bool fp8, int num_seqs, int max_ctx, const Plan &plan)
{
    const int sms = pa::num_sms() > 0 ? pa::num_sms() : 152;
    return !fp8 && plan.max_splits > CLUSTER_SPLITS && max_ctx <= CLUSTER_SPLITS * CLUSTER_MAX_SPLIT &&
           int64_t(num_seqs) * CLUSTER_SPLITS >= 4LL * sms;
}

template <int G, bool FP8>
pa_status launch_split(const DecodeParams &p, bool cluster, cudaStream_t stream)
{
    const dim3 block(NW * 32);
    if constexpr (FP8) {
        const dim3 grid(unsigned(p.num_seqs), unsigned(p.max_splits > 0 ? p.max_splits : 1));
        pa::launch_pdl(decode_fp8_mma_kernel<G>, grid, block, 0, stream, p);
    } else if constexpr (G >= MMA_GROUP_MIN) {
        const dim3 grid(unsigned(p.num_seqs), unsigned(p.max_splits > 0 ? p.max_splits : 1));
        if (p.cos_sin != nullptr)
            pa::launch_pdl(decode_bf16_mma_kernel<G, true>, grid, block, 0, stream, p);
        else
            pa::launch_pdl(decode_bf16_mma_kernel<G, false>, grid, block, 0, stream, p);
    } else if (cluster) {
        const dim3 grid(unsigned(p.num_seqs), unsigned(CLUSTER_SPLITS));
        if (p.cos_sin != nullptr)
            pa::launch_pdl_cluster_y(decode_split_kernel<G, true, true>, grid, block, 0, stream, CLUSTER_SPLITS, p);
        else
            pa::launch_pdl_cluster_y(decode_split_kernel<G, false, true>, grid, block, 0, stream, CLUSTER_SPLITS, p);
    } else {
        const dim3 grid(unsigned(p.num_seqs), unsigned(p.max_splits > 0 ? p.max_splits : 1));
        if (p.cos_sin != nullptr)
            pa::launch_pdl(decode_split_kernel<G, true, false>, grid, block, 0, stream, p);
        else
            pa::launch_pdl(decode_split_kernel<G, false, false>, grid, block, 0, stream, p);
    }
    return PA_OK;
}

pa_status check_args(const void *q, int64_t q_stride_seq, const void *k_cache, const void *v_cache,
                     int64_t num_blocks, int block_size, const int32_t *block_table, int max_blocks,
                     const int32_t *context_lens, int num_seqs, int max_ctx, int num_heads, int kv_heads,
                     int head_dim, const void *out)
{
    if (num_seqs < 0 || max_ctx < 0 || num_blocks < 0 || max_blocks < 0) return PA_ERR_INVALID_ARG;
    if (head_dim != D || !pa::pow2_in(kv_heads, 1, 8) || num_heads <= 0 || num_heads % kv_heads != 0 ||
        !pa::pow2_in(num_heads / kv_heads, 1, 8))
        return PA_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 1024 || block_size % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0) return PA_OK;
    if (!q || !k_cache || !v_cache || !block_table || !context_lens || !out) return PA_ERR_INVALID_ARG;
    if (max_blocks < 1) return PA_ERR_INVALID_ARG;
    if (q_stride_seq < int64_t(num_heads) * D || q_stride_seq % 8 != 0) return PA_ERR_INVALID_ARG;
    if (!pa::aligned(q, 16) || !pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16) || !pa::aligned(out, 16))
        return PA_ERR_INVALID_ARG;
    return PA_OK;
}

}  // namespace

extern "C" size_t pa_decode_workspace_bytes(int num_seqs, int num_heads, int head_dim, int max_context_len)
{
    if (num_seqs < 0 || num_heads <= 0 || head_dim != D || max_context_len < 0) return 0;
    return workspace_bytes(num_seqs, num_heads, make_plan(num_seqs, max_context_len, num_heads));
}

namespace {

pa_status decode_impl(const void *q, int64_t q_stride_seq, const void *k_cache, const void *v_cache, bool fp8,
                      float k_scale, float v_scale, int64_t num_blocks, int block_size, const int32_t *block_table,
                      int max_blocks_per_seq, const int32_t *context_lens, int num_seqs, int max_context_len,
                      int num_heads, int num_kv_heads, int head_dim, float scale, void *out, void *workspace,
                      size_t workspace_bytes_given, int32_t *dev_status, void *stream, const void *k_new = nullptr,
                      const void *v_new = nullptr, int64_t kv_new_stride = 0, const float *cos_sin = nullptr,
                      int64_t max_positions = 0, const void *q_weight = nullptr, const void *k_weight = nullptr,
                      float eps = 0.f)
{
    pa_status st = check_args(q, q_stride_seq, k_cache, v_cache, num_blocks, block_size, block_table,
                              max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads,
                              num_kv_heads, head_dim, out);
    if (st != PA_OK || num_seqs == 0) return st;
    const Plan plan = make_plan(num_seqs, max_context_len, num_heads, fp8 ? PLAN_CTAS_PER_SM_FP8 : PLAN_CTAS_PER_SM);
    if (plan.max_splits > 65535) return PA_ERR_UNSUPPORTED;
    const size_t need = workspace_bytes(num_seqs, num_heads, plan);
    if (need > 0 && (workspace == nullptr || workspace_bytes_given < need || !pa::aligned(workspace, 256)))
        return PA_ERR_INVALID_ARG;

    DecodeParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.q_stride = q_stride_seq;
    p.k_cache = k_cache;
    p.v_cache = v_cache;
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.block_table = block_table;
    p.max_blocks = max_blocks_per_seq;
    p.context_lens = context_lens;
    p.num_seqs = num_seqs;
    p.max_ctx = max_context_len;
    p.num_heads = num_heads;
    p.kv_heads = num_kv_heads;
    p.scale_log2 = scale * LOG2E * k_scale;
    p.out_scale = fp8 ? v_scale * 256.f : v_scale;  // (fp8 values enter the P.V MMAs times 2^-8)
    p.out = static_cast<uint16_t *>(out);
    p.k_new = static_cast<const uint16_t *>(k_new);
    p.v_new = static_cast<const uint16_t *>(v_new);
    p.kv_new_stride = kv_new_stride;
    p.cos_sin = cos_sin;
    p.max_positions = max_positions;
    p.q_weight = static_cast<const uint16_t *>(q_weight);
    p.k_weight = static_cast<const uint16_t *>(k_weight);
    p.eps = eps;
    const size_t n = size_t(num_seqs) * (plan.max_splits > 0 ? plan.max_splits : 1) * num_heads;
    p.ws_o = static_cast<float *>(workspace);
    p.ws_ml = need > 0 ? reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                                   (n * D * sizeof(float) + 255) / 256 * 256)
                       : nullptr;
    p.split_len = plan.split_len;
    p.max_splits = plan.max_splits;
    p.status = dev_status;
    p.code_mul = 128u;

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const int group = num_heads / num_kv_heads;
    const bool cl = num_heads / num_kv_heads < MMA_GROUP_MIN && use_cluster(fp8, num_seqs, max_context_len, plan);
    pa_status ls = PA_OK;
    if (fp8) {
        switch (group) {
        case 1: ls = launch_split<1, true>(p, false, s); break;
        case 2: ls = launch_split<2, true>(p, false, s); break;
        case 4: ls = launch_split<4, true>(p, false, s); break;
        default: ls = launch_split<8, true>(p, false, s); break;
        }
    } else {
        switch (group) {
        case 1: ls = launch_split<1, false>(p, cl, s); break;
        case 2: ls = launch_split<2, false>(p, cl, s); break;
        case 4: ls = launch_split<4, false>(p, cl, s); break;
        default: ls = launch_split<8, false>(p, cl, s); break;
        }
    }
    if (ls != PA_OK) return ls;
    if (plan.max_splits > 1 && !cl)
        pa::launch_pdl(decode_merge_kernel, dim3(unsigned(num_seqs), unsigned((num_heads * (D / 8) + 255) / 256)),
                       dim3(256), 0, s, p);
    return pa::launch_status();
}

}  // namespace

extern "C" pa_status pa_decode_paged(const void *q, int64_t q_stride_seq, const void *k_cache, const void *v_cache,
                                     int64_t num_blocks, int block_size, const int32_t *block_table,
                                     int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                     int max_context_len, int num_heads, int num_kv_heads, int head_dim,
                                     float scale, void *out, void *workspace, size_t workspace_bytes_given,
                                     int32_t *dev_status, void *stream)
{
    return decode_impl(q, q_stride_seq, k_cache, v_cache, false, 1.f, 1.f, num_blocks, block_size, block_table,
                       max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads, num_kv_heads,
                       head_dim, scale, out, workspace, workspace_bytes_given, dev_status, stream);
}

// The decode step's KV write and decode in one launch: the sequence's last
// split stores k_new[b] / v_new[b] at the pool row of position
// context_lens[b] - 1 (found through the block table, as the decode step's
// slot is) and decodes with it.
extern "C" pa_status pa_store_decode_paged(const void *q, int64_t q_stride_seq, const void *k_new, const void *v_new,
                                           int64_t kv_new_stride_seq, void *k_cache, void *v_cache,
                                           int64_t num_blocks, int block_size, const int32_t *block_table,
                                           int max_blocks_per_seq, const int32_t *context_lens, int num_seqs,
                                           int max_context_len, int num_heads, int num_kv_heads, int head_dim,
                                           float scale, void *out, void *workspace, size_t workspace_bytes_given,
                                           int32_t *dev_status, void *stream)
{
    if (num_seqs > 0 && (k_new == nullptr || v_new == nullptr || !pa::aligned(k_new, 16) ||
                         !pa::aligned(v_new, 16) || kv_new_stride_seq < int64_t(num_kv_heads) * head_dim ||
                         kv_new_stride_seq % 8 != 0))
        return PA_ERR_INVALID_ARG;
    return decode_impl(q, q_stride_seq, k_cache, v_cache, false, 1.f, 1.f, num_blocks, block_size, block_table,
                       max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads, num_kv_heads,
                       head_dim, scale, out, workspace, workspace_bytes_given, dev_status, stream, k_new, v_new,
                       kv_new_stride_seq);
}

// The decode step of one layer from the fused QKV projection's output, in one
// launch (plus the merge): q and the new k get the head norm and RoPE at
// position context_lens[b] - 1, the new k and v go to that position's pool row
// (through the block table), and the decode runs as pa_store_decode_paged's.
extern "C" pa_status pa_norm_rope_store_decode_paged(const void *qkv, int64_t qkv_stride_seq, const float *cos_sin,
                                                     int64_t max_positions, const void *q_norm_weight,
                                                     const void *k_norm_weight, float eps, void *k_cache,
                                                     void *v_cache, int64_t num_blocks, int block_size,
                                                     const int32_t *block_table, int max_blocks_per_seq,
                                                     const int32_t *context_lens, int num_seqs, int max_context_len,
                                                     int num_heads, int num_kv_heads, int head_dim, float scale,
                                                     void *out, void *workspace, size_t workspace_bytes_given,
                                                     int32_t *dev_status, void *stream)
{
    if (num_seqs > 0) {
        if (qkv == nullptr || cos_sin == nullptr || !pa::aligned(qkv, 16) || !pa::aligned(cos_sin, 16) ||
            max_positions < 1 || !(eps >= 0.f))
            return PA_ERR_INVALID_ARG;
        if (num_heads <= 0 || num_kv_heads <= 0 ||
            qkv_stride_seq < int64_t(num_heads + 2 * num_kv_heads) * head_dim || qkv_stride_seq % 8 != 0)
            return PA_ERR_INVALID_ARG;
        if ((q_norm_weight && !pa::aligned(q_norm_weight, 16)) || (k_norm_weight && !pa::aligned(k_norm_weight, 16)))
            return PA_ERR_INVALID_ARG;
    }
    const uint16_t *base = static_cast<const uint16_t *>(qkv);
    const int64_t kcol = int64_t(num_heads) * head_dim, vcol = kcol + int64_t(num_kv_heads) * head_dim;
    return decode_impl(qkv, qkv_stride_seq, k_cache, v_cache, false, 1.f, 1.f, num_blocks, block_size, block_table,
                       max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads, num_kv_heads,
                       head_dim, scale, out, workspace, workspace_bytes_given, dev_status, stream,
                       num_seqs > 0 ? base + kcol : nullptr, num_seqs > 0 ? base + vcol : nullptr, qkv_stride_seq,
                       cos_sin, max_positions, q_norm_weight, k_norm_weight, eps);
}

// Decode over fp8 (E4M3) pools written by pa_store_kvcache_fp8: the same
// kernel reading 1-byte elements (half the bytes per context token), with K
// scaled inside the score and V scaled once at the output.
extern "C" pa_status pa_decode_paged_fp8(const void *q, int64_t q_stride_seq, const void *k_cache,
                                         const void *v_cache, float k_scale, float v_scale, int64_t num_blocks,
                                         int block_size, const int32_t *block_table, int max_blocks_per_seq,
                                         const int32_t *context_lens, int num_seqs, int max_context_len,
                                         int num_heads, int num_kv_heads, int head_dim, float scale, void *out,
                                         void *workspace, size_t workspace_bytes_given, int32_t *dev_status,
                                         void *stream)
{
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || isinf(k_scale) || isinf(v_scale)) return PA_ERR_INVALID_ARG;
    return decode_impl(q, q_stride_seq, k_cache, v_cache, true, k_scale, v_scale, num_blocks, block_size,
                       block_table, max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads,
                       num_kv_heads, head_dim, scale, out, workspace, workspace_bytes_given, dev_status, stream);
}

// ---------------------------------------------------------------------------
// Decode without caller-provided scratch.
//
// Some callers cannot allocate device memory: code embedded in a host
// framework that owns the whole device memory pool and forbids foreign
// cudaMalloc calls, services that must not allocate once they are serving,
// and plain C callers with no device-memory manager at all.  For them the
// split partials live in this file-scope device array instead of a
// workspace argument.  Every GPU that loads this library holds the array
// until the process exits.
static __device__ __align__(256) unsigned char g_decode_noalloc_scratch[PA_DECODE_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of the scratch array on the current device, looked up once
// per device with that device current (in host code the array's name is
// only a host-side stand-in, never a device address).
pa_status noalloc_scratch_address(void **out)
{
    static std::mutex mu;
    static void *addr[64] = {nullptr};
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return PA_ERR_CUDA;
    std::lock_guard<std::mutex> lock(mu);
    if (addr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_decode_noalloc_scratch) != cudaSuccess || p == nullptr) return PA_ERR_CUDA;
        addr[dev] = p;
    }
    *out = addr[dev];
    return PA_OK;
}

}  // namespace

extern "C" pa_status pa_decode_paged_noalloc(const void *q, int64_t q_stride_seq, const void *k_cache,
                                             const void *v_cache, int64_t num_blocks, int block_size,
                                             const int32_t *block_table, int max_blocks_per_seq,
                                             const int32_t *context_lens, int num_seqs, int max_context_len,
                                             int num_heads, int num_kv_heads, int head_dim, float scale, void *out,
                                             int32_t *dev_status, void *stream)
{
    if (num_seqs < 0 || max_context_len < 0 || num_heads <= 0) return PA_ERR_INVALID_ARG;
    if (head_dim != D) return PA_ERR_UNSUPPORTED;
    if (pa_decode_workspace_bytes(num_seqs, num_heads, head_dim, max_context_len) > PA_DECODE_NOALLOC_SCRATCH_BYTES)
        return PA_ERR_UNSUPPORTED;
    void *scratch = nullptr;
    const pa_status st = noalloc_scratch_address(&scratch);
    if (st != PA_OK) return st;
    // The kernels write every partial they later read within one call, so
    // nothing in the scratch has to start at zero.
    return pa_decode_paged(q, q_stride_seq, k_cache, v_cache, num_blocks, block_size, block_table,
                           max_blocks_per_seq, context_lens, num_seqs, max_context_len, num_heads, num_kv_heads,
                           head_dim, scale, out, scratch, PA_DECODE_NOALLOC_SCRATCH_BYTES, dev_status, stream);
}
