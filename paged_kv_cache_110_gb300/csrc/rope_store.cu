// rope_store.cu -- per-head RMSNorm of Q and K, rotary position embedding of
// Q and K, and the KV write, in one pass over the fused QKV projection output.
//
// What it computes ("大模型推理入门与 nano-vLLM 源码详解" §12.2, §19.3, §19.7;
// "nano-vllm 技术分析" §4.3-4.4; "VLLM on Fain的Blog" #8 fused RoPE and paged
// KV store):
//   - each Q head and each K head (not V) of a token is RMS-normalised over its
//     128 features: statistics and scaling in fp32, the result rounded to bf16
//     and multiplied by the bf16 weight (rounded again); without a weight this
//     step is skipped;
//   - the normalised vector is rotated by the token's position: feature i is
//     paired with feature i + 64, and the pair (a, b) turns by the table's
//     angle: a' = a cos - b sin, b' = a sin + b cos (fp32, rounded to bf16);
//   - rotated Q goes to q_out; rotated K and the unchanged V go to pool row
//     slot_mapping[t] (slot -1: nothing is stored).
//
// Design: bound by HBM (per token at Hq = 16, Hkv = 8: 8 KiB of QKV read, 4 KiB
// of Q and 4 KiB of K/V written, 512 B of table read through L2).  A producer
// warp streams whole token rows into shared memory with bulk copies, several
// tokens ahead; the compute warps take a 256-byte head row per half-warp, lane
// j holding features 4j .. 4j+3 and their rotation partners 64+4j .. 64+4j+3
// (two 8-byte pieces), so the rotation needs no exchange between lanes; the
// sum of squares is reduced over the half-warp.
#include <mutex>

#include "pa_common.cuh"
#include "sm100_ptx.cuh"

namespace {

constexpr int D = pa::kHeadDim;
constexpr int HALF = D / 2;
constexpr unsigned FULL = 0xffffffffu;

struct RopeParams {
    const uint16_t *qkv;
    int64_t qkv_stride;  // elements
    int64_t num_tokens;
    int num_heads, kv_heads;
    const int32_t *positions;
    const float *cos_sin;  // [max_positions, 128]: cos of the 64 pairs, then sin
    int64_t max_positions;
    const uint16_t *q_weight, *k_weight;  // [128] bf16 or null
    float eps;
    uint16_t *q_out;
    int64_t q_out_stride;
    uint16_t *k_cache, *v_cache;
    int64_t num_slots;
    const int32_t *slots;
    int32_t *status;
    long long wait_limit;  // SM cycles a pipeline wait may take before the call gives up
    int test_stall;        // test hook: the compute warps first wait on a barrier nothing arrives on
};

// Norm (when w != null) and rotate the lane's 4 rotation pairs: lo holds
// features 4j .. 4j+3 and hi features 64+4j .. 64+4j+3 (j = the lane's index in
// its half-warp), so a pair (a, b) = (feature i, feature i + 64) sits in one
// lane; c / s are the cos and sin of those 4 pairs.  Every lane of the warp
// must call this (the sum of squares is reduced over the half-warp).
__device__ __forceinline__ void norm_rope_pairs(uint2 &lo, uint2 &hi, const uint2 *wlo, const uint2 *whi, float eps,
                                                const float (&c)[4], const float (&s)[4])
{
    float a[4] = {pa::bf16_lo(lo.x), pa::bf16_hi(lo.x), pa::bf16_lo(lo.y), pa::bf16_hi(lo.y)};
    float b[4] = {pa::bf16_lo(hi.x), pa::bf16_hi(hi.x), pa::bf16_lo(hi.y), pa::bf16_hi(hi.y)};
    float ss = 0.f;
#pragma unroll
    for (int i = 0; i < 4; ++i) ss = fmaf(b[i], b[i], fmaf(a[i], a[i], ss));
    // offsets below 16 stay within a half-warp
#pragma unroll
    for (int o = 8; o >= 1; o >>= 1) ss += __shfl_xor_sync(FULL, ss, o);
    if (wlo != nullptr) {
        const float r = 1.0f / sqrtf(ss * (1.0f / D) + eps);
        const float wa[4] = {pa::bf16_lo(wlo->x), pa::bf16_hi(wlo->x), pa::bf16_lo(wlo->y), pa::bf16_hi(wlo->y)};
        const float wb[4] = {pa::bf16_lo(whi->x), pa::bf16_hi(whi->x), pa::bf16_lo(whi->y), pa::bf16_hi(whi->y)};
        // v = bf16(bf16(v * r) * w), two elements per conversion instruction
#pragma unroll
        for (int i = 0; i < 4; i += 2) {
            const uint32_t ta = pa::pack_bf16x2(a[i] * r, a[i + 1] * r);
            const uint32_t ua = pa::pack_bf16x2(pa::bf16_lo(ta) * wa[i], pa::bf16_hi(ta) * wa[i + 1]);
            a[i] = pa::bf16_lo(ua), a[i + 1] = pa::bf16_hi(ua);
            const uint32_t tb = pa::pack_bf16x2(b[i] * r, b[i + 1] * r);
            const uint32_t ub = pa::pack_bf16x2(pa::bf16_lo(tb) * wb[i], pa::bf16_hi(tb) * wb[i + 1]);
            b[i] = pa::bf16_lo(ub), b[i + 1] = pa::bf16_hi(ub);
        }
    }
    // a' = a cos - b sin, b' = a sin + b cos (fp32, rounded to bf16)
    float oa[4], ob[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        oa[i] = fmaf(a[i], c[i], -b[i] * s[i]);
        ob[i] = fmaf(a[i], s[i], b[i] * c[i]);
    }
    lo = make_uint2(pa::pack_bf16x2(oa[0], oa[1]), pa::pack_bf16x2(oa[2], oa[3]));
    hi = make_uint2(pa::pack_bf16x2(ob[0], ob[1]), pa::pack_bf16x2(ob[2], ob[3]));
}

// Work: one token at a time per CTA (tokens blockIdx.x, + gridDim.x, ...).
// Warp 4 streams each token's whole QKV row (rows x 256 B, contiguous) and its
// cos / sin row into a ring of STAGES shared-memory stages with bulk copies,
// several tokens ahead, so the bytes in flight do not depend on registers;
// warps 0-3 take the rows of the token in the front stage, a half-warp per
// 256-byte row, and write Q and K out as two 8-byte pieces per lane (a lane's
// rotation pairs) and V rows with 16-byte stores.
constexpr int STAGES = 4;
constexpr int COMPUTE_WARPS = 4;
constexpr int RS_THREADS = (COMPUTE_WARPS + 1) * 32;
constexpr long long RS_WAIT_LIMIT = 1ll << 31;  // SM cycles (about a second)

struct StageInfo {
    int32_t pos, slot, ok, pad;
};

// Bytes of one stage: the QKV row, the 512-byte cos / sin row, the info,
// rounded to 128 bytes.
__host__ __device__ inline int stage_bytes(int rows) { return (rows * D * 2 + 2 * HALF * 4 + 16 + 127) / 128 * 128; }

__global__ void __launch_bounds__(RS_THREADS) norm_rope_store_kernel(const RopeParams p)
{
    extern __shared__ __align__(128) uint8_t sm[];
    using namespace pa::sm100;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, sub = lane & 15, hw = lane >> 4;
    const int rows = p.num_heads + 2 * p.kv_heads;
    const uint32_t row_bytes = uint32_t(rows) * D * 2;
    const int sbytes = stage_bytes(rows);
    const uint32_t sbase = smem_u32(sm);
    const uint32_t bars = sbase + STAGES * sbytes;  // full[STAGES], empty[STAGES]
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(sm + STAGES * sbytes + 2 * STAGES * 8);
    auto full = [&](int s) { return bars + 8u * uint32_t(s); };
    auto empty = [&](int s) { return bars + 8u * uint32_t(STAGES + s); };
    const uint32_t stall = bars + 8u * uint32_t(2 * STAGES) + 8u;  // after the abort flag; never arrived on
    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(full(s), 1);
            mbar_init(empty(s), COMPUTE_WARPS);
        }
        mbar_init(stall, 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    __syncthreads();
    // launched programmatically: the QKV rows, positions and slots come from
    // the kernels before this one
    pa::grid_dependency_wait();
    const int64_t T = p.num_tokens;

    if (warp == COMPUTE_WARPS) {
        // ------------------------------------------------ producer
        // the positions and slots of 32 of this CTA's tokens are read at once
        // (a lane each), then lane 0 issues their copies one stage at a time
        int k = 0;
        bool ok = true;
        for (int64_t t0 = blockIdx.x; ok && t0 < T; t0 += 32 * int64_t(gridDim.x)) {
            const int64_t tl = t0 + int64_t(lane) * gridDim.x;
            int32_t pos = 0, slot = -1;
            if (tl < T) {
                pos = p.positions[tl];
                slot = p.slots[tl];
            }
            for (int l = 0; l < 32; ++l, ++k) {
                const int64_t t = t0 + int64_t(l) * gridDim.x;
                if (t >= T) break;
                const int32_t pl = __shfl_sync(FULL, pos, l), sl = __shfl_sync(FULL, slot, l);
                const int s = k % STAGES;
                if (k >= STAGES) {
                    ok = __all_sync(FULL, mbar_wait(empty(s), uint32_t((k - STAGES) / STAGES) & 1u, abort_flag,
                                                    p.wait_limit));
                    if (!ok) break;
                }
                if (lane == 0) {
                    const bool good = pl >= 0 && pl < p.max_positions &&
                                      (sl == -1 || (sl >= 0 && int64_t(sl) < p.num_slots));
                    StageInfo *info = reinterpret_cast<StageInfo *>(sm + s * sbytes + row_bytes + 2 * HALF * 4);
                    *info = StageInfo{pl, sl, good ? 1 : 0, 0};
                    const uint32_t dst = sbase + uint32_t(s * sbytes);
                    mbar_arrive_expect_tx(full(s), row_bytes + (good ? 2u * HALF * 4u : 0u));
                    bulk_load(dst, p.qkv + t * p.qkv_stride, row_bytes, full(s));
                    if (good) bulk_load(dst + row_bytes, p.cos_sin + int64_t(pl) * D, 2 * HALF * 4, full(s));
                }
                __syncwarp();
            }
        }
        // copies still in flight must land before the CTA's shared memory goes
        // away: wait (bounded, whatever the abort flag says) for the last ones
        if (lane == 0) {
            volatile int32_t dummy = 0;
            for (int u = max(0, k - STAGES); u < k; ++u)
                mbar_wait(full(u % STAGES), uint32_t(u / STAGES) & 1u, &dummy, RS_WAIT_LIMIT);
        }
    } else {
        // ------------------------------------------------ compute warps
        // this lane's weights: features 4 sub .. +3 and 64 + 4 sub .. +3
        uint2 wq_lo = make_uint2(0, 0), wq_hi = wq_lo, wk_lo = wq_lo, wk_hi = wq_lo;
        if (p.q_weight) {
            wq_lo = *reinterpret_cast<const uint2 *>(p.q_weight + sub * 4);
            wq_hi = *reinterpret_cast<const uint2 *>(p.q_weight + HALF + sub * 4);
        }
        if (p.k_weight) {
            wk_lo = *reinterpret_cast<const uint2 *>(p.k_weight + sub * 4);
            wk_hi = *reinterpret_cast<const uint2 *>(p.k_weight + HALF + sub * 4);
        }
        const int iters = (rows + 2 * COMPUTE_WARPS - 1) / (2 * COMPUTE_WARPS);
        // (a test's stall: this wait runs out after the pipeline limit and the
        // CTA stops as after any timeout)
        const bool stalled = p.test_stall && !__all_sync(FULL, mbar_wait(stall, 0, abort_flag, p.wait_limit));
        int k = 0;
        for (int64_t t = blockIdx.x; !stalled && t < T; t += gridDim.x, ++k) {
            const int s = k % STAGES;
            if (!__all_sync(FULL, mbar_wait(full(s), uint32_t(k / STAGES) & 1u, abort_flag, p.wait_limit))) break;
            const uint8_t *stage = sm + s * sbytes;
            const StageInfo info = *reinterpret_cast<const StageInfo *>(stage + row_bytes + 2 * HALF * 4);
            if (!info.ok) {
                if (warp == 0 && lane == 0) pa::report(p.status, PA_ERR_BOUNDS);
            } else {
                const float *cs = reinterpret_cast<const float *>(stage + row_bytes) + sub * 4;
                float c[4], sn[4];
#pragma unroll
                for (int i = 0; i < 4; ++i) c[i] = cs[i], sn[i] = cs[HALF + i];
                for (int it = 0; it < iters; ++it) {
                    const int r = (it * COMPUTE_WARPS + warp) * 2 + hw;
                    const bool live = r < rows;
                    if (r - hw >= p.num_heads + p.kv_heads) {
                        // both rows of the pair are V rows: copied unchanged, no norm or
                        // rotation (a pair that holds a K and a V row, possible when
                        // Hq + Hkv is odd, goes through the path below)
                        if (live && info.slot != -1) {
                            const int g = r - p.num_heads - p.kv_heads;
                            *reinterpret_cast<uint4 *>(p.v_cache + (int64_t(info.slot) * p.kv_heads + g) * D +
                                                       sub * 8) =
                                *reinterpret_cast<const uint4 *>(stage + r * D * 2 + sub * 16);
                        }
                        continue;
                    }
                    uint2 lo = make_uint2(0, 0), hi = lo;
                    if (live) {
                        lo = *reinterpret_cast<const uint2 *>(stage + r * D * 2 + sub * 8);
                        hi = *reinterpret_cast<const uint2 *>(stage + r * D * 2 + HALF * 2 + sub * 8);
                    }
                    if (r - hw + 1 == p.num_heads + p.kv_heads) {
                        // the pair of the last K row and the first V row (Hq + Hkv odd):
                        // both half-warps take part in the norm's shuffles, the V half
                        // stores its row unchanged
                        const uint2 raw_lo = lo, raw_hi = hi;
                        norm_rope_pairs(lo, hi, p.k_weight ? &wk_lo : nullptr, &wk_hi, p.eps, c, sn);
                        if (live && info.slot != -1) {
                            const int g = hw == 0 ? r - p.num_heads : r - p.num_heads - p.kv_heads;
                            uint16_t *dst = (hw == 0 ? p.k_cache : p.v_cache) + (int64_t(info.slot) * p.kv_heads + g) * D;
                            *reinterpret_cast<uint2 *>(dst + sub * 4) = hw == 0 ? lo : raw_lo;
                            *reinterpret_cast<uint2 *>(dst + HALF + sub * 4) = hw == 0 ? hi : raw_hi;
                        }
                        continue;
                    }
                    // Q or K rows only
                    const bool is_q = r < p.num_heads;
                    const bool has_w = is_q ? p.q_weight != nullptr : p.k_weight != nullptr;
                    norm_rope_pairs(lo, hi, has_w ? (is_q ? &wq_lo : &wk_lo) : nullptr, is_q ? &wq_hi : &wk_hi, p.eps,
                                    c, sn);
                    if (!live) continue;
                    uint16_t *dst;
                    if (is_q) {
                        dst = p.q_out + t * p.q_out_stride + int64_t(r) * D;
                    } else if (info.slot != -1) {
                        dst = p.k_cache + (int64_t(info.slot) * p.kv_heads + (r - p.num_heads)) * D;
                    } else {
                        continue;
                    }
                    *reinterpret_cast<uint2 *>(dst + sub * 4) = lo;
                    *reinterpret_cast<uint2 *>(dst + HALF + sub * 4) = hi;
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(empty(s));
        }
    }
    if (threadIdx.x == 0 && *abort_flag) pa::report(p.status, PA_ERR_TIMEOUT);
}

// Row p of the table: cos(p * f_i) for i < head_dim / 2, then sin(p * f_i),
// f_i = base^(-2i / head_dim); double precision, stored as float.
__global__ void __launch_bounds__(256) rope_table_kernel(double base, int head_dim, int64_t max_positions,
                                                         float *table)
{
    const int half = head_dim / 2;
    const int64_t total = max_positions * half;
    for (int64_t k = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; k < total; k += int64_t(gridDim.x) * blockDim.x) {
        const int64_t p = k / half;
        const int i = int(k - p * half);
        const double inv_freq = 1.0 / pow(base, double(2 * i) / head_dim);
        double sn, cn;
        sincos(double(p) * inv_freq, &sn, &cn);
        table[p * head_dim + i] = float(cn);
        table[p * head_dim + half + i] = float(sn);
    }
}

}  // namespace

extern "C" pa_status pa_rope_cos_sin_table(double base, int head_dim, int64_t max_positions, float *table,
                                           void *stream)
{
    if (!(base > 1.0) || head_dim <= 0 || head_dim % 2 != 0 || head_dim > 1024 || max_positions < 0)
        return PA_ERR_INVALID_ARG;
    if (max_positions == 0) return PA_OK;
    if (table == nullptr) return PA_ERR_INVALID_ARG;
    const int64_t total = max_positions * (head_dim / 2);
    const int64_t blocks = (total + 255) / 256;
    const unsigned grid = unsigned(blocks < 4096 ? blocks : 4096);
    rope_table_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(base, head_dim, max_positions, table);
    return pa::launch_status();
}

extern "C" pa_status pa_norm_rope_store_kvcache(const void *qkv, int64_t qkv_stride_tok, int64_t num_tokens,
                                                int num_heads, int num_kv_heads, int head_dim,
                                                const int32_t *positions, const float *cos_sin,
                                                int64_t max_positions, const void *q_norm_weight,
                                                const void *k_norm_weight, float eps, void *q_out,
                                                int64_t q_out_stride_tok, void *k_cache, void *v_cache,
                                                int64_t num_blocks, int block_size, const int32_t *slot_mapping,
                                                int32_t *dev_status, void *stream)
{
    if (num_tokens < 0 || num_blocks < 0 || max_positions < 0) return PA_ERR_INVALID_ARG;
    if (head_dim != D || !pa::pow2_in(num_kv_heads, 1, 8) || num_heads <= 0 || num_heads % num_kv_heads != 0 ||
        !pa::pow2_in(num_heads / num_kv_heads, 1, 8))
        return PA_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 1024 || block_size % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!qkv || !positions || !cos_sin || !q_out || !k_cache || !v_cache || !slot_mapping || max_positions < 1)
        return PA_ERR_INVALID_ARG;
    if (qkv_stride_tok < int64_t(num_heads + 2 * num_kv_heads) * D || qkv_stride_tok % 8 != 0 ||
        q_out_stride_tok < int64_t(num_heads) * D || q_out_stride_tok % 8 != 0)
        return PA_ERR_INVALID_ARG;
    for (const void *ptr : {qkv, static_cast<const void *>(cos_sin), static_cast<const void *>(q_out),
                            static_cast<const void *>(k_cache), static_cast<const void *>(v_cache), q_norm_weight,
                            k_norm_weight})
        if (ptr != nullptr && !pa::aligned(ptr, 16)) return PA_ERR_INVALID_ARG;
    if (!(eps >= 0.f)) return PA_ERR_INVALID_ARG;

    RopeParams p;
    p.qkv = static_cast<const uint16_t *>(qkv);
    p.qkv_stride = qkv_stride_tok;
    p.num_tokens = num_tokens;
    p.num_heads = num_heads;
    p.kv_heads = num_kv_heads;
    p.positions = positions;
    p.cos_sin = cos_sin;
    p.max_positions = max_positions;
    p.q_weight = static_cast<const uint16_t *>(q_norm_weight);
    p.k_weight = static_cast<const uint16_t *>(k_norm_weight);
    p.eps = eps;
    p.q_out = static_cast<uint16_t *>(q_out);
    p.q_out_stride = q_out_stride_tok;
    p.k_cache = static_cast<uint16_t *>(k_cache);
    p.v_cache = static_cast<uint16_t *>(v_cache);
    p.num_slots = num_blocks * block_size;
    p.slots = slot_mapping;
    p.status = dev_status;
    // (the wait that drains the copies in flight after a timeout keeps RS_WAIT_LIMIT)
    p.wait_limit = pa::pipeline_wait_limit(RS_WAIT_LIMIT);
    p.test_stall = pa::pipeline_test_stall() ? 1 : 0;
    // a CTA per token at a time, six CTAs per SM (what shared memory allows at
    // 16 query and 8 KV heads)
    const int rows = num_heads + 2 * num_kv_heads;
    const size_t smem = size_t(STAGES) * stage_bytes(rows) + 2 * STAGES * 8 + 16;
    // the largest QKV row: 64 query heads and 8 KV heads
    const size_t most = size_t(STAGES) * stage_bytes(64 + 2 * 8) + 2 * STAGES * 8 + 16;
    if (pa::allow_dynamic_smem(reinterpret_cast<const void *>(norm_rope_store_kernel), int(most)) != cudaSuccess)
        return PA_ERR_CUDA;
    const int sms = pa::num_sms() > 0 ? pa::num_sms() : 148;
    const int64_t cap = int64_t(sms) * 6;
    const unsigned grid = unsigned(num_tokens < cap ? num_tokens : cap);
    pa::launch_pdl(norm_rope_store_kernel, dim3(grid), dim3(RS_THREADS), smem, static_cast<cudaStream_t>(stream), p);
    return pa::launch_status();
}
