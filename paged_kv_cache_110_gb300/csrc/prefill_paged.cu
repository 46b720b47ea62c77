// prefill_paged.cu -- causal varlen prefill over a block-paged KV cache with
// Blackwell tensor cores (tcgen05, accumulators in TMEM) and TMA page gathers.
//
// What it computes ("大模型推理入门与 nano-vLLM 源码详解" §11.2, §10.2, §13.3):
// sequence b has Lq new queries that are the last Lq positions of its Lk-key
// context; query i (absolute position p = Lk - Lq + i) reads keys 0..p.  Keys
// come from the paged pool through block_table (a cached prefix or an earlier
// chunk) or, without a table, from the new-token k / v rows.  Query head h
// reads KV head h / (Hq / Hkv).  Softmax is accumulated blockwise with a
// running max, a running sum and an unnormalised numerator (§13.3).
//
// One CTA computes a 128-query tile of one (sequence, query head):
//   warp 0      producer: the Q tile (cp.async) and, per 128-key tile, K and
//               V.  Paged keys arrive by TMA, one box per page run: the box
//               height is gcd(block_size, 128) rows, so a box never crosses a
//               page; without a table, rows are copied with cp.async.  All
//               tiles land in shared memory in the 128-byte-swizzled layout
//               the tensor cores read.  Two K/V stages.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of two TMEM
//               S buffers (M = N = 128, K = 128 in eight K = 16 steps), and
//               O += P_{j-1} V_{j-1} with P read from TMEM, so S_{j} is on the
//               tensor cores while the softmax warps work on S_{j-1}.
//   warps 4-7   softmax, one thread per query row: read the S row from TMEM,
//               mask (causal, bottom-right, and keys past the tile's last
//               visible key), base-2 exponentials with scale * log2(e) folded
//               in, row sums, P as bf16 written back over S in TMEM.  The
//               running max is only raised when a row's max grows by more
//               than 8 (a factor 256), and only then is the O row in TMEM
//               rescaled; the final O / l uses the same max, so the result is
//               exact.  Epilogue: O / l to bf16, one row per thread.
// Every wait is bounded: on a timeout the CTA records PA_ERR_TIMEOUT, drains
// what it issued, frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <cstring>
#include <mutex>

#include "pa_common.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace pa::sm100;

constexpr int D = pa::kHeadDim;
constexpr int BM = 128;             // queries per CTA (TMEM lanes)
constexpr int BN = 128;             // keys per tile
constexpr int STAGES = 2;
constexpr int NTHREADS = 256;
constexpr int HALF_BYTES = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte swizzle column block)
constexpr int TILE_BYTES = 2 * HALF_BYTES;  // 128 rows x 128 bf16
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;
constexpr int OFF_V = OFF_K + STAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_V + STAGES * TILE_BYTES;
enum {
    B_Q = 0,
    B_KF = 1,
    B_VF = B_KF + STAGES,
    B_KVE = B_VF + STAGES,
    B_SF = B_KVE + STAGES,
    B_PF = B_SF + 2,
    B_OD = B_PF + 2,
    B_DRAIN = B_OD + 1,
    NBAR = B_DRAIN + 1
};
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int SMEM_BYTES = OFF_MISC + 16 + 1024;  // + slack to align the base to 1024 bytes
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_S0 = 0, COL_S1 = 128, COL_O = 256;
constexpr long long WAIT_LIMIT = 1ll << 31;  // SM cycles (about a second)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units
constexpr unsigned FULL = 0xffffffffu;

struct TcParams {
    CUtensorMap kmap;  // paged pool, [num_blocks * block_size rows, Hkv * 128 cols]
    CUtensorMap vmap;
    const uint16_t *q;
    int64_t q_stride;
    const uint16_t *k;  // no-table path
    const uint16_t *v;
    int64_t kv_stride;
    const int32_t *block_table;
    int max_blocks;
    int block_size;
    int64_t num_blocks;
    int box_rows;
    const int32_t *cu_q;
    const int32_t *cu_k;
    int max_q;
    int n_mtiles;
    int num_heads;
    int kv_heads;
    float scale_log2;
    uint16_t *out;
    int32_t *status;
};

__device__ __forceinline__ uint32_t swz128(int row, int chunk)  // byte offset in a 128-row, 128-byte-row block
{
    return uint32_t(row * 128 + ((chunk ^ (row & 7)) << 4));
}

__global__ void __launch_bounds__(NTHREADS, 1) prefill_tc_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
    const uint32_t sb = smem_u32(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + OFF_MISC + 4);
    auto bar = [&](int i) { return sb + OFF_BAR + 8u * uint32_t(i); };

    const int b = blockIdx.z, h = blockIdx.y;
    const int mt = p.n_mtiles - 1 - int(blockIdx.x);  // the tiles with the most keys start first
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = p.cu_q[b], lq = p.cu_q[b + 1] - q0;
    const int k0 = p.cu_k[b], lk = p.cu_k[b + 1] - k0;
    const bool paged = p.block_table != nullptr;
    const bool bad_shape = lk < lq || (!paged && (lk != lq || k0 != q0)) ||
                           (paged && int64_t(lk) > int64_t(p.max_blocks) * p.block_size);
    if (blockIdx.x == 0 && h == 0 && threadIdx.x == 0) {
        if (bad_shape) pa::report(p.status, (lk < lq || !paged) ? PA_ERR_INVALID_ARG : PA_ERR_BOUNDS);
        else if (lq > p.max_q) pa::report(p.status, PA_ERR_BOUNDS);
    }
    if (lq <= 0 || mt * BM >= lq || bad_shape) return;

    const int g = h / (p.num_heads / p.kv_heads);
    const int m0 = mt * BM;
    const int rows = min(BM, lq - m0);
    const int offset = lk - lq;            // absolute position of query 0
    const int kend = offset + m0 + rows;   // keys visible to the tile's last row
    const int ntiles = (kend + BN - 1) / BN;

    if (threadIdx.x == 0) {
        mbar_init(bar(B_Q), 32);
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(bar(B_KF + s), paged ? 1 : 32);
            mbar_init(bar(B_VF + s), paged ? 1 : 32);
            mbar_init(bar(B_KVE + s), 1);
        }
        for (int s = 0; s < 2; ++s) {
            mbar_init(bar(B_SF + s), 1);
            mbar_init(bar(B_PF + s), 128);
        }
        mbar_init(bar(B_OD), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        bool bad = false;
        if (paged && lane == 0) {
            tma_prefetch_desc(&p.kmap);
            tma_prefetch_desc(&p.vmap);
        }
        for (int idx = lane; idx < BM * 16; idx += 32) {
            const int r = idx >> 4, c = idx & 15;
            const bool valid = r < rows;
            const uint16_t *src = valid ? p.q + int64_t(q0 + m0 + r) * p.q_stride + h * D + c * 8 : p.q;
            cp_async16(sb + OFF_Q + (c >> 3) * HALF_BYTES + swz128(r, c & 7), src, valid);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(bar(B_Q));

        int issued_upto = 0;  // tiles whose loads were issued
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % STAGES;
            if (j >= STAGES && !mbar_wait(bar(B_KVE + st), ((j / STAGES) - 1) & 1, abort_flag, WAIT_LIMIT)) break;
            const int j0 = j * BN;
            const uint32_t kdst = sb + OFF_K + st * TILE_BYTES, vdst = sb + OFF_V + st * TILE_BYTES;
            if (paged) {
                if (lane == 0) {
                    const int nbox = BN / p.box_rows;
                    const int32_t *table = p.block_table + int64_t(b) * p.max_blocks;
                    uint32_t bytes = 0;
                    for (int bx = 0; bx < nbox; ++bx) {
                        const int kb = j0 + bx * p.box_rows;
                        if (kb >= kend) break;
                        const int32_t phys = table[kb / p.block_size];
                        if (phys < 0 || int64_t(phys) >= p.num_blocks) { bad = true; continue; }
                        bytes += uint32_t(p.box_rows) * 128u * 2u;
                    }
                    mbar_arrive_expect_tx(bar(B_KF + st), bytes);
                    mbar_arrive_expect_tx(bar(B_VF + st), bytes);
                    for (int bx = 0; bx < nbox; ++bx) {
                        const int kb = j0 + bx * p.box_rows;
                        if (kb >= kend) break;
                        const int32_t phys = table[kb / p.block_size];
                        if (phys < 0 || int64_t(phys) >= p.num_blocks) continue;
                        const int y = int(int64_t(phys) * p.block_size + kb % p.block_size);
                        const uint32_t off = uint32_t(bx * p.box_rows * 128);
                        for (int hf = 0; hf < 2; ++hf) {
                            tma_load_2d(kdst + hf * HALF_BYTES + off, &p.kmap, g * D + hf * 64, y, bar(B_KF + st));
                            tma_load_2d(vdst + hf * HALF_BYTES + off, &p.vmap, g * D + hf * 64, y, bar(B_VF + st));
                        }
                    }
                }
                __syncwarp();
            } else {
                for (int idx = lane; idx < BN * 16; idx += 32) {
                    const int r = idx >> 4, c = idx & 15;
                    const bool valid = j0 + r < kend;
                    const int64_t row = int64_t(k0) + j0 + r;
                    const uint16_t *ks = valid ? p.k + row * p.kv_stride + g * D + c * 8 : p.q;
                    const uint16_t *vs = valid ? p.v + row * p.kv_stride + g * D + c * 8 : p.q;
                    const uint32_t o = (c >> 3) * HALF_BYTES + swz128(r, c & 7);
                    cp_async16(kdst + o, ks, valid);
                    cp_async16(vdst + o, vs, valid);
                }
                cp_async_wait_all();
                fence_proxy_async_smem();
                mbar_arrive(bar(B_KF + st));
                mbar_arrive(bar(B_VF + st));
            }
            issued_upto = j + 1;
        }
        if (bad && lane == 0) pa::report(p.status, PA_ERR_BOUNDS);
        if (*abort_flag && paged && lane == 0) {
            // let copies already in flight land before the CTA's shared memory goes away
            for (int j = max(0, issued_upto - STAGES); j < issued_upto; ++j) {
                volatile int32_t dummy = 0;
                mbar_wait(bar(B_KF + j % STAGES), (j / STAGES) & 1, &dummy, WAIT_LIMIT);
                mbar_wait(bar(B_VF + j % STAGES), (j / STAGES) & 1, &dummy, WAIT_LIMIT);
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
            constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, 0, 1);   // P from TMEM, V MN-major
            bool ok = mbar_wait(bar(B_Q), 0, abort_flag, WAIT_LIMIT);
            tc_fence_after();
            for (int j = 0; ok && j <= ntiles; ++j) {
                if (j < ntiles) {
                    const int st = j % STAGES;
                    if (!(ok = mbar_wait(bar(B_KF + st), (j / STAGES) & 1, abort_flag, WAIT_LIMIT))) break;
                    tc_fence_after();
                    const uint32_t d = tmem + ((j & 1) ? COL_S1 : COL_S0);
#pragma unroll
                    for (int kk = 0; kk < D / 16; ++kk) {
                        const uint32_t hf = kk >> 2, ko = (kk & 3) * 32;
                        const uint64_t a = smem_desc(sb + OFF_Q + hf * HALF_BYTES + ko, 16, 1024);
                        const uint64_t bk = smem_desc(sb + OFF_K + st * TILE_BYTES + hf * HALF_BYTES + ko, 16, 1024);
                        mma_ss(d, a, bk, IDESC_QK, kk > 0);
                    }
                    mma_commit(bar(B_SF + (j & 1)));
                }
                if (j >= 1) {
                    const int jp = j - 1, sp = jp % STAGES;
                    if (!(ok = mbar_wait(bar(B_PF + (jp & 1)), (jp >> 1) & 1, abort_flag, WAIT_LIMIT))) break;
                    if (!(ok = mbar_wait(bar(B_VF + sp), (jp / STAGES) & 1, abort_flag, WAIT_LIMIT))) break;
                    tc_fence_after();
                    const uint32_t pcol = tmem + ((jp & 1) ? COL_S1 : COL_S0);
#pragma unroll
                    for (int s = 0; s < BN / 16; ++s) {
                        const uint64_t bv = smem_desc(sb + OFF_V + sp * TILE_BYTES + s * 2048, HALF_BYTES, 1024);
                        mma_ts(tmem + COL_O, pcol + s * 8, bv, IDESC_PV, (jp > 0 || s > 0) ? 1u : 0u);
                    }
                    mma_commit(bar(B_KVE + sp));
                    mma_commit(bar(B_OD));
                }
            }
            if (!ok) {
                // wait for the MMAs already issued before TMEM and shared memory are released
                volatile int32_t dummy = 0;
                mma_commit(bar(B_DRAIN));
                mbar_wait(bar(B_DRAIN), 0, &dummy, WAIT_LIMIT);
            }
        }
        __syncwarp();
    } else if (warp >= 4) {
        // ------------------------------------------------------------ softmax + epilogue
        const int quarter = warp - 4;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = uint32_t(quarter * 32) << 16;
        const int pos = offset + m0 + r;
        const int last_visible = min(pos, kend - 1);
        float m_used = -INFINITY, l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            ok = __all_sync(FULL, mbar_wait(bar(B_SF + (j & 1)), (j >> 1) & 1, abort_flag, WAIT_LIMIT));
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = tmem + lane_base + ((j & 1) ? COL_S1 : COL_S0);
            uint32_t sr[4][32];
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) tmem_ld32(scol + cc * 32, sr[cc]);
            tmem_ld_wait();
            const int j0 = j * BN;
            const bool mask = j0 + BN - 1 > offset + m0;
            const int limit = last_visible - j0;
            float mx = -INFINITY;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    float s = __uint_as_float(sr[cc][i]) * p.scale_log2;
                    if (mask && cc * 32 + i > limit) s = -INFINITY;
                    sr[cc][i] = __float_as_uint(s);
                    mx = fmaxf(mx, s);
                }
            }
            const bool need = mx > m_used + RESCALE_THRESHOLD;
            const float m_new = need ? mx : m_used;
            const float factor = need ? exp2f(m_used - m_new) : 1.f;
            if (j > 0 && __any_sync(FULL, need)) {
                ok = __all_sync(FULL, mbar_wait(bar(B_OD), (j - 1) & 1, abort_flag, WAIT_LIMIT));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32(tmem + lane_base + COL_O + cc * 32, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
                    tmem_st32(tmem + lane_base + COL_O + cc * 32, o);
                }
                tmem_st_wait();
            }
            l *= factor;
            m_used = m_new;
            const float msub = (m_used == -INFINITY) ? 0.f : m_used;
            float rs = 0.f;
#pragma unroll
            for (int hf = 0; hf < 2; ++hf) {
                uint32_t pk[32];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    const int c0 = hf * 64 + 2 * i;
                    const float p0 = exp2f(__uint_as_float(sr[c0 >> 5][c0 & 31]) - msub);
                    const float p1 = exp2f(__uint_as_float(sr[(c0 + 1) >> 5][(c0 + 1) & 31]) - msub);
                    rs += p0 + p1;
                    pk[i] = pa::pack_bf16x2(p0, p1);
                }
                tmem_st32(scol + hf * 32, pk);
            }
            l += rs;
            if (paged && j == ntiles - 1 && kend < j0 + BN) {
                // rows past the last visible key may be unused pool slots (any bits): make them 0
                // so that 0 * V stays 0 in P.V
                const int st = j % STAGES;
                if (!(ok = mbar_wait(bar(B_VF + st), (j / STAGES) & 1, abort_flag, WAIT_LIMIT))) break;
                if (j0 + r >= kend) {
                    uint4 *row0 = reinterpret_cast<uint4 *>(smem + OFF_V + st * TILE_BYTES + r * 128);
                    uint4 *row1 = reinterpret_cast<uint4 *>(smem + OFF_V + st * TILE_BYTES + HALF_BYTES + r * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) row0[c] = row1[c] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tmem_st_wait();
            tc_fence_before();
            mbar_arrive(bar(B_PF + (j & 1)));
        }
        if (ok) ok = __all_sync(FULL, mbar_wait(bar(B_OD), (ntiles - 1) & 1, abort_flag, WAIT_LIMIT));
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            uint16_t *dst = p.out + (int64_t(q0 + m0 + r) * p.num_heads + h) * D;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32(tmem + lane_base + COL_O + cc * 32, o);
                tmem_ld_wait();
                if (r < rows) {
                    uint4 *d4 = reinterpret_cast<uint4 *>(dst + cc * 32);
#pragma unroll
                    for (int v = 0; v < 4; ++v) {
                        uint4 u;
                        u.x = pa::pack_bf16x2(__uint_as_float(o[8 * v + 0]) * inv, __uint_as_float(o[8 * v + 1]) * inv);
                        u.y = pa::pack_bf16x2(__uint_as_float(o[8 * v + 2]) * inv, __uint_as_float(o[8 * v + 3]) * inv);
                        u.z = pa::pack_bf16x2(__uint_as_float(o[8 * v + 4]) * inv, __uint_as_float(o[8 * v + 5]) * inv);
                        u.w = pa::pack_bf16x2(__uint_as_float(o[8 * v + 6]) * inv, __uint_as_float(o[8 * v + 7]) * inv);
                        d4[v] = u;
                    }
                }
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) pa::report(p.status, PA_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn()
{
    static std::once_flag once;
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

bool make_pool_map(CUtensorMap *map, const void *base, int64_t rows, int kv_heads, int box_rows)
{
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cuuint64_t(kv_heads) * D, cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(kv_heads) * D * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gcd(int a, int b) { return b == 0 ? a : gcd(b, a % b); }

}  // namespace

extern "C" pa_status pa_prefill_paged(const void *q, int64_t q_stride_tok, const void *k, const void *v,
                                      int64_t kv_stride_tok, const void *k_cache, const void *v_cache,
                                      int64_t num_blocks, int block_size, const int32_t *block_table,
                                      int max_blocks_per_seq, const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_k, int num_seqs, int max_seqlen_q,
                                      int max_seqlen_k, int num_heads, int num_kv_heads, int head_dim,
                                      float scale, void *out, int32_t *dev_status, void *stream)
{
    if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (head_dim != D || !pa::pow2_in(num_kv_heads, 1, 8) || num_heads <= 0 || num_heads % num_kv_heads != 0 ||
        !pa::pow2_in(num_heads / num_kv_heads, 1, 8))
        return PA_ERR_UNSUPPORTED;
    if (block_table != nullptr && (block_size < 16 || block_size > 1024 || block_size % 16 != 0))
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_seqlen_q == 0) return PA_OK;
    if (!q || !cu_seqlens_q || !cu_seqlens_k || !out) return PA_ERR_INVALID_ARG;
    if (q_stride_tok < int64_t(num_heads) * D || q_stride_tok % 8 != 0 || !pa::aligned(q, 16))
        return PA_ERR_INVALID_ARG;
    if (!pa::aligned(out, 16)) return PA_ERR_INVALID_ARG;
    if (block_table == nullptr) {
        if (!k || !v || max_seqlen_k != max_seqlen_q) return PA_ERR_INVALID_ARG;
        if (kv_stride_tok < int64_t(num_kv_heads) * D || kv_stride_tok % 8 != 0 || !pa::aligned(k, 16) ||
            !pa::aligned(v, 16))
            return PA_ERR_INVALID_ARG;
    } else {
        if (!k_cache || !v_cache || max_blocks_per_seq < 1 || num_blocks < 1) return PA_ERR_INVALID_ARG;
        if (!pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
        if (num_blocks * block_size >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
    }
    if (num_seqs > 65535 || num_heads > 65535) return PA_ERR_UNSUPPORTED;

    TcParams p;
    memset(&p, 0, sizeof(p));
    p.q = static_cast<const uint16_t *>(q);
    p.q_stride = q_stride_tok;
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.kv_stride = kv_stride_tok;
    p.block_table = block_table;
    p.max_blocks = max_blocks_per_seq;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.box_rows = block_table ? gcd(block_size, BN) : BN;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.max_q = max_seqlen_q;
    p.n_mtiles = (max_seqlen_q + BM - 1) / BM;
    p.num_heads = num_heads;
    p.kv_heads = num_kv_heads;
    p.scale_log2 = scale * LOG2E;
    p.out = static_cast<uint16_t *>(out);
    p.status = dev_status;
    if (block_table != nullptr) {
        const int64_t rows = num_blocks * block_size;
        if (!make_pool_map(&p.kmap, k_cache, rows, num_kv_heads, p.box_rows) ||
            !make_pool_map(&p.vmap, v_cache, rows, num_kv_heads, p.box_rows))
            return PA_ERR_CUDA;
    }
    static std::once_flag attr_once;
    static cudaError_t attr_err = cudaSuccess;
    std::call_once(attr_once, [] {
        attr_err = cudaFuncSetAttribute(prefill_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES);
    });
    if (attr_err != cudaSuccess) return PA_ERR_CUDA;
    const dim3 grid(unsigned(p.n_mtiles), unsigned(num_heads), unsigned(num_seqs));
    prefill_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(p);
    return pa::launch_status();
}
