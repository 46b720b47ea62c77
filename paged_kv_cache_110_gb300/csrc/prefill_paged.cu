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
//   warps 0, 2  producers: warp 0 the Q tile (cp.async) and K, warp 2 V.  Paged keys arrive by TMA, one box per page run: the box
//               height is gcd(block_size, 128) rows, so a box never crosses a
//               page; without a table, rows are copied with cp.async.  All
//               tiles land in shared memory in the 128-byte-swizzled layout
//               the tensor cores read.  Three K stages (a K tile is released
//               as soon as its S is computed) and two V stages; K runs one
//               tile ahead of V.
//   warp 1      MMA issuer (one thread): S_j = Q K_j^T into one of three TMEM
//               S buffers (M = N = 128, K = 128 in eight K = 16 steps), and
//               O += P_j V_j with P read from TMEM, issued from a polling
//               loop so S runs up to three tiles ahead of P.V.  An S buffer
//               is reused only after the P.V that reads its P has completed
//               (tensor-core reads and writes of one TMEM region by
//               different MMAs are ordered explicitly).
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
constexpr int KSTAGES = 2;          // K tiles in flight (released as soon as S = Q K^T is done)
constexpr int VSTAGES = 4;          // V tiles in flight (released after O += P V, so kept longer)
constexpr int SBUF = 3;             // TMEM S buffers (P is written back over S)
constexpr int NTHREADS = 256;
constexpr int HALF_BYTES = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte swizzle column block)
constexpr int TILE_BYTES = 2 * HALF_BYTES;  // 128 rows x 128 bf16
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + TILE_BYTES;
constexpr int OFF_V = OFF_K + KSTAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_V + VSTAGES * TILE_BYTES;
enum {
    B_Q = 0,
    B_KF = 1,
    B_KE = B_KF + KSTAGES,
    B_VF = B_KE + KSTAGES,
    B_VE = B_VF + VSTAGES,
    B_SF = B_VE + VSTAGES,
    B_PF = B_SF + SBUF,
    B_SFREE = B_PF + SBUF,
    B_OFIN = B_SFREE + SBUF,
    B_DRAIN = B_OFIN + 1,
    NBAR = B_DRAIN + 1
};
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;
constexpr int TABLE_SMEM = 512;                   // block-table entries staged in shared memory
constexpr int OFF_TABLE = OFF_MISC + 16;
constexpr int SMEM_BYTES = OFF_TABLE + TABLE_SMEM * 4;  // the base is 1024-byte aligned (checked)
constexpr uint32_t TMEM_COLS = 512;
constexpr uint32_t COL_O = 384;     // S buffers at columns 0, 128, 256
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

// Where one producer warp reads a tile from: the TMA map of the paged pool
// (with the sequence's block ids, staged in shared memory when they fit; -1
// marks an id that failed validation), or the new-token rows when there is
// no table.
struct TileSource {
    const CUtensorMap *map;  // paged
    const int32_t *table;    // paged
    int box_rows;
    int block_size;
    const uint16_t *rows;    // no table: first row of the sequence, head g
    int64_t stride;          // no table: row stride in elements
    const uint16_t *dummy;   // any mapped address (zero-byte cp.async source)
};

// Issue the loads of the 128-key tile starting at key j0 into `dst`,
// arriving on `bar`.  Paged: lane 0 issues one TMA box per page run; boxes
// at or past kend and boxes on invalid ids are skipped.  No table: the 32
// lanes copy rows with cp.async (rows past kend zero-filled) and then arrive.
__device__ __forceinline__ void load_tile(const TileSource &src, int xcol, int j0, int kend, uint32_t dst,
                                          uint32_t bar, int lane)
{
    if (src.map != nullptr) {
        if (lane == 0) {
            const int nbox = BN / src.box_rows;
            uint32_t bytes = 0;
            for (int bx = 0; bx < nbox; ++bx) {
                const int kb = j0 + bx * src.box_rows;
                if (kb >= kend) break;
                if (src.table[kb / src.block_size] >= 0) bytes += uint32_t(src.box_rows) * 128u * 2u;
            }
            mbar_arrive_expect_tx(bar, bytes);
            for (int bx = 0; bx < nbox; ++bx) {
                const int kb = j0 + bx * src.box_rows;
                if (kb >= kend) break;
                const int32_t phys = src.table[kb / src.block_size];
                if (phys < 0) continue;
                const int y = int(int64_t(phys) * src.block_size + kb % src.block_size);
                const uint32_t off = uint32_t(bx * src.box_rows * 128);
                tma_load_2d(dst + off, src.map, xcol, y, bar);
                tma_load_2d(dst + HALF_BYTES + off, src.map, xcol + 64, y, bar);
            }
        }
        __syncwarp();
    } else {
        for (int idx = lane; idx < BN * 16; idx += 32) {
            const int r = idx >> 4, c = idx & 15;
            const bool valid = j0 + r < kend;
            const uint16_t *ptr = valid ? src.rows + int64_t(j0 + r) * src.stride + c * 8 : src.dummy;
            cp_async16(dst + (c >> 3) * HALF_BYTES + swz128(r, c & 7), ptr, valid);
        }
        cp_async_wait_all();
        fence_proxy_async_smem();
        mbar_arrive(bar);
    }
}

__global__ void __launch_bounds__(NTHREADS, 1) prefill_tc_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ __align__(1024) uint8_t smem_raw[];
    uint8_t *smem = smem_raw;
    const uint32_t sb = smem_u32(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + OFF_MISC + 4);
    auto bar = [&](int i) { return sb + OFF_BAR + 8u * uint32_t(i); };

    // CTAs launch in blockIdx.x-fastest order: x walks (head, sequence) and y
    // the query tile from the last one down, so across the whole batch the
    // tiles with the most keys start first
    const int h = int(blockIdx.x) % p.num_heads, b = int(blockIdx.x) / p.num_heads;
    const int mt = p.n_mtiles - 1 - int(blockIdx.y);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = p.cu_q[b], lq = p.cu_q[b + 1] - q0;
    const int k0 = p.cu_k[b], lk = p.cu_k[b + 1] - k0;
    const bool paged = p.block_table != nullptr;
    const bool bad_shape = lk < lq || (!paged && (lk != lq || k0 != q0)) ||
                           (paged && int64_t(lk) > int64_t(p.max_blocks) * p.block_size);
    if (blockIdx.y == 0 && h == 0 && threadIdx.x == 0) {
        if (bad_shape) pa::report(p.status, (lk < lq || !paged) ? PA_ERR_INVALID_ARG : PA_ERR_BOUNDS);
        else if (lq > p.max_q) pa::report(p.status, PA_ERR_BOUNDS);
    }
    if (lq <= 0 || mt * BM >= lq || bad_shape) return;

    // the 128-byte swizzle pattern of TMA and the tensor cores is anchored at 1024-byte boundaries
    if ((smem_u32(smem) & 1023u) != 0) {
        if (threadIdx.x == 0) pa::report(p.status, PA_ERR_UNSUPPORTED);
        return;
    }
    const int g = h / (p.num_heads / p.kv_heads);
    const int m0 = mt * BM;
    const int rows = min(BM, lq - m0);
    const int offset = lk - lq;            // absolute position of query 0
    const int kend = offset + m0 + rows;   // keys visible to the tile's last row
    const int ntiles = (kend + BN - 1) / BN;

    if (threadIdx.x == 0) {
        const uint32_t loader_count = paged ? 1 : 32;
        mbar_init(bar(B_Q), 32);
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(bar(B_KF + s), loader_count);
            mbar_init(bar(B_KE + s), 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
            mbar_init(bar(B_VF + s), loader_count);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int s = 0; s < SBUF; ++s) {
            mbar_init(bar(B_SF + s), 1);
            mbar_init(bar(B_PF + s), 128);
            mbar_init(bar(B_SFREE + s), 1);
        }
        mbar_init(bar(B_OFIN), 1);
        mbar_init(bar(B_DRAIN), 1);
        *abort_flag = 0;
        fence_barrier_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_holder), TMEM_COLS);
        tmem_relinquish();
    }
    // Stage the sequence's block ids (validated) in shared memory, so that
    // issuing a tile never waits on a global load.
    const int nblk = paged ? (kend + p.block_size - 1) / p.block_size : 0;
    const bool table_in_smem = paged && nblk <= TABLE_SMEM;
    if (paged && (warp == 2 || warp == 3)) {
        const int32_t *gtable = p.block_table + int64_t(b) * p.max_blocks;
        int32_t *st = reinterpret_cast<int32_t *>(smem + OFF_TABLE);
        bool bad = false;
        for (int i = threadIdx.x - 64; i < nblk; i += 64) {
            int32_t phys = gtable[i];
            if (phys < 0 || int64_t(phys) >= p.num_blocks) {
                bad = true;
                phys = -1;
            }
            if (table_in_smem) st[i] = phys;
        }
        if (bad) pa::report(p.status, PA_ERR_BOUNDS);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_holder;

    TileSource src;
    src.table = table_in_smem ? reinterpret_cast<const int32_t *>(smem + OFF_TABLE)
                              : (paged ? p.block_table + int64_t(b) * p.max_blocks : nullptr);
    src.box_rows = p.box_rows;
    src.block_size = p.block_size;
    src.stride = p.kv_stride;
    src.dummy = p.q;
    if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers
        // warp 0: K_0, then Q, then K_1.. (a K stage is reused once the S that
        // read it is done); warp 2: V_0, V_1.. (a V stage is reused once the
        // P.V that read it is done).  Two warps, so K and V issue overlap.
        const bool is_k = warp == 0;
        src.map = paged ? (is_k ? &p.kmap : &p.vmap) : nullptr;
        src.rows = paged ? nullptr : (is_k ? p.k : p.v) + int64_t(k0) * p.kv_stride + g * D;
        if (paged && lane == 0) tma_prefetch_desc(src.map);
        const int nst = is_k ? KSTAGES : VSTAGES;
        const uint32_t base = sb + (is_k ? OFF_K : OFF_V);
        const int full0 = is_k ? B_KF : B_VF, empty0 = is_k ? B_KE : B_VE;
        int issued = 0;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int st = j % nst;
            if (j >= nst && !(ok = mbar_wait(bar(empty0 + st), ((j / nst) - 1) & 1, abort_flag, WAIT_LIMIT))) break;
            load_tile(src, g * D, j * BN, kend, base + st * TILE_BYTES, bar(full0 + st), lane);
            issued = j + 1;
            if (is_k && j == 0) {
                for (int idx = lane; idx < BM * 16; idx += 32) {
                    const int r = idx >> 4, c = idx & 15;
                    const bool valid = r < rows;
                    const uint16_t *qp = valid ? p.q + int64_t(q0 + m0 + r) * p.q_stride + h * D + c * 8 : p.q;
                    cp_async16(sb + OFF_Q + (c >> 3) * HALF_BYTES + swz128(r, c & 7), qp, valid);
                }
                cp_async_wait_all();
                fence_proxy_async_smem();
                mbar_arrive(bar(B_Q));
            }
        }
        (void)ok;
        if (*abort_flag && paged && lane == 0) {
            // let copies already in flight land before the CTA's shared memory goes away
            volatile int32_t dummy = 0;
            for (int j = max(0, issued - nst); j < issued; ++j)
                mbar_wait(bar(full0 + j % nst), (j / nst) & 1, &dummy, WAIT_LIMIT);
        }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // A polling state machine: S_j is issued as soon as K_j is in and its
        // TMEM buffer is free (the P.V of tile j - SBUF has completed), and
        // P.V_j as soon as P_j and V_j are in, so S runs up to SBUF tiles ahead
        // of P.V and a late V tile does not hold back the softmax.
        if (lane == 0) {
            constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
            constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, 0, 1);   // P from TMEM, V MN-major
            bool ok = mbar_wait(bar(B_Q), 0, abort_flag, WAIT_LIMIT);
            int ns = 0, npv = 0;  // next S tile, next P.V tile
            long long t0 = clock64();
            while (ok && npv < ntiles) {
                bool progressed = false;
                if (ns < ntiles && ns - npv < SBUF) {
                    const int st = ns % KSTAGES, sbuf = ns % SBUF;
                    if (mbar_poll(bar(B_KF + st), (ns / KSTAGES) & 1) &&
                        (ns < SBUF || mbar_poll(bar(B_SFREE + sbuf), ((ns / SBUF) - 1) & 1))) {
                        tc_fence_after();
                        const uint32_t d = tmem + uint32_t(sbuf) * 128u;
#pragma unroll
                        for (int kk = 0; kk < D / 16; ++kk) {
                            const uint32_t hf = kk >> 2, ko = (kk & 3) * 32;
                            const uint64_t a = smem_desc(sb + OFF_Q + hf * HALF_BYTES + ko, 16, 1024);
                            const uint64_t bk = smem_desc(sb + OFF_K + st * TILE_BYTES + hf * HALF_BYTES + ko, 16, 1024);
                            mma_ss(d, a, bk, IDESC_QK, kk > 0);
                        }
                        mma_commit(bar(B_SF + sbuf));
                        mma_commit(bar(B_KE + st));
                        ++ns;
                        progressed = true;
                    }
                }
                if (npv < ns) {
                    const int sv = npv % VSTAGES, pbuf = npv % SBUF;
                    if (mbar_poll(bar(B_PF + pbuf), (npv / SBUF) & 1) && mbar_poll(bar(B_VF + sv), (npv / VSTAGES) & 1)) {
                        tc_fence_after();
                        const uint32_t pcol = tmem + uint32_t(pbuf) * 128u;
#pragma unroll
                        for (int s = 0; s < BN / 16; ++s) {
                            const uint64_t bv = smem_desc(sb + OFF_V + sv * TILE_BYTES + s * 2048, HALF_BYTES, 1024);
                            mma_ts(tmem + COL_O, pcol + s * 8, bv, IDESC_PV, (npv > 0 || s > 0) ? 1u : 0u);
                        }
                        mma_commit(bar(B_VE + sv));
                        mma_commit(bar(B_SFREE + pbuf));
                        if (npv == ntiles - 1) mma_commit(bar(B_OFIN));
                        ++npv;
                        progressed = true;
                    }
                }
                if (progressed) {
                    t0 = clock64();
                } else if (__nanosleep(20), *abort_flag) {  // yield issue slots to the softmax warp on this SMSP
                    ok = false;
                } else if (clock64() - t0 > WAIT_LIMIT) {
                    *abort_flag = 1;
                    ok = false;
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
        const float sl2 = p.scale_log2;
        float m_used = -INFINITY;  // running max in scaled base-2 units
        float l = 0.f;
        bool ok = true;
        for (int j = 0; j < ntiles; ++j) {
            const int sbuf = j % SBUF;
            ok = __all_sync(FULL, mbar_wait(bar(B_SF + sbuf), (j / SBUF) & 1, abort_flag, WAIT_LIMIT));
            if (!ok) break;
            tc_fence_after();
            const uint32_t scol = tmem + lane_base + uint32_t(sbuf) * 128u;
            uint32_t sr[128];
            tmem_ld128_sync(scol, sr);
            const int j0 = j * BN;
            if (j0 + BN - 1 > offset + m0) {  // the tile crosses some row's causal bound
                const int limit = last_visible - j0;
#pragma unroll
                for (int c = 0; c < 128; ++c)
                    if (c > limit) sr[c] = 0xff800000u;  // -inf
            }
            // raw row max with 8 independent three-input max chains
            float mx8[8];
#pragma unroll
            for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[8 + k]));
#pragma unroll
            for (int c = 16; c < 128; c += 16) {
#pragma unroll
                for (int k = 0; k < 8; ++k)
                    mx8[k] = fmax3(mx8[k], __uint_as_float(sr[c + k]), __uint_as_float(sr[c + 8 + k]));
            }
            const float mx = fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * sl2;
            const bool need = mx > m_used + RESCALE_THRESHOLD;
            const float m_new = need ? mx : m_used;
            const float factor = need ? ex2_approx(m_used - m_new) : 1.f;
            if (j > 0 && __any_sync(FULL, need)) {
                // O must hold P.V_{j-1} before it is rescaled.  Its completion is
                // tracked by the free barrier of that tile's S buffer; the S_j
                // commit already implies P.V_{j-1-SBUF}.. so that barrier is at
                // most one phase behind the one awaited.
                ok = __all_sync(FULL, mbar_wait(bar(B_SFREE + (j - 1) % SBUF), ((j - 1) / SBUF) & 1, abort_flag,
                                                WAIT_LIMIT));
                if (!ok) break;
                tc_fence_after();
#pragma unroll
                for (int cc = 0; cc < 4; ++cc) {
                    uint32_t o[32];
                    tmem_ld32_sync(tmem + lane_base + COL_O + cc * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * factor);
                    tmem_st32_sync(tmem + lane_base + COL_O + cc * 32, o);
                }
            }
            l *= factor;
            m_used = m_new;
            const float nm = (m_used == -INFINITY) ? 0.f : -m_used;
            // p = 2^(s * scale * log2 e - m): paired FMAs, MUFU exponentials, paired sums
            float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
            uint32_t pk[64];
#pragma unroll
            for (int i = 0; i < 64; ++i) {
                float x0, x1;
                ffma2(x0, x1, __uint_as_float(sr[2 * i]), __uint_as_float(sr[2 * i + 1]), sl2, sl2, nm, nm);
                const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                fadd2(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], p0, p1);
                pk[i] = pa::pack_bf16x2(p0, p1);
            }
            l += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
            if (paged && j == ntiles - 1 && kend < j0 + BN) {
                // rows past the last visible key may be unused pool slots (any bits): make them 0
                // so that 0 * V stays 0 in P.V
                const int sv = j % VSTAGES;
                ok = __all_sync(FULL, mbar_wait(bar(B_VF + sv), (j / VSTAGES) & 1, abort_flag, WAIT_LIMIT));
                if (!ok) break;
                if (j0 + r >= kend) {
                    uint4 *row0 = reinterpret_cast<uint4 *>(smem + OFF_V + sv * TILE_BYTES + r * 128);
                    uint4 *row1 = reinterpret_cast<uint4 *>(smem + OFF_V + sv * TILE_BYTES + HALF_BYTES + r * 128);
#pragma unroll
                    for (int c = 0; c < 8; ++c) row0[c] = row1[c] = make_uint4(0, 0, 0, 0);
                }
                fence_proxy_async_smem();
            }
            tmem_st64_sync(scol, pk);
            tc_fence_before();
            mbar_arrive(bar(B_PF + sbuf));
        }
        // The final O waits on its own single-use barrier: several P.V may still
        // be in flight here, so a parity wait on a per-tile barrier could
        // alias an older phase.
        if (ok) ok = __all_sync(FULL, mbar_wait(bar(B_OFIN), 0, abort_flag, WAIT_LIMIT));
        if (ok) {
            tc_fence_after();
            const float inv = 1.f / l;
            uint16_t *dst = p.out + (int64_t(q0 + m0 + r) * p.num_heads + h) * D;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) {
                uint32_t o[32];
                tmem_ld32_sync(tmem + lane_base + COL_O + cc * 32, o);
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
    if (int64_t(num_seqs) * num_heads > 0x7fffffff || (max_seqlen_q + BM - 1) / BM > 65535) return PA_ERR_UNSUPPORTED;

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
    const dim3 grid(unsigned(num_heads * num_seqs), unsigned(p.n_mtiles));
    prefill_tc_kernel<<<grid, NTHREADS, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(p);
    return pa::launch_status();
}
