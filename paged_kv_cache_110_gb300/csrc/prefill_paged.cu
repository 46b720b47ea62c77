// prefill_paged.cu -- causal varlen prefill over a block-paged KV cache with
// Blackwell tensor cores (tcgen05, accumulators in TMEM) and TMA page gathers.
//
// What it computes ("大模型推理入门与 nano-vLLM 源码详解" §11.2, §10.2, §13.3):
// sequence b has Lq new queries that are the last Lq positions of its Lk-key
// context; query i (absolute position p = Lk - Lq + i) reads keys 0..p.  Keys
// come from the paged pool through block_table (a cached prefix or an earlier
// chunk) or, without a table, from the new-token k / v rows.  Query head h
// reads KV head h / (Hq / Hkv) (§19.6).  Softmax is accumulated blockwise with
// a running max, a running sum and an unnormalised numerator (§13.3).
//
// A persistent kernel: one CTA per SM; the valid work items, heaviest first,
// are dealt to the CTAs statically in snake order (CTA c of C takes the
// valid items of rank c, 2C - 1 - c, 2C + c, ...), so that no counter in
// device memory is needed: every CTA ranks the items itself, 32 at a time.  An item is a PAIR of 128-row query tiles that read the same
// keys: the same rows of two query heads of one KV group (GQA), or, when every
// KV head has a single query head, two consecutive row tiles of one head.
// Each K and V tile is loaded once for both, and while one tile's softmax runs
// the tensor cores work on the other's, so the two dependency chains
// (S -> softmax -> P.V) hide each other.
//   warp 3      scheduler: walks this CTA's items, decodes each once and
//               publishes it in a ring of 4, stages its block ids (validated)
//               and loads its two Q tiles by TMA into two Q buffers.
//   warp 0      K producer, warp 2 V producer: paged tiles arrive by TMA, one
//               box per page run (box height gcd(block_size, 128) rows, so a
//               box never crosses a page); without a table one box of 128
//               token rows.  Tiles land in shared memory in the
//               128-byte-swizzled layout the tensor cores read; two stages
//               each.  Rows a tile holds beyond a sequence (the next
//               sequence's rows, TMA zero fill, unused pool slots) are masked
//               out of S, and the V rows of the item's last tile past its last
//               key are set to zero before P.V, so that they add 0.
//   warp 1      MMA issuer (the warp runs the loop, one elected lane issues):
//               per K/V tile j, O_0 += P_0 V_j (keys 0-63 as soon as their P is
//               written, then 64-127) then S_0 = Q_0 K_{j+1}^T, then the same
//               for query tile 1.  S and O of each query tile live in TMEM (S
//               at columns 0 / 128, O at 256 / 384); P is written back over S,
//               and the next S is issued after the P.V that reads P (tcgen05
//               operations run in order).
//   warps 4-7, 8-11   softmax of query tile 0 and 1, one thread per row: read
//               the S row from TMEM once, mask (causal, bottom-right, keys past
//               the last visible key), row max, base-2 exponentials with
//               scale * log2(e) folded into paired FMAs, row sums, P as bf16
//               over S.  The running max is raised only when a row max grows
//               by more than 8 (a factor 256), and only then is the O row
//               rescaled in TMEM; O / l uses the same max, so the result is
//               exact.  Epilogue: O / l to bf16, one row per thread.
// Every wait is bounded: on a timeout the CTA records PA_ERR_TIMEOUT, drains
// what it issued (TMA loads of Q, K and V, and MMAs), frees its TMEM and exits.
#include <cudaTypedefs.h>

#include <algorithm>
#include <atomic>
#include <cstring>
#include <mutex>

#include "pa_common.cuh"
#include "sm100_ptx.cuh"

namespace {

using namespace pa::sm100;

constexpr int D = pa::kHeadDim;
constexpr int BM = 128;             // query rows per query tile (TMEM lanes)
constexpr int QT = 2;               // query tiles per work item, sharing every K/V tile
constexpr int BN = 128;             // keys per tile
constexpr int KSTAGES = 2;          // K tiles in flight
constexpr int VSTAGES = 2;          // V tiles in flight
constexpr int QSLOTS = 2;           // Q tile buffers: one item's pair
constexpr int RING = 4;             // work items fetched ahead by the scheduler warp
constexpr int NTHREADS = 384;
constexpr uint32_t REGS_CONTROL = 136;  // per thread, warps 0-3 (one warpgroup)
constexpr uint32_t REGS_SOFTMAX = 184;  // per thread, warps 4-11
constexpr int HALF_BYTES = 128 * 128;       // 128 rows x 64 bf16 (one 128-byte swizzle column block)
constexpr int TILE_BYTES = 2 * HALF_BYTES;  // 128 rows x 128 bf16
constexpr int OFF_Q = 0;
constexpr int OFF_K = OFF_Q + QSLOTS * TILE_BYTES;
constexpr int OFF_V = OFF_K + KSTAGES * TILE_BYTES;
constexpr int OFF_BAR = OFF_V + VSTAGES * TILE_BYTES;
enum {
    B_QF = 0,                    // Q buffer loaded (TMA transaction bytes)
    B_QE = B_QF + QSLOTS,        // Q buffer free (its tile's last S done)
    B_KF = B_QE + QSLOTS,        // K stage loaded
    B_KE = B_KF + KSTAGES,       // K stage free (every S reading it done)
    B_VF = B_KE + KSTAGES,       // V stage loaded
    B_VE = B_VF + VSTAGES,       // V stage free (every P.V reading it done)
    B_SF = B_VE + VSTAGES,       // S of query tile a computed, per a
    B_PF = B_SF + QT,            // P of query tile a written over its S (128 arrivals), per a
    B_PL = B_PF + QT,            // its first half (keys 0-63) written (128 arrivals), per a
    B_OF = B_PL + QT,            // O of query tile a complete for the item, per a
    B_TF = B_OF + QT,            // block-id buffer staged (32 arrivals)
    B_TE = B_TF + 2,             // block-id buffer free (both producers done, 2 arrivals)
    B_IRF = B_TE + 2,            // item-ring slot published (1 arrival)
    B_IRE = B_IRF + RING,        // item-ring slot read by every role (11 arrivals)
    B_DRAIN = B_IRE + RING,
    B_STALL = B_DRAIN + 1,       // never arrived on: the wait a test makes run out
    NBAR = B_STALL + 1
};
constexpr int IR_READERS = 2 + 1 + 8;             // producer warps, MMA warp, softmax warps
constexpr int OFF_MISC = OFF_BAR + NBAR * 8;      // TMEM address, abort flag
constexpr int OFF_RING = OFF_MISC + 16;           // the item ring (RingSlot x RING)
constexpr int RING_SLOT_BYTES = 96;
constexpr int TABLE_SMEM = 256;                   // block ids staged per item (more: read from global)
constexpr int OFF_TABLE = OFF_RING + RING * RING_SLOT_BYTES;  // two buffers
constexpr int SMEM_BYTES = OFF_TABLE + 2 * TABLE_SMEM * 4;  // the base is 1024-byte aligned (checked)
static_assert(SMEM_BYTES <= 227 * 1024, "shared memory per CTA");
constexpr uint32_t TMEM_COLS = 512;                  // S of tiles 0 / 1 at 0 / 128, O at 256 / 384
constexpr uint32_t COL_O = 256;
constexpr long long WAIT_LIMIT = 1ll << 31;  // SM cycles (about a second)
constexpr float LOG2E = 1.4426950408889634f;
constexpr float RESCALE_THRESHOLD = 8.0f;   // log2 units
constexpr unsigned FULL = 0xffffffffu;
constexpr uint32_t NEG_INF_BITS = 0xff800000u;

struct TcParams {
    CUtensorMap qmap;  // [num_tokens rows, Hq * 128 cols]
    CUtensorMap kmap;  // paged pool [num_blocks * block_size rows, Hkv * 128 cols], or k [num_tokens rows, ...]
    CUtensorMap vmap;
    int64_t num_tokens;
    const int32_t *block_table;
    int max_blocks;
    int block_size;
    int64_t num_blocks;
    int box_rows;
    const int32_t *cu_q;
    const int32_t *cu_k;
    int max_q;
    int n_mtiles;
    int n_steps;      // item rows: query tiles (head pairs) or query-tile pairs (single heads)
    int units;        // items per sequence and step: head pairs, or heads
    int pair_heads;   // 1: an item's two tiles are two query heads; 0: two row tiles of one head
    int num_heads;
    int num_seqs;
    int kv_heads;
    float scale_log2;
    uint16_t *out;
    int out_v8;       // out is 32-byte aligned: the epilogue stores 32 bytes per instruction
    int32_t *status;
    long long wait_limit;     // SM cycles a pipeline wait may take before the call gives up
    int test_stall;           // test hook: the MMA warp first waits on a barrier nothing arrives on
    int kv_splits;            // key ranges per item (1: no split); split items write partials
    float *ws_o;              // [unit][QT][BM][D] unnormalised O of split items
    float2 *ws_ml;            // [unit][QT][BM] (running max in scaled log2 units, exponent sum)
};

// The CTA (of C) that takes the valid item of rank r in the snake order.
__device__ __forceinline__ int owner_of(int r, int nctas)
{
    const int round = r / nctas, pos = r % nctas;
    return (round & 1) ? nctas - 1 - pos : pos;
}

// Parity of completion number n of a barrier used by every nbuf-th round.
__device__ __forceinline__ uint32_t par(int n, int nbuf) { return uint32_t(n / nbuf) & 1u; }

// One work unit: the K/V tiles jb .. jb+nmax-1 of an item, which is two
// 128-row query tiles of one sequence that read the same KV head.  nt[a] counts
// query tile a's tiles in this unit (0: nothing to do for it).  When an item's
// keys are split over several units (split), each unit's softmax statistics
// and unnormalised O go to the workspace and a merge kernel combines them
// exactly ("大模型推理入门与 nano-vLLM 源码详解" §9.5).
struct Item {
    int b, g, q0, k0, offset;
    int h[QT], m0[QT], rows[QT], kend[QT], nt[QT];
    int nmax, kend_max;  // K/V tiles of the unit; keys the item reads
    int jb;              // first K/V tile of the unit
    bool valid, bad, split, last;
    int bad_code;
};

// Units are numbered item-major with the key split innermost; items walk
// (unit, sequence) and then the step from the last one down, so the heaviest
// tiles come first.
template <bool SPLIT>
__device__ __forceinline__ Item decode_item(const TcParams &p, int w)
{
    Item it;
    int ks = 0;
    if (SPLIT) {
        ks = w % p.kv_splits;
        w /= p.kv_splits;
    }
    const int xb = p.units * p.num_seqs;
    const int y = w / xb, x = w % xb;
    const int u = x % p.units;
    it.b = x / p.units;
    const int step = p.n_steps - 1 - y;
    it.q0 = p.cu_q[it.b];
    const int lq = p.cu_q[it.b + 1] - it.q0;
    it.k0 = p.cu_k[it.b];
    const int lk = p.cu_k[it.b + 1] - it.k0;
    const bool paged = p.block_table != nullptr;
    const bool rows_out = it.q0 < 0 || lq < 0 || int64_t(it.q0) + lq > p.num_tokens;
    it.bad = lk < lq || rows_out || (!paged && (lk != lq || it.k0 != it.q0)) ||
             (paged && int64_t(lk) > int64_t(p.max_blocks) * p.block_size);
    it.bad_code = (lk < lq || rows_out || !paged) ? PA_ERR_INVALID_ARG : PA_ERR_BOUNDS;
    it.offset = lk - lq;
    // rows beyond the stated maximum are not computed (the call reports it)
    const int lq_c = min(lq, p.max_q);
    it.nmax = 0;
    it.kend_max = 0;
#pragma unroll
    for (int a = 0; a < QT; ++a) {
        const int mt = p.pair_heads ? step : 2 * step + a;
        it.h[a] = p.pair_heads ? 2 * u + a : u;
        it.m0[a] = mt * BM;
        it.rows[a] = max(0, min(BM, lq_c - it.m0[a]));
        it.kend[a] = it.rows[a] > 0 ? it.offset + it.m0[a] + it.rows[a] : 0;
        it.nt[a] = (it.kend[a] + BN - 1) / BN;
        it.nmax = max(it.nmax, it.nt[a]);
        it.kend_max = max(it.kend_max, it.kend[a]);
    }
    it.g = it.h[0] / (p.num_heads / p.kv_heads);
    it.jb = 0;
    it.split = false;
    it.last = true;
    if (SPLIT) {  // this unit's share of the item's K/V tiles
        const int per = (it.nmax + p.kv_splits - 1) / p.kv_splits;
        it.jb = ks * per;
        const int je = min(it.nmax, it.jb + per);
        it.split = per < it.nmax;
        it.last = je == it.nmax;
#pragma unroll
        for (int a = 0; a < QT; ++a) it.nt[a] = max(0, min(je, it.nt[a]) - it.jb);
        it.nmax = max(0, je - it.jb);
    }
    it.valid = it.rows[0] > 0 && !it.bad && it.nmax > 0;
    if (lq > p.max_q && !it.bad) {
        it.bad = true;
        it.bad_code = PA_ERR_BOUNDS;
    }
    return it;
}

// An item as the scheduler publishes it (w = -1 ends the stream).
struct RingSlot {
    int w;
    Item it;
};
static_assert(sizeof(RingSlot) <= RING_SLOT_BYTES, "ring slot size");

// Where one producer warp reads a tile from: the TMA map of the paged pool
// with the item's block ids (-1 marks an id that failed validation), or, when
// there is no table, the map of the new-token rows from row0 on.
struct TileSource {
    const CUtensorMap *map;
    const int32_t *table;    // paged
    int box_rows;
    int block_size;
    int row0;                // no table: the sequence's first token row
};

// Issue the loads of the 128-key tile starting at key j0 into `dst`,
// arriving on `bar` (lane 0 issues).  Paged: one TMA box per page run; boxes
// at or past kend and boxes on invalid ids are skipped.  No table: one box of
// 128 token rows (rows past the last token are zero-filled by TMA).
__device__ __forceinline__ void load_tile(const TileSource &src, int xcol, int j0, int kend, uint32_t dst,
                                          uint32_t bar, int lane, int64_t num_blocks)
{
    if (src.table == nullptr) {
        if (lane == 0) {
            mbar_arrive_expect_tx(bar, TILE_BYTES);
            tma_load_2d(dst, src.map, xcol, src.row0 + j0, bar);
            tma_load_2d(dst + HALF_BYTES, src.map, xcol + 64, src.row0 + j0, bar);
        }
        __syncwarp();
    } else {
        if (lane == 0) {
            const int nbox = BN / src.box_rows;
            uint32_t bytes = 0;
            for (int bx = 0; bx < nbox; ++bx) {
                const int kb = j0 + bx * src.box_rows;
                if (kb >= kend) break;
                const int32_t phys = src.table[kb / src.block_size];
                if (phys >= 0 && int64_t(phys) < num_blocks) bytes += uint32_t(src.box_rows) * 128u * 2u;
            }
            mbar_arrive_expect_tx(bar, bytes);
            for (int bx = 0; bx < nbox; ++bx) {
                const int kb = j0 + bx * src.box_rows;
                if (kb >= kend) break;
                const int32_t phys = src.table[kb / src.block_size];
                if (phys < 0 || int64_t(phys) >= num_blocks) continue;
                const int y = int(int64_t(phys) * src.block_size + kb % src.block_size);
                const uint32_t off = uint32_t(bx * src.box_rows * 128);
                tma_load_2d(dst + off, src.map, xcol, y, bar);
                tma_load_2d(dst + HALF_BYTES + off, src.map, xcol + 64, y, bar);
            }
        }
        __syncwarp();
    }
}

// Mask keys past `limit` (tile-relative) to -inf.
template <int N>
__device__ __forceinline__ void mask_tail(uint32_t (&s)[N], int base, int limit)
{
#pragma unroll
    for (int c = 0; c < N; ++c)
        if (base + c > limit) s[c] = NEG_INF_BITS;
}

template <bool SPLIT>
__global__ void __launch_bounds__(NTHREADS, 1) prefill_tc_kernel(const __grid_constant__ TcParams p)
{
    extern __shared__ __align__(1024) uint8_t smem[];
    const uint32_t sb = smem_u32(smem);
    uint32_t *tmem_holder = reinterpret_cast<uint32_t *>(smem + OFF_MISC);
    volatile int32_t *abort_flag = reinterpret_cast<volatile int32_t *>(smem + OFF_MISC + 4);
    RingSlot *ring = reinterpret_cast<RingSlot *>(smem + OFF_RING);
    auto bar = [&](int i) { return sb + OFF_BAR + 8u * uint32_t(i); };
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    // the 128-byte swizzle pattern of TMA and the tensor cores is anchored at 1024-byte boundaries
    // (every CTA of a launch sees the same alignment, so none has touched the counters)
    if ((sb & 1023u) != 0) {
        if (threadIdx.x == 0) pa::report(p.status, PA_ERR_UNSUPPORTED);
        return;
    }
    const bool paged = p.block_table != nullptr;
    const int n_items = p.n_steps * p.units * p.num_seqs * p.kv_splits;

    if (threadIdx.x == 0) {
        for (int s = 0; s < QSLOTS; ++s) {
            mbar_init(bar(B_QF + s), 1);
            mbar_init(bar(B_QE + s), 1);
        }
        for (int s = 0; s < KSTAGES; ++s) {
            mbar_init(bar(B_KF + s), 1);
            mbar_init(bar(B_KE + s), 1);
        }
        for (int s = 0; s < VSTAGES; ++s) {
            mbar_init(bar(B_VF + s), 1);
            mbar_init(bar(B_VE + s), 1);
        }
        for (int a = 0; a < QT; ++a) {
            mbar_init(bar(B_SF + a), 1);
            mbar_init(bar(B_PF + a), 128);
            mbar_init(bar(B_PL + a), 128);
            mbar_init(bar(B_OF + a), 1);
        }
        for (int i = 0; i < 2; ++i) {
            mbar_init(bar(B_TF + i), 32);
            mbar_init(bar(B_TE + i), 2);
        }
        for (int s = 0; s < RING; ++s) {
            mbar_init(bar(B_IRF + s), 1);
            mbar_init(bar(B_IRE + s), IR_READERS);
        }
        mbar_init(bar(B_DRAIN), 1);
        mbar_init(bar(B_STALL), 1);
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
    // launched programmatically: the setup above (barriers, tensor memory) may
    // overlap the kernel before; everything below may read what it wrote (the
    // KV write of this step's tokens)
    pa::grid_dependency_wait();
    // the softmax warpgroups hold a 64-column slice of S, its P and O rows in
    // registers; the scheduler, producer and MMA warps need few
    static_assert(128 * REGS_CONTROL + 256 * REGS_SOFTMAX <= 168 * NTHREADS, "register split");
    // (the softmax warpgroups raise theirs at the start of their role below, so
    // that their code is compiled against the raised budget)
    if (warp < 4) regs_decrease<REGS_CONTROL>();

    // Read item n from the ring (every lane of the calling warp waits; lane 0
    // releases the slot).  Returns the item number, -1 at the end, -2 on abort.
    auto read_ring = [&](int n, Item &it) -> int {
        const int slot = n % RING;
        if (!__all_sync(FULL, mbar_wait(bar(B_IRF + slot), par(n, RING), abort_flag, p.wait_limit))) return -2;
        const int w = ring[slot].w;
        if (w >= 0) it = ring[slot].it;
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(B_IRE + slot));
        return w;
    };

    if (warp == 3) {
        // ------------------------------------------------------------ scheduler
        // Walk this CTA's items (heaviest first), publish each in the item ring,
        // stage its block ids (validated) for the producers and load its two Q
        // tiles.
        if (lane == 0) tma_prefetch_desc(&p.qmap);
        int n = 0;      // items published
        int qdone = 0;  // Q tiles announced (a TMA load, or an arrival for an empty tile)
        // The items are ranked 32 groups at a time (a lane each).  A group is the
        // items sharing (step, sequence), which are valid or not together: the
        // `units` head pairs of one row tile (one item each when the keys are not
        // split), or a single item when they are (the key splits of an item can
        // differ) or when there would be more than 32 in a group.  Window `win`
        // of the groups, `vbase` valid items before it; each lane keeps the mask
        // of its group's items this CTA takes, consumed lane by lane in order.
        const int per_group = (SPLIT || p.units > 32) ? 1 : p.units;
        const int n_groups = n_items / per_group;
        int win = 0, vbase = 0;
        uint32_t lane_mask = 0, lanes_left = 0, cur_bits = 0;
        int cur_group = 0;
        while (true) {
            int w = -1;
            while (true) {
                if (cur_bits != 0) {
                    w = cur_group * per_group + __ffs(cur_bits) - 1;
                    cur_bits &= cur_bits - 1u;
                    break;
                }
                if (lanes_left != 0) {
                    const int l = __ffs(lanes_left) - 1;
                    lanes_left &= lanes_left - 1u;
                    cur_bits = __shfl_sync(FULL, lane_mask, l);
                    cur_group = win - 32 + l;
                    continue;
                }
                if (win >= n_groups) break;
                const int gi = win + lane;
                int cnt = 0;
                if (gi < n_groups) {
                    const Item it = decode_item<SPLIT>(p, gi * per_group);
                    cnt = it.valid ? per_group : 0;
                    if (it.bad) pa::report(p.status, it.bad_code);
                }
                int incl = cnt;  // inclusive prefix sum over the lanes
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    const int v = __shfl_up_sync(FULL, incl, o);
                    if (lane >= o) incl += v;
                }
                const int first = vbase + incl - cnt;
                lane_mask = 0;
                for (int e = 0; e < cnt; ++e)
                    if (owner_of(first + e, int(gridDim.x)) == int(blockIdx.x)) lane_mask |= 1u << e;
                lanes_left = __ballot_sync(FULL, lane_mask != 0);
                vbase += __shfl_sync(FULL, incl, 31);
                win += 32;
            }
            const int slot = n % RING, tb = n & 1;
            if (n >= RING &&
                !__all_sync(FULL, mbar_wait(bar(B_IRE + slot), par(n - RING, RING), abort_flag, p.wait_limit)))
                break;
            Item it;
            if (w >= 0) {
                it = decode_item<SPLIT>(p, w);
                if (n >= 2 && !__all_sync(FULL, mbar_wait(bar(B_TE + tb), par(n - 2, 2), abort_flag, p.wait_limit)))
                    break;
                if (paged) {
                    const int nblk = (it.kend_max + p.block_size - 1) / p.block_size;
                    const int32_t *gtable = p.block_table + int64_t(it.b) * p.max_blocks;
                    int32_t *st = reinterpret_cast<int32_t *>(smem + OFF_TABLE) + tb * TABLE_SMEM;
                    bool bad = false;
                    for (int i = lane; i < nblk; i += 32) {
                        int32_t phys = gtable[i];
                        if (phys < 0 || int64_t(phys) >= p.num_blocks) {
                            bad = true;
                            phys = -1;
                        }
                        if (nblk <= TABLE_SMEM) st[i] = phys;
                    }
                    if (bad) pa::report(p.status, PA_ERR_BOUNDS);
                }
                mbar_arrive(bar(B_TF + tb));
            }
            if (lane == 0) {
                ring[slot].w = w;
                if (w >= 0) ring[slot].it = it;
                mbar_arrive(bar(B_IRF + slot));
            }
            if (w < 0) break;
            // the item's Q tiles into Q buffers 2n and 2n+1 (mod 2)
            // (rows past the sequence are other sequences' rows or TMA zero fill:
            // their results are not stored)
            bool ok = true;
            for (int a = 0; a < QT && ok; ++a) {
                const int qn = 2 * n + a, qs = qn % QSLOTS;
                if (qn >= QSLOTS &&
                    !(ok = __all_sync(FULL, mbar_wait(bar(B_QE + qs), par(qn - QSLOTS, QSLOTS), abort_flag, p.wait_limit))))
                    break;
                if (lane == 0) {
                    if (it.rows[a] > 0) {
                        const uint32_t dst = sb + OFF_Q + qs * TILE_BYTES, qb = bar(B_QF + qs);
                        mbar_arrive_expect_tx(qb, TILE_BYTES);
                        tma_load_2d(dst, &p.qmap, it.h[a] * D, it.q0 + it.m0[a], qb);
                        tma_load_2d(dst + HALF_BYTES, &p.qmap, it.h[a] * D + 64, it.q0 + it.m0[a], qb);
                    } else {
                        mbar_arrive(bar(B_QF + qs));
                    }
                }
                __syncwarp();
                ++qdone;
            }
            if (!ok) break;
            ++n;
        }
        if (lane == 0) {
            // the Q tiles in flight land before the CTA's shared memory goes away
            volatile int32_t dummy = 0;
            for (int qn = max(0, qdone - QSLOTS); qn < qdone; ++qn)
                mbar_wait(bar(B_QF + qn % QSLOTS), par(qn, QSLOTS), &dummy, WAIT_LIMIT);
        }
        __syncwarp();
    } else if (warp == 0 || warp == 2) {
        // ------------------------------------------------------------ producers (K, V)
        const bool is_k = warp == 0;
        TileSource src;
        src.map = is_k ? &p.kmap : &p.vmap;
        src.box_rows = p.box_rows;
        src.block_size = p.block_size;
        if (lane == 0) tma_prefetch_desc(src.map);
        const int nst = is_k ? KSTAGES : VSTAGES;
        const uint32_t base = sb + (is_k ? OFF_K : OFF_V);
        const int full0 = is_k ? B_KF : B_VF, empty0 = is_k ? B_KE : B_VE;
        int t = 0;  // tiles issued
        bool ok = true;
        for (int n = 0;; ++n) {
            Item it;
            const int w = read_ring(n, it);
            if (w == -2) ok = false;
            if (w < 0) break;
            const int tb = n & 1;
            if (!(ok = __all_sync(FULL, mbar_wait(bar(B_TF + tb), par(n, 2), abort_flag, p.wait_limit)))) break;
            const int nblk = paged ? (it.kend_max + p.block_size - 1) / p.block_size : 0;
            src.table = (paged && nblk <= TABLE_SMEM)
                            ? reinterpret_cast<const int32_t *>(smem + OFF_TABLE) + tb * TABLE_SMEM
                            : (paged ? p.block_table + int64_t(it.b) * p.max_blocks : nullptr);
            src.row0 = it.k0;
            for (int j = 0; j < it.nmax; ++j, ++t) {
                const int st = t % nst;
                if (t >= nst &&
                    !(ok = __all_sync(FULL, mbar_wait(bar(empty0 + st), par(t - nst, nst), abort_flag, p.wait_limit))))
                    break;
                load_tile(src, it.g * D, ((SPLIT ? it.jb : 0) + j) * BN, it.kend_max, base + st * TILE_BYTES,
                          bar(full0 + st), lane, p.num_blocks);
            }
            if (!ok) break;
            if (lane == 0) mbar_arrive(bar(B_TE + tb));  // this producer no longer reads the block ids
        }
        if (lane == 0) {
            // copies still in flight land before the CTA's shared memory goes away
            // (after a timeout anywhere in the CTA; otherwise these phases are
            // complete already)
            volatile int32_t dummy = 0;
            for (int u = max(0, t - nst); u < t; ++u)
                mbar_wait(bar(full0 + u % nst), par(u, nst), &dummy, WAIT_LIMIT);
        }
        __syncwarp();
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        // Issue blocks while the tensor pipe is busy, so the issue order below is
        // the execution order: per K/V tile j, P_0.V_j, S_0 of tile j+1, P_1.V_j,
        // S_1 of tile j+1.  The softmax of one query tile thus runs while the
        // tensor cores work on the other.  The whole warp runs this loop (every
        // decision is warp-uniform) and one elected lane issues each tcgen05
        // instruction: issued that way an MMA costs the issuer a fraction of the
        // cycles it costs from a lone lane, which would leave the pipe idle.
        // shared-memory descriptors of the first Q, K and V buffers; a buffer or
        // k-step further on adds its byte offset / 16 (the 14-bit address field
        // cannot overflow below 256 KB)
        const uint64_t desc_q = smem_desc(sb + OFF_Q, 16, 1024);
        const uint64_t desc_k = smem_desc(sb + OFF_K, 16, 1024);
        const uint64_t desc_v = smem_desc(sb + OFF_V, HALF_BYTES, 1024);
        int t = 0;               // K/V tiles consumed
        int c[QT] = {0, 0};      // S / P tiles per query tile
        bool ok = true;
        auto commit = [&](int b) {
            if (elect_one()) mma_commit(bar(b));
            __syncwarp();
        };
        // (a test's stall: this wait runs out after the pipeline limit and the
        // whole CTA stops as after any timeout)
        if (p.test_stall) ok = __all_sync(FULL, mbar_wait(bar(B_STALL), 0, abort_flag, p.wait_limit));
        for (int n = 0; ok; ++n) {
            const int slot = n % RING;
            if (!__all_sync(FULL, mbar_wait(bar(B_IRF + slot), par(n, RING), abort_flag, p.wait_limit))) break;
            const int w = ring[slot].w;
            if (w < 0) break;
            const Item it = ring[slot].it;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar(B_IRE + slot));
            constexpr uint32_t IDESC_QK = idesc_bf16(BM, BN, 0, 0);  // Q, K both K-major
            constexpr uint32_t IDESC_PV = idesc_bf16(BM, D, 0, 1);   // P from TMEM, V MN-major
            auto wait = [&](int b, uint32_t parity) {
                ok = ok && __all_sync(FULL, mbar_wait(bar(b), parity, abort_flag, p.wait_limit));
                return ok;
            };
            auto issue_s = [&](int a, int qs, int kst) {
                const uint64_t qd = desc_q + uint64_t((qs * TILE_BYTES) >> 4);
                const uint64_t kd = desc_k + uint64_t((kst * TILE_BYTES) >> 4);
                const uint32_t dst = tmem + 128u * a;
#pragma unroll
                for (int kk = 0; kk < D / 16; ++kk) {
                    const uint64_t off = uint64_t(((kk >> 2) * HALF_BYTES + (kk & 3) * 32) >> 4);
                    if (elect_one()) mma_ss(dst, qd + off, kd + off, IDESC_QK, kk > 0);
                }
                __syncwarp();
                commit(B_SF + a);
            };
            // first S of each query tile: its S columns still hold P of the
            // previous item, whose P.V was issued before (tcgen05 runs in order)
            if (wait(B_KF + t % KSTAGES, par(t, KSTAGES))) {
                tc_fence_after();
                // every Q buffer's landing is waited for in order, used or not, so
                // that no parity wait runs ahead of an earlier phase of its barrier
                for (int a = 0; a < QT; ++a) {
                    const int qn = 2 * n + a, qs = qn % QSLOTS;
                    if (!wait(B_QF + qs, par(qn, QSLOTS))) break;
                    if (it.nt[a] == 0) {
                        commit(B_QE + qs);
                        continue;
                    }
                    tc_fence_after();
                    issue_s(a, qs, t % KSTAGES);
                    if (it.nt[a] == 1) commit(B_QE + qs);  // the tile's last S
                }
                if (ok) commit(B_KE + t % KSTAGES);
            }
            for (int j = 0; ok && j < it.nmax; ++j) {
                const int tv = t + j;
                bool v_in = false, k_in = false;
                for (int a = 0; a < QT; ++a) {
                    if (j >= it.nt[a]) continue;
                    // P.V in two halves of the keys: the first runs while the
                    // softmax still computes the second half of P
                    if (!wait(B_PL + a, uint32_t(c[a]) & 1u)) break;
                    if (!v_in && !(v_in = wait(B_VF + tv % VSTAGES, par(tv, VSTAGES)))) break;
                    tc_fence_after();
                    const uint64_t vd = desc_v + uint64_t(((tv % VSTAGES) * TILE_BYTES) >> 4);
                    const uint32_t dst = tmem + COL_O + 128u * a, src = tmem + 128u * a;
                    const uint32_t acc0 = j > 0 ? 1u : 0u;
#pragma unroll
                    for (int kk = 0; kk < BN / 32; ++kk)
                        if (elect_one())
                            mma_ts(dst, src + kk * 8, vd + uint64_t((kk * 2048) >> 4), IDESC_PV, kk > 0 ? 1u : acc0);
                    __syncwarp();
                    if (!wait(B_PF + a, uint32_t(c[a]) & 1u)) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = BN / 32; kk < BN / 16; ++kk)
                        if (elect_one())
                            mma_ts(dst, src + kk * 8, vd + uint64_t((kk * 2048) >> 4), IDESC_PV, 1u);
                    __syncwarp();
                    ++c[a];
                    if (j + 1 < it.nt[a]) {
                        if (!k_in && !(k_in = wait(B_KF + (tv + 1) % KSTAGES, par(tv + 1, KSTAGES)))) break;
                        tc_fence_after();
                        const int qs = (2 * n + a) % QSLOTS;
                        issue_s(a, qs, (tv + 1) % KSTAGES);
                        if (j + 2 == it.nt[a]) commit(B_QE + qs);  // the tile's last S
                    }
                }
                if (!ok) break;
                commit(B_VE + tv % VSTAGES);
                if (j + 1 < it.nmax) commit(B_KE + (tv + 1) % KSTAGES);
            }
            if (ok) {
                for (int a = 0; a < QT; ++a)
                    if (it.nt[a] > 0) commit(B_OF + a);
            }
            t += it.nmax;
        }
        // every MMA issued is complete before TMEM and shared memory are released
        {
            volatile int32_t dummy = 0;
            commit(B_DRAIN);
            mbar_wait(bar(B_DRAIN), 0, &dummy, WAIT_LIMIT);
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ softmax + epilogue
        regs_increase<REGS_SOFTMAX>();
        const int a = (warp - 4) >> 2;  // the query tile of each item this warpgroup owns
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;
        const uint32_t lane_base = uint32_t(quarter * 32) << 16;
        const uint32_t scol = tmem + lane_base + 128u * a;
        const uint32_t ocol = tmem + lane_base + COL_O + 128u * a;
        const float sl2 = p.scale_log2;
        int c = 0, no = 0, t = 0;  // tiles of this query tile, items with work, K/V tiles of all items
        bool ok = true;
        // The epilogue of an item is deferred: its O stays in TMEM until this
        // warpgroup has written the next item's first P, and is read just before
        // that P is released to the MMA warp (the item's first P.V overwrites O).
        // The wait for the last P.V and the normalise-and-store then overlap the
        // next item's MMAs instead of holding them up.
        bool pend = false;  // an item's O waits in TMEM
        bool pe_split = false;
        int pe_w = 0, pe_rows = 0, pe_tok = 0, pe_h = 0;
        float pe_m = 0.f, pe_l = 0.f;
        auto finish = [&](bool release_p) {
            pend = false;
            ok = __all_sync(FULL, mbar_wait(bar(B_OF + a), uint32_t(no) & 1u, abort_flag, p.wait_limit));
            ++no;
            if (!ok) return;
            tc_fence_after();
            auto release = [&]() {
                tc_fence_before();
                mbar_arrive(bar(B_PL + a));
                mbar_arrive(bar(B_PF + a));
            };
            if (SPLIT && pe_split) {
                // a share of a split item: unnormalised O and (max, sum) for the merge
                const int64_t row = (int64_t(pe_w) * QT + a) * BM + r;
                float *dst = p.ws_o + row * D;  // 256-byte aligned rows
#pragma unroll
                for (int hh = 0; hh < 2; ++hh) {
                    uint32_t o[64];
                    tmem_ld64_sync(ocol + 64 * hh, o);
                    if (release_p && hh == 1) release();
                    if (r < pe_rows) {
#pragma unroll
                        for (int v = 0; v < 8; ++v) {
                            uint32_t w8[8];
#pragma unroll
                            for (int e = 0; e < 8; ++e) w8[e] = o[8 * v + e];
                            st_global_v8(dst + 64 * hh + 8 * v, w8);
                        }
                    }
                }
                if (r < pe_rows) p.ws_ml[row] = make_float2(pe_m, pe_l);
                return;
            }
            // O / l, packed to bf16 pairs as it is read (half the registers of
            // the fp32 row: this runs inside the next item's tile loop)
            const float inv = r < pe_rows ? 1.f / pe_l : 0.f;
            uint32_t ob[64];
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
                uint32_t o[64];
                tmem_ld64_sync(ocol + 64 * hh, o);
#pragma unroll
                for (int i = 0; i < 32; ++i)
                    ob[32 * hh + i] = pa::pack_bf16x2(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            }
            if (release_p) release();
            if (r >= pe_rows) return;
            uint16_t *dst = p.out + (int64_t(pe_tok + r) * p.num_heads + pe_h) * D;
            if (p.out_v8) {
#pragma unroll
                for (int v = 0; v < 8; ++v) {
                    uint32_t w8[8];
#pragma unroll
                    for (int e = 0; e < 8; ++e) w8[e] = ob[8 * v + e];
                    st_global_v8(dst + 16 * v, w8);
                }
            } else {
                uint4 *d4 = reinterpret_cast<uint4 *>(dst);
#pragma unroll
                for (int v = 0; v < 16; ++v) d4[v] = make_uint4(ob[4 * v], ob[4 * v + 1], ob[4 * v + 2], ob[4 * v + 3]);
            }
        };
        for (int n = 0;; ++n) {
            Item it;
            const int w = read_ring(n, it);
            if (w == -2) ok = false;
            if (w < 0) break;
            const int tbase = t;
            t += it.nmax;
            if (it.nt[a] == 0) continue;
            // rows past the last key of the item's last K/V tile may be unused
            // pool slots (any bits) or another sequence's rows: the warpgroup of
            // the first query tile that reads that tile sets those V rows to 0
            // so that 0 * V stays 0
            const int jb = SPLIT ? it.jb : 0;  // first K/V tile of the unit
            const bool zeroer = a == (it.nt[0] == it.nmax ? 0 : 1) && (!SPLIT || it.last) &&
                                it.kend_max < (jb + it.nmax) * BN;
            const int pos = it.offset + it.m0[a] + r;
            const int last_visible = min(pos, it.kend[a] - 1);
            float m_used = -INFINITY;  // running max in scaled base-2 units
            float l = 0.f;
            for (int j = 0; j < it.nt[a]; ++j, ++c) {
                ok = __all_sync(FULL, mbar_wait(bar(B_SF + a), uint32_t(c) & 1u, abort_flag, p.wait_limit));
                if (!ok) break;
                tc_fence_after();
                const int j0 = (jb + j) * BN;
                const bool masked = j0 + BN - 1 > it.offset + it.m0[a];  // the tile crosses some row's causal bound
                const int limit = last_visible - j0;
                // one pass over the row: its 128 scores are loaded from TMEM once,
                // the row max taken in registers, then P = 2^(s * scale * log2 e - m)
                // is formed from the same registers, 64 keys at a time; P (bf16
                // pairs) goes over the S columns already read
                uint32_t sr[128];
                tmem_ld128_sync(scol, sr);
                if (masked) mask_tail(sr, 0, limit);
                float mx8[8];
#pragma unroll
                for (int k = 0; k < 8; ++k) mx8[k] = fmaxf(__uint_as_float(sr[k]), __uint_as_float(sr[8 + k]));
#pragma unroll
                for (int cc = 16; cc < 128; cc += 16) {
#pragma unroll
                    for (int k = 0; k < 8; ++k)
                        mx8[k] = fmax3(mx8[k], __uint_as_float(sr[cc + k]), __uint_as_float(sr[cc + 8 + k]));
                }
                const float mx =
                    fmax3(fmax3(mx8[0], mx8[1], mx8[2]), fmax3(mx8[3], mx8[4], mx8[5]), fmaxf(mx8[6], mx8[7])) * sl2;
                const bool need = mx > m_used + RESCALE_THRESHOLD;
                const float m_new = need ? mx : m_used;
                const float factor = need ? ex2_approx(m_used - m_new) : 1.f;
                const bool rescale_o = j > 0 && __any_sync(FULL, need);
                l *= factor;
                m_used = m_new;
                const float nm = (m_used == -INFINITY) ? 0.f : -m_used;
                // (before the first half of P is released: P.V of keys 0-63 may read them)
                if (zeroer && j == it.nmax - 1) {
                    const int tv = tbase + j, sv = tv % VSTAGES;
                    ok = __all_sync(FULL, mbar_wait(bar(B_VF + sv), par(tv, VSTAGES), abort_flag, p.wait_limit));
                    if (!ok) break;
                    if (j0 + r >= it.kend_max) {
                        uint4 *row0 = reinterpret_cast<uint4 *>(smem + OFF_V + sv * TILE_BYTES + r * 128);
                        uint4 *row1 = reinterpret_cast<uint4 *>(smem + OFF_V + sv * TILE_BYTES + HALF_BYTES + r * 128);
#pragma unroll
                        for (int cc = 0; cc < 8; ++cc) row0[cc] = row1[cc] = make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();
                }
                float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
#pragma unroll
                for (int hf = 0; hf < 2; ++hf) {
                    uint32_t pk[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        float x0, x1;
                        ffma2(x0, x1, __uint_as_float(sr[64 * hf + 2 * i]), __uint_as_float(sr[64 * hf + 2 * i + 1]), sl2,
                              sl2, nm, nm);
                        const float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
                        fadd2(acc[2 * (i & 3)], acc[2 * (i & 3) + 1], p0, p1);
                        pk[i] = pa::pack_bf16x2(p0, p1);
                    }
                    tmem_st32_sync(scol + hf * 32, pk);
                    if (hf == 0) {
                        if (rescale_o) {
                            // O holds the previous tile's P.V: that P.V was issued before
                            // this tile's S, whose completion the S barrier reported; the
                            // P.V of this tile starts only after the arrival below
#pragma unroll
                            for (int cc = 0; cc < 4; ++cc) {
                                uint32_t o[32];
                                tmem_ld32_sync(ocol + cc * 32, o);
#pragma unroll
                                for (int q = 0; q < 32; ++q) o[q] = __float_as_uint(__uint_as_float(o[q]) * factor);
                                tmem_st32_sync(ocol + cc * 32, o);
                            }
                        }
                        if (j > 0 || !pend) {
                            tc_fence_before();
                            mbar_arrive(bar(B_PL + a));
                        }
                    }
                }
                l += ((acc[0] + acc[1]) + (acc[2] + acc[3])) + ((acc[4] + acc[5]) + (acc[6] + acc[7]));
                if (j == 0 && pend) {
                    finish(true);  // the previous item's epilogue, then this P is released
                    if (!ok) break;
                } else {
                    tc_fence_before();
                    mbar_arrive(bar(B_PF + a));
                }
            }
            if (!ok) break;
            pend = true;
            pe_split = SPLIT && it.split;
            pe_w = w;
            pe_rows = it.rows[a];
            pe_tok = it.q0 + it.m0[a];
            pe_h = it.h[a];
            pe_m = m_used;
            pe_l = l;
        }
        if (ok && pend) finish(false);
    }

    tc_fence_before();
    __syncthreads();
    if (threadIdx.x == 0 && *abort_flag) pa::report(p.status, PA_ERR_TIMEOUT);
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem, TMEM_COLS);
    }
}

// Combine the key-range shares of every split item: per query row,
// M = max_s m_s, L = sum_s l_s 2^(m_s - M), out = sum_s O_s 2^(m_s - M) / L
// ("大模型推理入门与 nano-vLLM 源码详解" §9.5).  A CTA per (item, query tile, 16
// rows); 16 threads per row, 8 columns each, so that a row's 512-byte shares
// are read by contiguous threads.
constexpr int MERGE_ROWS = 16;
__global__ void __launch_bounds__(MERGE_ROWS * 16) prefill_merge_kernel(const __grid_constant__ TcParams p)
{
    pa::grid_dependency_wait();  // the shares of the split kernel
    const int a = blockIdx.y;
    const int r = blockIdx.z * MERGE_ROWS + int(threadIdx.x >> 4);
    const int c8 = int(threadIdx.x & 15) * 8;  // this thread's first column
    const int w0 = blockIdx.x * p.kv_splits;
    const Item first = decode_item<true>(p, w0);
    if (!first.split || first.bad || r >= first.rows[a]) return;
    float mm = -INFINITY;
    for (int s = 0; s < p.kv_splits; ++s) {
        const Item it = decode_item<true>(p, w0 + s);
        if (it.valid && it.nt[a] > 0) mm = fmaxf(mm, p.ws_ml[(int64_t(w0 + s) * QT + a) * BM + r].x);
    }
    float acc[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
    float ll = 0.f;
    for (int s = 0; s < p.kv_splits; ++s) {
        const Item it = decode_item<true>(p, w0 + s);
        if (!it.valid || it.nt[a] == 0) continue;
        const int64_t row = (int64_t(w0 + s) * QT + a) * BM + r;
        const float2 ml = p.ws_ml[row];
        const float wgt = ml.x == -INFINITY ? 0.f : ex2_approx(ml.x - mm);
        ll = fmaf(ml.y, wgt, ll);
        const float4 *src = reinterpret_cast<const float4 *>(p.ws_o + row * D + c8);
        const float4 x0 = src[0], x1 = src[1];
        acc[0] = fmaf(x0.x, wgt, acc[0]);
        acc[1] = fmaf(x0.y, wgt, acc[1]);
        acc[2] = fmaf(x0.z, wgt, acc[2]);
        acc[3] = fmaf(x0.w, wgt, acc[3]);
        acc[4] = fmaf(x1.x, wgt, acc[4]);
        acc[5] = fmaf(x1.y, wgt, acc[5]);
        acc[6] = fmaf(x1.z, wgt, acc[6]);
        acc[7] = fmaf(x1.w, wgt, acc[7]);
    }
    const float inv = 1.f / ll;
    uint4 u;
    u.x = pa::pack_bf16x2(acc[0] * inv, acc[1] * inv);
    u.y = pa::pack_bf16x2(acc[2] * inv, acc[3] * inv);
    u.z = pa::pack_bf16x2(acc[4] * inv, acc[5] * inv);
    u.w = pa::pack_bf16x2(acc[6] * inv, acc[7] * inv);
    *reinterpret_cast<uint4 *>(p.out + (int64_t(first.q0 + first.m0[a] + r) * p.num_heads + first.h[a]) * D + c8) = u;
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

// A 2-D map over `rows` rows of `heads` * 128 bf16 each, rows `stride`
// elements apart, read in boxes of 64 columns x box_rows rows with the
// 128-byte swizzle.
bool make_rows_map(CUtensorMap *map, const void *base, int64_t rows, int heads, int64_t stride, int box_rows)
{
    auto fn = encode_fn();
    if (fn == nullptr) return false;
    const cuuint64_t dims[2] = {cuuint64_t(heads) * D, cuuint64_t(rows)};
    const cuuint64_t strides[1] = {cuuint64_t(stride) * 2};
    const cuuint32_t box[2] = {64, cuuint32_t(box_rows)};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box, estr,
              CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int gcd(int a, int b) { return b == 0 ? a : gcd(b, a % b); }


// How many key ranges each item is split into: 1 when the call has enough
// items to fill the GPU twice over; otherwise the count that minimises
// rounds x (tiles per unit + a unit's fixed cost, about two tiles' worth of
// time for its fill and drain), each unit at least SPLIT_MIN_TILES K/V tiles.
constexpr int SPLIT_MIN_TILES = 4;
constexpr int UNIT_COST_TILES = 2;

struct PrefillPlan {
    int n_mtiles, n_steps, units, pair_heads, kv_splits;
    int64_t items;  // before the key split
};

PrefillPlan make_prefill_plan(int num_seqs, int max_seqlen_q, int max_seqlen_k, int num_heads, int num_kv_heads)
{
    PrefillPlan pl;
    pl.n_mtiles = (max_seqlen_q + BM - 1) / BM;
    pl.pair_heads = num_heads / num_kv_heads >= 2 ? 1 : 0;
    pl.n_steps = pl.pair_heads ? pl.n_mtiles : (pl.n_mtiles + 1) / 2;
    pl.units = pl.pair_heads ? num_heads / 2 : num_heads;
    pl.items = int64_t(pl.n_steps) * pl.units * num_seqs;
    pl.kv_splits = 1;
    const int sms = pa::num_sms() > 0 ? pa::num_sms() : 148;
    const int64_t want = 2LL * sms;
    const int kv_tiles = (max_seqlen_k + BN - 1) / BN;
    if (pl.items > 0 && pl.items < want && kv_tiles >= 2 * SPLIT_MIN_TILES) {
        const int most = std::min(64, kv_tiles / SPLIT_MIN_TILES);
        int64_t best = -1;
        for (int s = 1; s <= most; ++s) {
            const int64_t rounds = (pl.items * s + sms - 1) / sms;
            const int64_t cost = rounds * ((kv_tiles + s - 1) / s + UNIT_COST_TILES);
            if (best < 0 || cost < best) {
                best = cost;
                pl.kv_splits = s;
            }
        }
    }
    return pl;
}

size_t prefill_workspace(const PrefillPlan &pl)
{
    if (pl.kv_splits <= 1) return 0;
    const size_t rows = size_t(pl.items) * pl.kv_splits * QT * BM;
    return (rows * D * sizeof(float) + 255) / 256 * 256 + rows * sizeof(float2);
}

}  // namespace

extern "C" pa_status pa_prefill_paged(const void *q, int64_t q_stride_tok, int64_t num_tokens, const void *k,
                                      const void *v,
                                      int64_t kv_stride_tok, const void *k_cache, const void *v_cache,
                                      int64_t num_blocks, int block_size, const int32_t *block_table,
                                      int max_blocks_per_seq, const int32_t *cu_seqlens_q,
                                      const int32_t *cu_seqlens_k, int num_seqs, int max_seqlen_q,
                                      int max_seqlen_k, int num_heads, int num_kv_heads, int head_dim,
                                      float scale, void *out, void *workspace, size_t workspace_bytes,
                                      int32_t *dev_status, void *stream)
{
    if (num_seqs < 0 || max_seqlen_q < 0 || max_seqlen_k < 0 || num_blocks < 0 || num_tokens < 0)
        return PA_ERR_INVALID_ARG;
    if (head_dim != D || !pa::pow2_in(num_kv_heads, 1, 8) || num_heads <= 0 || num_heads % num_kv_heads != 0 ||
        !pa::pow2_in(num_heads / num_kv_heads, 1, 8))
        return PA_ERR_UNSUPPORTED;
    if (block_table != nullptr && (block_size < 16 || block_size > 1024 || block_size % 16 != 0))
        return PA_ERR_UNSUPPORTED;
    if (num_seqs == 0 || max_seqlen_q == 0 || num_tokens == 0) return PA_OK;
    if (num_tokens >= (int64_t(1) << 31)) return PA_ERR_UNSUPPORTED;
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
    const PrefillPlan pl = make_prefill_plan(num_seqs, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads);
    if (pl.items * pl.kv_splits > 0x7fffffff) return PA_ERR_UNSUPPORTED;
    const size_t need = prefill_workspace(pl);
    if (need > 0 && (workspace == nullptr || workspace_bytes < need || !pa::aligned(workspace, 256)))
        return PA_ERR_INVALID_ARG;

    TcParams p;
    memset(&p, 0, sizeof(p));
    p.num_tokens = num_tokens;
    p.block_table = block_table;
    p.max_blocks = max_blocks_per_seq;
    p.block_size = block_size;
    p.num_blocks = num_blocks;
    p.box_rows = block_table ? gcd(block_size, BN) : BN;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.max_q = max_seqlen_q;
    p.n_mtiles = pl.n_mtiles;
    p.pair_heads = pl.pair_heads;
    p.n_steps = pl.n_steps;
    p.units = pl.units;
    p.kv_splits = pl.kv_splits;
    {
        const size_t rows = size_t(pl.items) * pl.kv_splits * QT * BM;
        p.ws_o = need > 0 ? static_cast<float *>(workspace) : nullptr;
        p.ws_ml = need > 0 ? reinterpret_cast<float2 *>(static_cast<char *>(workspace) +
                                                       (rows * D * sizeof(float) + 255) / 256 * 256)
                           : nullptr;
    }
    p.num_heads = num_heads;
    p.num_seqs = num_seqs;
    p.kv_heads = num_kv_heads;
    p.scale_log2 = scale * LOG2E;
    p.out = static_cast<uint16_t *>(out);
    p.out_v8 = pa::aligned(out, 32) ? 1 : 0;
    p.status = dev_status;
    // (the waits that drain copies and MMAs after a timeout keep WAIT_LIMIT)
    p.wait_limit = pa::pipeline_wait_limit(WAIT_LIMIT);
    p.test_stall = pa::pipeline_test_stall() ? 1 : 0;
    if (!make_rows_map(&p.qmap, q, num_tokens, num_heads, q_stride_tok, BM)) return PA_ERR_CUDA;
    if (block_table != nullptr) {
        const int64_t rows = num_blocks * block_size, row = int64_t(num_kv_heads) * D;
        if (!make_rows_map(&p.kmap, k_cache, rows, num_kv_heads, row, p.box_rows) ||
            !make_rows_map(&p.vmap, v_cache, rows, num_kv_heads, row, p.box_rows))
            return PA_ERR_CUDA;
    } else {
        if (!make_rows_map(&p.kmap, k, num_tokens, num_kv_heads, kv_stride_tok, BN) ||
            !make_rows_map(&p.vmap, v, num_tokens, num_kv_heads, kv_stride_tok, BN))
            return PA_ERR_CUDA;
    }
    if (pa::allow_dynamic_smem(reinterpret_cast<const void *>(prefill_tc_kernel<false>), SMEM_BYTES) != cudaSuccess ||
        pa::allow_dynamic_smem(reinterpret_cast<const void *>(prefill_tc_kernel<true>), SMEM_BYTES) != cudaSuccess)
        return PA_ERR_CUDA;
    const int64_t units = pl.items * pl.kv_splits;
    const int sms = pa::num_sms() > 0 ? pa::num_sms() : 148;
    const dim3 grid(unsigned(units < sms ? units : sms));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    if (pl.kv_splits > 1)
        pa::launch_pdl(prefill_tc_kernel<true>, grid, dim3(NTHREADS), SMEM_BYTES, s, p);
    else
        pa::launch_pdl(prefill_tc_kernel<false>, grid, dim3(NTHREADS), SMEM_BYTES, s, p);
    if (pl.kv_splits > 1)
        pa::launch_pdl(prefill_merge_kernel, dim3(unsigned(pl.items), QT, BM / MERGE_ROWS), dim3(MERGE_ROWS * 16), 0,
                       s, p);
    return pa::launch_status();
}

extern "C" size_t pa_prefill_workspace_bytes(int num_seqs, int max_seqlen_q, int max_seqlen_k, int num_heads,
                                             int num_kv_heads)
{
    if (num_seqs <= 0 || max_seqlen_q <= 0 || max_seqlen_k < 0 || num_heads <= 0 || num_kv_heads <= 0 ||
        num_heads % num_kv_heads != 0)
        return 0;
    return prefill_workspace(make_prefill_plan(num_seqs, max_seqlen_q, max_seqlen_k, num_heads, num_kv_heads));
}
