// prefill_paged.cu -- causal varlen prefill over a block-paged KV cache.
//
// What it computes ("大模型推理入门与 nano-vLLM 源码详解" §11.2, §10.2, §13.3):
// sequence b has Lq new queries that are the last Lq positions of its Lk-key
// context; query i (absolute position p = Lk - Lq + i) reads keys 0..p.  Keys
// come from the paged pool through block_table (a cached prefix or an earlier
// chunk) or, without a table, from the new-token k / v rows.  Query head h
// reads KV head h / (Hq / Hkv).  Softmax is computed blockwise with a running
// max, sum and unnormalised numerator (§13.3).
//
// Kernel: a CTA takes a 64-query tile of one (sequence, query head); four
// warps each own 16 query rows.  K/V tiles of 64 keys are gathered page by
// page with 16-byte cp.async into XOR-swizzled shared memory (double
// buffered), QK^T and PV run as bf16 tensor-core MMAs with fp32
// accumulators, and the online softmax runs in base 2 with scale * log2(e)
// folded in.  Key tiles past the tile's last visible key are never loaded;
// masking touches only tiles that cross the causal diagonal.
#include "pa_common.cuh"

namespace {

constexpr int D = pa::kHeadDim;
constexpr int BM = 64;   // queries per CTA
constexpr int BN = 64;   // keys per tile
constexpr int NWARP = 4;
constexpr int NTHREAD = NWARP * 32;
constexpr float LOG2E = 1.4426950408889634f;
constexpr int TILE_BYTES = BN * D * 2;  // 16 KiB per K or V tile; Q tile is the same size
constexpr int SMEM_BYTES = TILE_BYTES * 5;  // Q + 2 x (K, V)

struct PrefillParams {
    const uint16_t *q;
    int64_t q_stride;
    const uint16_t *k;
    const uint16_t *v;
    int64_t kv_stride;
    const uint16_t *k_cache;
    const uint16_t *v_cache;
    int64_t num_blocks;
    int block_size;
    const int32_t *block_table;  // nullptr: contiguous k / v
    int max_blocks;
    const int32_t *cu_q;
    const int32_t *cu_k;
    int max_q;
    int num_heads;
    int kv_heads;
    float scale_log2;
    uint16_t *out;
    int32_t *status;
};

__device__ __forceinline__ uint32_t smem_addr(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// byte offset of 16-byte chunk `ch` of row `row` in a [rows][256 B] tile,
// chunks XOR-swizzled by the row's low 3 bits (ldmatrix reads 8 rows at the
// same logical chunk without bank conflicts)
__device__ __forceinline__ uint32_t swz(int row, int ch)
{
    return uint32_t(row * 256 + ((ch ^ (row & 7)) << 4));
}

__device__ __forceinline__ void cp_async16(uint32_t dst, const void *src, bool valid)
{
    const int n = valid ? 16 : 0;  // 0 bytes read: the 16 destination bytes are zero-filled
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"(dst), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N)); }

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}
__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2, uint32_t &r3)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3)
                 : "r"(addr));
}

__device__ __forceinline__ void mma_bf16(float (&c)[4], const uint32_t (&a)[4], uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, "
        "{%0,%1,%2,%3};"
        : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
        : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

// Issue the cp.async copies of key tile [j0, j0 + BN) of one sequence into
// (ks, vs).  Keys at or beyond kend are zero-filled.
__device__ __forceinline__ void load_kv_tile(const PrefillParams &p, int b, int g, int key_base, int j0,
                                             int kend, uint8_t *ks, uint8_t *vs, bool &bad)
{
    const int ch = threadIdx.x & 15;
    const int64_t row_elems = int64_t(p.kv_heads) * D;
#pragma unroll
    for (int it = 0; it < BN / (NTHREAD / 16); ++it) {
        const int r = (threadIdx.x >> 4) + it * (NTHREAD / 16);
        const int j = j0 + r;
        bool valid = j < kend;
        const uint16_t *ksrc = p.q;  // any mapped address; nothing is read when !valid
        const uint16_t *vsrc = p.q;
        if (valid) {
            if (p.block_table != nullptr) {
                const int32_t phys = p.block_table[int64_t(b) * p.max_blocks + j / p.block_size];
                if (phys < 0 || int64_t(phys) >= p.num_blocks) {
                    bad = true;
                    valid = false;
                } else {
                    const int64_t row = int64_t(phys) * p.block_size + j % p.block_size;
                    ksrc = p.k_cache + row * row_elems + g * D + ch * 8;
                    vsrc = p.v_cache + row * row_elems + g * D + ch * 8;
                }
            } else {
                const int64_t row = int64_t(key_base) + j;
                ksrc = p.k + row * p.kv_stride + g * D + ch * 8;
                vsrc = p.v + row * p.kv_stride + g * D + ch * 8;
            }
        }
        cp_async16(smem_addr(ks + swz(r, ch)), ksrc, valid);
        cp_async16(smem_addr(vs + swz(r, ch)), vsrc, valid);
    }
}

__global__ void __launch_bounds__(NTHREAD) prefill_mma_kernel(const PrefillParams p)
{
    extern __shared__ __align__(128) uint8_t smem[];
    uint8_t *qs = smem;
    uint8_t *ks[2] = {smem + TILE_BYTES, smem + 3 * TILE_BYTES};
    uint8_t *vs[2] = {smem + 2 * TILE_BYTES, smem + 4 * TILE_BYTES};

    const int b = blockIdx.z, h = blockIdx.y, mt = blockIdx.x;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int q0 = p.cu_q[b], lq = p.cu_q[b + 1] - q0;
    const int k0 = p.cu_k[b], lk = p.cu_k[b + 1] - k0;
    if (mt == 0 && threadIdx.x == 0) {
        if (lk < lq || (p.block_table == nullptr && (lk != lq || k0 != q0))) pa::report(p.status, PA_ERR_INVALID_ARG);
        else if (lq > p.max_q) pa::report(p.status, PA_ERR_BOUNDS);
        else if (p.block_table != nullptr && int64_t(lk) > int64_t(p.max_blocks) * p.block_size)
            pa::report(p.status, PA_ERR_BOUNDS);
    }
    if (lq <= 0 || mt * BM >= lq) return;
    if (lk < lq || (p.block_table == nullptr && (lk != lq || k0 != q0))) return;
    if (p.block_table != nullptr && int64_t(lk) > int64_t(p.max_blocks) * p.block_size) return;

    const int group = p.num_heads / p.kv_heads;
    const int g = h / group;
    const int m0 = mt * BM;
    const int offset = lk - lq;                       // absolute position of query 0
    const int rows = min(BM, lq - m0);
    const int kend = offset + m0 + rows;              // keys visible to the tile's last row
    const int ntiles = (kend + BN - 1) / BN;
    bool bad = false;

    // Q tile (rows past lq zero-filled) and the first K/V tile
    {
        const int ch = threadIdx.x & 15;
#pragma unroll
        for (int it = 0; it < BM / (NTHREAD / 16); ++it) {
            const int r = (threadIdx.x >> 4) + it * (NTHREAD / 16);
            const bool valid = r < rows;
            const uint16_t *src = valid ? p.q + int64_t(q0 + m0 + r) * p.q_stride + h * D + ch * 8 : p.q;
            cp_async16(smem_addr(qs + swz(r, ch)), src, valid);
        }
    }
    load_kv_tile(p, b, g, k0, 0, kend, ks[0], vs[0], bad);
    cp_async_commit();

    float oacc[D / 8][4];
#pragma unroll
    for (int i = 0; i < D / 8; ++i) oacc[i][0] = oacc[i][1] = oacc[i][2] = oacc[i][3] = 0.f;
    float mrow[2] = {-INFINITY, -INFINITY};
    float lrow[2] = {0.f, 0.f};
    uint32_t qa[D / 16][4];
    const int wrow = warp * 16;                        // first tile row of this warp
    const int pos0 = offset + m0 + wrow + (lane >> 2); // absolute position of this thread's first row

    for (int jt = 0; jt < ntiles; ++jt) {
        const int cur = jt & 1;
        if (jt + 1 < ntiles) {
            load_kv_tile(p, b, g, k0, (jt + 1) * BN, kend, ks[cur ^ 1], vs[cur ^ 1], bad);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        if (jt == 0) {
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
                const int r = wrow + (lane & 7) + ((lane >> 3) & 1) * 8;
                const int ch = kk * 2 + (lane >> 4);
                ldsm_x4(smem_addr(qs + swz(r, ch)), qa[kk][0], qa[kk][1], qa[kk][2], qa[kk][3]);
            }
        }
        const int j0 = jt * BN;
        // rows of this warp whose last visible key precedes the tile skip it
        if (j0 <= offset + m0 + wrow + 15) {
            float sacc[BN / 8][4];
#pragma unroll
            for (int i = 0; i < BN / 8; ++i) sacc[i][0] = sacc[i][1] = sacc[i][2] = sacc[i][3] = 0.f;
#pragma unroll
            for (int kk = 0; kk < D / 16; ++kk) {
#pragma unroll
                for (int np = 0; np < BN / 16; ++np) {
                    const int r = np * 16 + (lane & 7) + (lane >> 4) * 8;
                    const int ch = kk * 2 + ((lane >> 3) & 1);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4(smem_addr(ks[cur] + swz(r, ch)), b0, b1, b2, b3);
                    mma_bf16(sacc[2 * np], qa[kk], b0, b1);
                    mma_bf16(sacc[2 * np + 1], qa[kk], b2, b3);
                }
            }
            // scale, causal mask, online softmax
            const bool diag = j0 + BN - 1 > offset + m0 + wrow;
            float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    float sv = sacc[nt][e] * p.scale_log2;
                    if (diag) {
                        const int key = j0 + nt * 8 + (lane & 3) * 2 + (e & 1);
                        const int pos = pos0 + (e >> 1) * 8;
                        if (key > pos) sv = -INFINITY;
                    }
                    sacc[nt][e] = sv;
                    mx[e >> 1] = fmaxf(mx[e >> 1], sv);
                }
            }
            float alpha[2];
#pragma unroll
            for (int r = 0; r < 2; ++r) {
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
                mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
                const float mnew = fmaxf(mrow[r], mx[r]);
                // a row with no visible key so far keeps m = -inf; avoid (-inf) - (-inf)
                const float msafe = mnew == -INFINITY ? 0.f : mnew;
                alpha[r] = exp2f(mrow[r] - msafe);
                mrow[r] = mnew;
                mx[r] = msafe;
            }
            float rs[2] = {0.f, 0.f};
            uint32_t pa_[BN / 16][4];
#pragma unroll
            for (int nt = 0; nt < BN / 8; ++nt) {
                const float p0 = exp2f(sacc[nt][0] - mx[0]);
                const float p1 = exp2f(sacc[nt][1] - mx[0]);
                const float p2 = exp2f(sacc[nt][2] - mx[1]);
                const float p3 = exp2f(sacc[nt][3] - mx[1]);
                rs[0] += p0 + p1;
                rs[1] += p2 + p3;
                pa_[nt >> 1][(nt & 1) * 2 + 0] = pa::pack_bf16x2(p0, p1);
                pa_[nt >> 1][(nt & 1) * 2 + 1] = pa::pack_bf16x2(p2, p3);
            }
            lrow[0] = lrow[0] * alpha[0] + rs[0];
            lrow[1] = lrow[1] * alpha[1] + rs[1];
#pragma unroll
            for (int i = 0; i < D / 8; ++i) {
                oacc[i][0] *= alpha[0];
                oacc[i][1] *= alpha[0];
                oacc[i][2] *= alpha[1];
                oacc[i][3] *= alpha[1];
            }
#pragma unroll
            for (int s2 = 0; s2 < BN / 16; ++s2) {
#pragma unroll
                for (int dp = 0; dp < D / 16; ++dp) {
                    const int r = s2 * 16 + (lane & 7) + ((lane >> 3) & 1) * 8;
                    const int ch = dp * 2 + (lane >> 4);
                    uint32_t b0, b1, b2, b3;
                    ldsm_x4_t(smem_addr(vs[cur] + swz(r, ch)), b0, b1, b2, b3);
                    mma_bf16(oacc[2 * dp], pa_[s2], b0, b1);
                    mma_bf16(oacc[2 * dp + 1], pa_[s2], b2, b3);
                }
            }
        }
        __syncthreads();
    }
    if (bad && (threadIdx.x & 15) == 0) pa::report(p.status, PA_ERR_BOUNDS);

    // finalize: O / l, bf16, rows below lq only
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 1);
        lrow[r] += __shfl_xor_sync(0xffffffffu, lrow[r], 2);
    }
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        const int row = wrow + (lane >> 2) + r * 8;
        if (row >= rows) continue;
        const float inv = 1.f / lrow[r];
        uint16_t *dst = p.out + (int64_t(q0 + m0 + row) * p.num_heads + h) * D + (lane & 3) * 2;
#pragma unroll
        for (int nt = 0; nt < D / 8; ++nt) {
            *reinterpret_cast<uint32_t *>(dst + nt * 8) =
                pa::pack_bf16x2(oacc[nt][2 * r] * inv, oacc[nt][2 * r + 1] * inv);
        }
    }
}

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
    if (!pa::aligned(out, 4)) return PA_ERR_INVALID_ARG;
    if (block_table == nullptr) {
        if (!k || !v || max_seqlen_k != max_seqlen_q) return PA_ERR_INVALID_ARG;
        if (kv_stride_tok < int64_t(num_kv_heads) * D || kv_stride_tok % 8 != 0 || !pa::aligned(k, 16) ||
            !pa::aligned(v, 16))
            return PA_ERR_INVALID_ARG;
    } else {
        if (!k_cache || !v_cache || max_blocks_per_seq < 1) return PA_ERR_INVALID_ARG;
        if (!pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
    }
    if (num_seqs > 65535 || num_heads > 65535) return PA_ERR_UNSUPPORTED;

    PrefillParams p;
    p.q = static_cast<const uint16_t *>(q);
    p.q_stride = q_stride_tok;
    p.k = static_cast<const uint16_t *>(k);
    p.v = static_cast<const uint16_t *>(v);
    p.kv_stride = kv_stride_tok;
    p.k_cache = static_cast<const uint16_t *>(k_cache);
    p.v_cache = static_cast<const uint16_t *>(v_cache);
    p.num_blocks = num_blocks;
    p.block_size = block_size;
    p.block_table = block_table;
    p.max_blocks = max_blocks_per_seq;
    p.cu_q = cu_seqlens_q;
    p.cu_k = cu_seqlens_k;
    p.max_q = max_seqlen_q;
    p.num_heads = num_heads;
    p.kv_heads = num_kv_heads;
    p.scale_log2 = scale * LOG2E;
    p.out = static_cast<uint16_t *>(out);
    p.status = dev_status;

    static bool attr_set = false;  // per process; harmless to repeat
    if (!attr_set) {
        if (cudaFuncSetAttribute(prefill_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, SMEM_BYTES) !=
            cudaSuccess)
            return PA_ERR_CUDA;
        attr_set = true;
    }
    const dim3 grid(unsigned((max_seqlen_q + BM - 1) / BM), unsigned(num_heads), unsigned(num_seqs));
    prefill_mma_kernel<<<grid, NTHREAD, SMEM_BYTES, static_cast<cudaStream_t>(stream)>>>(p);
    return pa::launch_status();
}
