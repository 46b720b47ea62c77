// store_kvcache.cu -- the KV write: scatter each new token's K and V rows into
// the paged pool at the row named by slot_mapping.
//
// "大模型推理入门与 nano-vLLM 源码详解" §13.1: the Hkv heads of one token are one
// contiguous row of Hkv * head_dim values; row `slot` of the layer's cache
// receives it, and slot == -1 (a padded row) is skipped.
//
// Design: a pure copy bound by HBM bandwidth (2 x 2 KiB read + 2 x 2 KiB
// written per token at Hkv = 8, head_dim = 128).  A CTA of 256 threads moves
// whole rows with 16-byte vectors; the work of one token is a power-of-two
// number of vectors (Hkv * head_dim / 8 for each of K and V), so token and
// vector indices come from shifts, and each vector is one coalesced 16-byte
// load and store.  Sources whose base or stride is not 16-byte aligned fall
// back to 4- or 2-byte vectors.
#include <cuda_fp8.h>

#include "pa_common.cuh"

namespace {

template <int VEC>
struct Vec;
template <>
struct Vec<16> { using T = uint4; };
template <>
struct Vec<4> { using T = uint32_t; };
template <>
struct Vec<2> { using T = uint16_t; };

template <int VEC>
__device__ __forceinline__ typename Vec<VEC>::T load_once(const char *p)
{
    if constexpr (VEC == 16) {
        return pa::ld_stream16(p);
    } else {
        return *reinterpret_cast<const typename Vec<VEC>::T *>(p);
    }
}

// One thread per (token, K-or-V, vector).  log2_vecs = log2(row_bytes / VEC).
template <int VEC>
__global__ void __launch_bounds__(256)
store_kvcache_kernel(const char *__restrict__ k, int64_t k_stride_bytes,
                     const char *__restrict__ v, int64_t v_stride_bytes,
                     int64_t num_tokens, int log2_vecs, char *__restrict__ k_cache,
                     char *__restrict__ v_cache, int64_t num_slots, int64_t row_bytes,
                     const int32_t *__restrict__ slot_mapping, int32_t *status)
{
    using T = typename Vec<VEC>::T;
    // launched programmatically: the previous kernel's writes (a decode that
    // read the pool, the projection that wrote k / v) are complete only after this
    pa::grid_dependency_wait();
    pa::grid_dependents_launch();  // a short kernel: the next one may launch now
    const int64_t per_token = int64_t(2) << log2_vecs;
    const int64_t total = num_tokens * per_token;
    const int64_t step = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
        const int64_t t = i >> (log2_vecs + 1);
        const int r = int(i & (per_token - 1));
        const bool is_v = (r >> log2_vecs) != 0;
        const int64_t vec = r & ((1 << log2_vecs) - 1);
        const int64_t slot = slot_mapping[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) {
            if (r == 0) pa::report(status, PA_ERR_BOUNDS);
            continue;
        }
        const char *src = is_v ? v + t * v_stride_bytes : k + t * k_stride_bytes;
        char *dst = (is_v ? v_cache : k_cache) + slot * row_bytes;
        const T x = load_once<VEC>(src + vec * VEC);
        *reinterpret_cast<T *>(dst + vec * VEC) = x;
    }
}

template <int VEC>
void launch(const void *k, int64_t ks, const void *v, int64_t vs, int64_t num_tokens, int64_t row_bytes,
            void *kc, void *vc, int64_t num_slots, const int32_t *slots, int32_t *status, cudaStream_t stream)
{
    int log2_vecs = 0;
    while ((int64_t(VEC) << log2_vecs) < row_bytes) ++log2_vecs;
    const int64_t total = num_tokens * (int64_t(2) << log2_vecs);
    const int threads = 256;
    int64_t blocks = (total + threads - 1) / threads;
    const int64_t cap = int64_t(pa::num_sms() > 0 ? pa::num_sms() : 152) * 64;
    if (blocks > cap) blocks = cap;
    pa::launch_pdl(store_kvcache_kernel<VEC>, dim3(unsigned(blocks)), dim3(threads), 0, stream,
                   static_cast<const char *>(k), ks * 2, static_cast<const char *>(v), vs * 2, num_tokens, log2_vecs,
                   static_cast<char *>(kc), static_cast<char *>(vc), num_slots, row_bytes, slots, status);
}

}  // namespace

extern "C" pa_status pa_store_kvcache(const void *k, int64_t k_stride_tok, const void *v, int64_t v_stride_tok,
                                      int64_t num_tokens, int num_kv_heads, int head_dim, void *k_cache,
                                      void *v_cache, int64_t num_blocks, int block_size,
                                      const int32_t *slot_mapping, int32_t *dev_status, void *stream)
{
    if (num_tokens < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (head_dim != pa::kHeadDim || !pa::pow2_in(num_kv_heads, 1, 8)) return PA_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 1024 || block_size % 16 != 0) return PA_ERR_UNSUPPORTED;
    const int64_t row = int64_t(num_kv_heads) * head_dim;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (k_stride_tok < row || v_stride_tok < row) return PA_ERR_INVALID_ARG;
    if (!pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16)) return PA_ERR_INVALID_ARG;
    const int64_t num_slots = num_blocks * block_size;
    const int64_t row_bytes = row * 2;
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    const bool a16 = pa::aligned(k, 16) && pa::aligned(v, 16) && (k_stride_tok % 8 == 0) && (v_stride_tok % 8 == 0);
    const bool a4 = pa::aligned(k, 4) && pa::aligned(v, 4) && (k_stride_tok % 2 == 0) && (v_stride_tok % 2 == 0);
    if (a16)
        launch<16>(k, k_stride_tok, v, v_stride_tok, num_tokens, row_bytes, k_cache, v_cache, num_slots,
                   slot_mapping, dev_status, s);
    else if (a4)
        launch<4>(k, k_stride_tok, v, v_stride_tok, num_tokens, row_bytes, k_cache, v_cache, num_slots,
                  slot_mapping, dev_status, s);
    else
        launch<2>(k, k_stride_tok, v, v_stride_tok, num_tokens, row_bytes, k_cache, v_cache, num_slots,
                  slot_mapping, dev_status, s);
    return pa::launch_status();
}

// ---------------------------------------------------------------------------
// KV write into an fp8 pool.
//
// Each element is stored as the OCP FP8 E4M3 code of x / scale (division in
// fp32, round to nearest even, saturating to +-448), one byte; a layer's K
// and V each carry one scale.  The pages name the KV precision as the lever
// for fitting longer contexts ("大模型推理入门与 nano-vLLM 源码详解" §17.3) and
// count FP8 at one byte per element ("VLLM on Fain的Blog", arithmetic
// intensity table); the E4M3 format and per-tensor scales are this library's
// choice.  One thread per (token, K-or-V, 16 elements): 32 bytes of bf16 in,
// 16 bytes of codes out.

namespace {

__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d, float scale)
{
    const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(a, scale), __fdiv_rn(b, scale)),
                                                 __NV_SATFINITE, __NV_E4M3);
    const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(__fdiv_rn(c, scale), __fdiv_rn(d, scale)),
                                                 __NV_SATFINITE, __NV_E4M3);
    return lo | (hi << 16);
}

__device__ __forceinline__ uint2 quant8(const uint4 &u, float scale)
{
    return make_uint2(e4m3x4(pa::bf16_lo(u.x), pa::bf16_hi(u.x), pa::bf16_lo(u.y), pa::bf16_hi(u.y), scale),
                      e4m3x4(pa::bf16_lo(u.z), pa::bf16_hi(u.z), pa::bf16_lo(u.w), pa::bf16_hi(u.w), scale));
}

__global__ void __launch_bounds__(256)
store_kvcache_fp8_kernel(const uint16_t *__restrict__ k, int64_t k_stride, const uint16_t *__restrict__ v,
                         int64_t v_stride, int64_t num_tokens, int vecs_per_row, float k_scale, float v_scale,
                         uint8_t *__restrict__ k_cache, uint8_t *__restrict__ v_cache, int64_t num_slots,
                         int64_t row, const int32_t *__restrict__ slot_mapping, int32_t *status)
{
    const int64_t per_token = 2 * int64_t(vecs_per_row);
    const int64_t total = num_tokens * per_token;
    const int64_t step = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total; i += step) {
        const int64_t t = i / per_token;
        const int r = int(i - t * per_token);
        const bool is_v = r >= vecs_per_row;
        const int vec = is_v ? r - vecs_per_row : r;
        const int64_t slot = slot_mapping[t];
        if (slot == -1) continue;
        if (slot < 0 || slot >= num_slots) {
            if (r == 0) pa::report(status, PA_ERR_BOUNDS);
            continue;
        }
        const uint16_t *src = (is_v ? v + t * v_stride : k + t * k_stride) + vec * 16;
        const float scale = is_v ? v_scale : k_scale;
        const uint2 a = quant8(pa::ld_stream16(src), scale);
        const uint2 b = quant8(pa::ld_stream16(src + 8), scale);
        *reinterpret_cast<uint4 *>((is_v ? v_cache : k_cache) + slot * row + vec * 16) = make_uint4(a.x, a.y, b.x, b.y);
    }
}

}  // namespace

extern "C" pa_status pa_store_kvcache_fp8(const void *k, int64_t k_stride_tok, const void *v, int64_t v_stride_tok,
                                          int64_t num_tokens, int num_kv_heads, int head_dim, float k_scale,
                                          float v_scale, void *k_cache, void *v_cache, int64_t num_blocks,
                                          int block_size, const int32_t *slot_mapping, int32_t *dev_status,
                                          void *stream)
{
    if (num_tokens < 0 || num_blocks < 0) return PA_ERR_INVALID_ARG;
    if (head_dim != pa::kHeadDim || !pa::pow2_in(num_kv_heads, 1, 8)) return PA_ERR_UNSUPPORTED;
    if (block_size < 16 || block_size > 1024 || block_size % 16 != 0) return PA_ERR_UNSUPPORTED;
    if (!(k_scale > 0.f) || !(v_scale > 0.f) || isinf(k_scale) || isinf(v_scale)) return PA_ERR_INVALID_ARG;
    const int64_t row = int64_t(num_kv_heads) * head_dim;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    if (k_stride_tok < row || v_stride_tok < row || k_stride_tok % 8 != 0 || v_stride_tok % 8 != 0)
        return PA_ERR_INVALID_ARG;
    if (!pa::aligned(k, 16) || !pa::aligned(v, 16) || !pa::aligned(k_cache, 16) || !pa::aligned(v_cache, 16))
        return PA_ERR_INVALID_ARG;
    const int vecs = int(row / 16);
    const int64_t total = num_tokens * 2 * vecs;
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = int64_t(pa::num_sms() > 0 ? pa::num_sms() : 152) * 64;
    if (blocks > cap) blocks = cap;
    store_kvcache_fp8_kernel<<<dim3(unsigned(blocks)), 256, 0, static_cast<cudaStream_t>(stream)>>>(
        static_cast<const uint16_t *>(k), k_stride_tok, static_cast<const uint16_t *>(v), v_stride_tok, num_tokens,
        vecs, k_scale, v_scale, static_cast<uint8_t *>(k_cache), static_cast<uint8_t *>(v_cache),
        num_blocks * block_size, row, slot_mapping, dev_status);
    return pa::launch_status();
}
