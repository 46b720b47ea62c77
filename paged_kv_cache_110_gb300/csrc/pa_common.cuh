// pa_common.cuh -- small device and host helpers shared by libpa's kernels.
#pragma once

#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "pa.h"

namespace pa {

constexpr int kHeadDim = 128;

// First nonzero code wins; later reports leave it unchanged.
__device__ __forceinline__ void report(int32_t *status, int code)
{
    if (status != nullptr) atomicCAS(status, 0, code);
}

// A bf16 pair packed in 32 bits: low element in bits 0..15.
__device__ __forceinline__ float bf16_lo(uint32_t u) { return __uint_as_float(u << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t u) { return __uint_as_float(u & 0xffff0000u); }

__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi)
{
    __nv_bfloat162 p = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&p);
}

// 16-byte global load that is read once: bypass L1 allocation.
__device__ __forceinline__ uint4 ld_stream16(const void *p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

inline bool aligned(const void *p, size_t bytes)
{
    return (reinterpret_cast<uintptr_t>(p) % bytes) == 0;
}

inline bool pow2_in(int x, int lo, int hi)
{
    return x >= lo && x <= hi && (x & (x - 1)) == 0;
}

// Number of SMs of the current device (cached per device).
int num_sms();

// PA_OK if cudaGetLastError() is clean, else PA_ERR_CUDA.
pa_status launch_status();

}  // namespace pa
