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

// Programmatic dependent launch.  A kernel launched with launch_pdl may start
// while the kernel before it in the stream is still finishing; it must call
// grid_dependency_wait() before it reads or writes anything that kernel (or
// any earlier work) may touch: the wait returns once the earlier grid has
// completed and its memory operations are visible.  Without a programmatic
// predecessor the wait returns at once.  grid_dependents_launch() lets the
// NEXT kernel start early (once every CTA of this one has called it or
// exited); its CTAs then occupy SM slots while they wait, so a long kernel
// calls it only near its end.
__device__ __forceinline__ void grid_dependency_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dependents_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                       Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
}

// launch_pdl with the grid cut into clusters of cluster_y CTAs along y
// (co-scheduled, sharing distributed shared memory).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl_cluster_y(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t stream,
                                 unsigned cluster_y, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = 1;
    attr[1].val.clusterDim.y = cluster_y;
    attr[1].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, kernel, static_cast<KArgs>(args)...);
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

// Let `kernel` use `bytes` of dynamic shared memory on the current device (an
// opt-in each device needs once; cached per device and kernel).  Callers pass
// the largest size any launch of that kernel uses.
cudaError_t allow_dynamic_smem(const void *kernel, int bytes);

// The limit, in SM cycles, of the waits inside a kernel's pipeline: `dflt`,
// unless a test set another with pa_test_stall_pipelines; and whether such a
// test asked one wait per CTA to be on a barrier nothing arrives on.
long long pipeline_wait_limit(long long dflt);
bool pipeline_test_stall();

// PA_OK if cudaGetLastError() is clean, else PA_ERR_CUDA.
pa_status launch_status();

}  // namespace pa
