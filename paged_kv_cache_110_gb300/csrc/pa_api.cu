// pa_api.cu -- status strings, sizes and device queries of libpa.
#include <atomic>
#include <mutex>
#include <set>
#include <utility>

#include "pa_common.cuh"

namespace pa {

int num_sms()
{
    static std::mutex mu;
    static int cached[64] = {0};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::lock_guard<std::mutex> lock(mu);
    if (cached[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
        cached[dev] = n;
    }
    return cached[dev];
}

cudaError_t allow_dynamic_smem(const void *kernel, int bytes)
{
    // the attribute belongs to the device current at the time of the call
    static std::mutex mu;
    static std::set<std::pair<const void *, int>> done;
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({kernel, dev}) != 0) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, bytes);
    if (e == cudaSuccess) done.insert({kernel, dev});
    return e;
}

namespace {
std::atomic<long long> g_test_wait_limit{0};
}

long long pipeline_wait_limit(long long dflt)
{
    const long long v = g_test_wait_limit.load(std::memory_order_relaxed);
    return v > 0 ? v : dflt;
}

bool pipeline_test_stall() { return g_test_wait_limit.load(std::memory_order_relaxed) > 0; }

pa_status launch_status()
{
    return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace pa

extern "C" const char *pa_status_string(int status)
{
    switch (status) {
    case PA_OK: return "ok";
    case PA_ERR_INVALID_ARG: return "invalid argument";
    case PA_ERR_UNSUPPORTED: return "unsupported shape";
    case PA_ERR_CUDA: return "CUDA error";
    case PA_ERR_BOUNDS: return "index out of bounds";
    case PA_ERR_TIMEOUT: return "bounded wait timed out";
    default: return "unknown status";
    }
}

extern "C" int pa_abi_version(void) { return 100; }

extern "C" void pa_test_stall_pipelines(long long cycles)
{
    pa::g_test_wait_limit.store(cycles > 0 ? cycles : 0, std::memory_order_relaxed);
}

extern "C" size_t pa_kv_bytes_per_token(int layers, int kv_heads, int head_dim, int elem_bytes)
{
    if (layers <= 0 || kv_heads <= 0 || head_dim <= 0 || elem_bytes <= 0) return 0;
    return (size_t)2 * layers * kv_heads * head_dim * elem_bytes;
}
