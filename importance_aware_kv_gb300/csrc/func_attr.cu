// Kernel attribute settings made once per (kernel, device), from any thread.
//
// cudaFuncSetAttribute applies to the kernel on the current device, so a
// plain "already set" flag would skip the second device a process uses; the
// settings and the occupancy queries are kept in mutex-guarded tables keyed by
// kernel and device instead.
#include <map>
#include <mutex>
#include <tuple>

#include "hikv_internal.cuh"

namespace hikv {
namespace {

std::mutex g_attr_mu;
std::map<std::pair<const void*, int>, size_t> g_smem;                          // dynamic smem opted into
std::map<std::pair<const void*, int>, bool> g_nonportable;                     // cluster sizes above 8 allowed
std::map<std::tuple<const void*, int, int, size_t>, int> g_active;             // (kernel, device, cs, smem)

int current_device() {
    int d = 0;
    cudaGetDevice(&d);
    return d;
}

}  // namespace

cudaError_t func_smem_optin(const void* func, size_t bytes) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_attr_mu);
    size_t& have = g_smem[{func, dev}];
    if (bytes <= have) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) have = bytes;
    return e;
}

cudaError_t func_allow_nonportable_clusters(const void* func) {
    const int dev = current_device();
    std::lock_guard<std::mutex> lk(g_attr_mu);
    bool& done = g_nonportable[{func, dev}];
    if (done) return cudaSuccess;
    const cudaError_t e = cudaFuncSetAttribute(func, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) done = true;
    return e;
}

int func_active_clusters(const void* func, int cs, const cudaLaunchConfig_t& cfg) {
    const int dev = current_device();
    const auto key = std::make_tuple(func, dev, cs, (size_t)cfg.dynamicSmemBytes);
    {
        std::lock_guard<std::mutex> lk(g_attr_mu);
        auto it = g_active.find(key);
        if (it != g_active.end()) return it->second;
    }
    int active = 0;
    if (cudaOccupancyMaxActiveClusters(&active, func, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;   // not cached: a later call asks again
    }
    std::lock_guard<std::mutex> lk(g_attr_mu);
    g_active[key] = active;
    return active;
}

}  // namespace hikv
