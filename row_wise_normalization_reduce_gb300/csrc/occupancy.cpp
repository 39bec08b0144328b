// occupancy.cpp -- resident CTAs per SM of a kernel, asked from the runtime
// once per (device, kernel, block size, dynamic shared memory) and cached, for
// the launchers that size grids to the resident capacity or set prefetch
// distances in waves of resident CTAs.
#include <cuda_runtime_api.h>

#include <map>
#include <mutex>
#include <tuple>
#include <utility>

#include "nrm_internal.h"

namespace nrm {

cudaError_t resident_ctas(const void *kernel, int threads, size_t smem, int *per_sm) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        cudaGetLastError();
        return cudaErrorInvalidDevice;
    }
    static std::mutex mu;
    static std::map<std::tuple<int, const void *, int, size_t>, int> cache;
    static std::map<std::pair<int, const void *>, size_t> smem_limit;  // raised so far
    std::lock_guard<std::mutex> lock(mu);
    const auto key = std::make_tuple(dev, kernel, threads, smem);
    const auto it = cache.find(key);
    if (it != cache.end()) {
        *per_sm = it->second;
        return cudaSuccess;
    }
    // the kernel's dynamic shared-memory limit only ever grows, so launches
    // sized earlier stay valid
    size_t &limit = smem_limit[std::make_pair(dev, kernel)];
    if (smem > limit) {
        const cudaError_t e =
            cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        limit = smem;
    }
    int n = 0;
    const cudaError_t e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, kernel, threads, smem);
    if (e != cudaSuccess) return e;
    cache.emplace(key, n);
    *per_sm = n;
    return cudaSuccess;
}

}  // namespace nrm
