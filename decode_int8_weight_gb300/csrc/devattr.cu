// Per-device kernel attributes (host side of libq3i8.so).
//
// cudaFuncSetAttribute applies to the current device only, so a kernel that
// needs more than the default 48 KB of dynamic shared memory must be opted in
// once on every device it runs on.  The record of which (kernel, device)
// pairs are done is shared by all threads of the process.
#include <mutex>
#include <set>
#include <utility>

#include "kernels.h"

namespace q3 {

cudaError_t allow_max_dynamic_smem(const void* fn) {
    static std::mutex mu;
    static std::set<std::pair<const void*, int>> done;
    int dev = -1;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (done.count({fn, dev})) return cudaSuccess;
    int optin = 0;
    e = cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    if (e != cudaSuccess) return e;
    cudaFuncAttributes fa;
    e = cudaFuncGetAttributes(&fa, fn);
    if (e != cudaSuccess) return e;
    // the limit covers the kernel's static shared memory too
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, optin - (int)fa.sharedSizeBytes);
    if (e != cudaSuccess) return e;
    done.insert({fn, dev});
    return cudaSuccess;
}

}  // namespace q3
