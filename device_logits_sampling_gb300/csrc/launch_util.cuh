// Host-side launch helpers shared by the translation units that launch
// kernels: per-device function attributes, cluster launches (with optional
// programmatic dependent launch) and the cluster occupancy check.
#pragma once

#include <cuda_runtime.h>

#include <atomic>
#include <cstdint>
#include <cstring>
#include <map>
#include <mutex>
#include <tuple>

namespace arc {

constexpr int kSmemPerBlock = 232448;  // 227 KB opt-in limit of sm_100-class GPUs
constexpr int kLaunchThreads = 256;    // threads of every CTA of the library's kernels

// Function attributes are set once per (device, kernel): the first call on a
// device must come before any stream capture that contains a call.
// `carveout` is the preferred shared-memory share of the SM's L1/shared
// storage in percent: 0 for the streaming kernels, which use (almost) no
// shared memory and keep more loads in flight with a larger L1, 100 for
// the kernels that stage rows or penalty tables in shared memory.
template <class K>
inline cudaError_t prepare(K kernel, int dev, std::atomic<uint64_t>& done, int carveout) {
    const uint64_t bit = uint64_t{1} << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    // the largest dynamic shared memory a CTA of this kernel can have next to
    // its static shared memory
    cudaFuncAttributes fa;
    cudaError_t e = cudaFuncGetAttributes(&fa, kernel);
    if (e == cudaSuccess)
        e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kSmemPerBlock - static_cast<int>(fa.sharedSizeBytes));
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e == cudaSuccess) e = cudaFuncSetAttribute(kernel, cudaFuncAttributePreferredSharedMemoryCarveout, carveout);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();  // a refused attribute must not surface as a later launch error
        return e;
    }
    done.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

template <class K, class A>
inline cudaError_t launch_cluster(K kernel, int64_t grid, int s, int smem, cudaStream_t st, const A& args,
                           bool early = false) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kLaunchThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // early: the kernel may start before the previous kernel on the stream has
    // finished (programmatic dependent launch); it waits for that kernel's
    // results with griddepcontrol.wait before reading them
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = early ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

// Whether a cluster launch of this kernel and shape fits the device (cached;
// asked once per device, kernel, cluster size and shared-memory size).
template <class K>
inline bool cluster_fits(K kernel, int dev, int dt, bool hist, int s, int smem) {
    static std::mutex mu;
    static std::map<std::tuple<int, int, int, int, int>, bool> known;
    const auto key = std::make_tuple(dev, dt, hist ? 1 : 0, s, smem);
    std::lock_guard<std::mutex> lock(mu);
    auto it = known.find(key);
    if (it != known.end()) return it->second;
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(s), 1, 1);
    cfg.blockDim = dim3(kLaunchThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    const bool ok = cudaOccupancyMaxActiveClusters(&n, kernel, &cfg) == cudaSuccess && n >= 1;
    if (!ok) (void)cudaGetLastError();
    known[key] = ok;
    return ok;
}


}  // namespace arc
