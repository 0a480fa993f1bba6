// The sampling kernels of one (logit dtype, history) pair behind plain host
// functions.  Each pair is instantiated in a translation unit of its own
// (kernels_<dtype>[_hist].cu), so the four compile in parallel; the C ABI
// (arc_sample.cu) sees only these declarations.
#pragma once

#include <cuda_runtime.h>

#include <cstdint>

#include "stream_kernel.cuh"

namespace arc {

template <int DT, bool HIST>
struct KernelSet {
    // scan_kernel over B rows of s slices, then finish_kernel (fa.fin_g CTAs
    // per row, a cluster) behind it under programmatic dependent launch; sets
    // the kernels' attributes on the first call on a device
    static cudaError_t launch_two(const ScanArgs& sa, const FinishArgs& fa, int s, int64_t B, int scan_smem,
                                  int fin_smem, int dev, cudaStream_t st);
    // whether finish_kernel with clusters of g CTAs per row and `smem` bytes
    // of dynamic shared memory can run on the device (attributes set, cached)
    static bool finish_cluster_ok(int g, int smem, int dev);
    // whether cluster_kernel with clusters of s CTAs and `dyn` bytes of
    // dynamic shared memory can run on the device (attributes set, cached)
    static bool cluster_ok(int s, int dyn, int dev);
    // cluster_kernel: B clusters of s CTAs, one launch (cluster_ok first)
    static cudaError_t launch_fused(const FusedArgs& fu, int64_t B, int s, int dyn, cudaStream_t st);
};

}  // namespace arc
