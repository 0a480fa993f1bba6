// Definitions of KernelSet (kernel_set.cuh), included only by the
// translation units that instantiate one (dtype, history) pair.
#pragma once

#include <algorithm>
#include <atomic>

#include "kernel_set.cuh"
#include "launch_util.cuh"

namespace arc {

template <int DT, bool HIST>
struct KernelPrep {
    static std::atomic<uint64_t> scan, fin, cluster;  // per-device "attributes set" bits
};
template <int DT, bool HIST>
std::atomic<uint64_t> KernelPrep<DT, HIST>::scan{0};
template <int DT, bool HIST>
std::atomic<uint64_t> KernelPrep<DT, HIST>::fin{0};
template <int DT, bool HIST>
std::atomic<uint64_t> KernelPrep<DT, HIST>::cluster{0};

template <int DT, bool HIST>
cudaError_t KernelSet<DT, HIST>::launch_two(const ScanArgs& sa, const FinishArgs& fa, int s, int64_t B,
                                            int scan_smem, int fin_smem, int dev, cudaStream_t st) {
    // carveout 0 for the streaming scan (a larger L1 keeps more loads in
    // flight) unless it stages penalty tables in shared memory
    cudaError_t err = prepare(scan_kernel<DT, HIST>, dev, KernelPrep<DT, HIST>::scan, HIST ? 100 : 0);
    if (err == cudaSuccess) err = prepare(finish_kernel<DT, HIST>, dev, KernelPrep<DT, HIST>::fin, 100);
    if (err != cudaSuccess) return err;
    // slices x rows; rows past 65,535 fold into z (grid y is 16-bit)
    const unsigned gy = static_cast<unsigned>(std::min<int64_t>(B, 65535));
    const unsigned gz = static_cast<unsigned>((B + gy - 1) / gy);
    scan_kernel<DT, HIST><<<dim3(static_cast<unsigned>(s), gy, gz), kThreads, scan_smem, st>>>(sa);
    err = cudaGetLastError();
    if (err == cudaSuccess)
        err = launch_cluster(finish_kernel<DT, HIST>, B * fa.fin_g, fa.fin_g, fin_smem, st, fa, /*early=*/true);
    return err;
}

template <int DT, bool HIST>
bool KernelSet<DT, HIST>::finish_cluster_ok(int g, int smem, int dev) {
    return prepare(finish_kernel<DT, HIST>, dev, KernelPrep<DT, HIST>::fin, 100) == cudaSuccess &&
           cluster_fits(finish_kernel<DT, HIST>, dev, DT + 2, HIST, g, smem);
}

template <int DT, bool HIST>
bool KernelSet<DT, HIST>::cluster_ok(int s, int dyn, int dev) {
    return prepare(cluster_kernel<DT, HIST>, dev, KernelPrep<DT, HIST>::cluster, 100) == cudaSuccess &&
           cluster_fits(cluster_kernel<DT, HIST>, dev, DT, HIST, s, dyn);
}

template <int DT, bool HIST>
cudaError_t KernelSet<DT, HIST>::launch_fused(const FusedArgs& fu, int64_t B, int s, int dyn, cudaStream_t st) {
    return launch_cluster(cluster_kernel<DT, HIST>, B * s, s, dyn, st, fu);
}

}  // namespace arc
