// Streaming greedy argmax: out[r] = smallest index of max logits[r, :].
//
// A cluster of s CTAs shares each row; every CTA streams its slice once with
// 16-byte non-temporal loads (four in flight per thread), keeps a running
// (max, first index) per thread, reduces it across the CTA with warp shuffles
// and across the cluster through distributed shared memory.  Nothing is
// staged in shared memory, so many CTAs stay resident per SM.
#pragma once

#include "arc_device.cuh"

namespace arc {

struct ArgmaxArgs {
    const void* logits;
    int64_t ld;
    int V;
    int L;  // slice elements per CTA (multiple of the vector width)
    int aligned;
    int32_t* out;
    uint32_t* err_word;
};

template <int DT>
__global__ void __launch_bounds__(kThreads) argmax_kernel(const ArgmaxArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int U = 4;
    __shared__ uint64_t red[kWarps];
    __shared__ uint64_t slot[2];
    cg::cluster_group cl = cg::this_cluster();
    const int s = static_cast<int>(cl.num_blocks()), rank = static_cast<int>(cl.block_rank());
    const int row = blockIdx.x / s;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int a0 = rank * a.L, a1 = min(a0 + a.L, a.V);
    const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;

    float bv = -INFINITY;
    int bi = -1;
    bool nanf = false;
    auto take = [&](float z, int i) {
        nanf |= (z != z);
        if (z > bv) {
            bv = z;
            bi = i;
        }
    };
    int tail0 = a0;
    if (a.aligned && a1 > a0) {
        const int nvf = (a1 - a0) / VEC;
        const uint4* vp = reinterpret_cast<const uint4*>(rowp + static_cast<int64_t>(a0) * E::kBytes);
        int v = tid;
        for (; v + (U - 1) * kThreads < nvf; v += U * kThreads) {
            uint4 r[U];
#pragma unroll
            for (int u = 0; u < U; ++u) r[u] = ld_nc_v4(vp + v + u * kThreads);
#pragma unroll
            for (int u = 0; u < U; ++u) {
                float z[VEC];
                E::unpack(r[u], z);
                const int g = a0 + (v + u * kThreads) * VEC;
#pragma unroll
                for (int e = 0; e < VEC; ++e) take(z[e], g + e);
            }
        }
        for (; v < nvf; v += kThreads) {
            float z[VEC];
            E::unpack(ld_nc_v4(vp + v), z);
            const int g = a0 + v * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e) take(z[e], g + e);
        }
        tail0 = a0 + nvf * VEC;
    }
    for (int i = tail0 + tid; i < a1; i += kThreads) take(E::load_scalar(rowp, i), i);

    warp_argmax(bv, bi);
    const bool wnan = __any_sync(0xFFFFFFFFu, nanf);
    if (lane == 0) red[warp] = (static_cast<uint64_t>(static_cast<uint32_t>(bi)) << 32) | __float_as_uint(bv);
    __shared__ uint32_t nan_flag;
    if (tid == 0) nan_flag = 0;
    __syncthreads();
    if (lane == 0 && wnan) atomicOr(&nan_flag, 1u);
    __syncthreads();
    if (tid == 0) {
        float v = -INFINITY;
        int i = -1;
        for (int w = 0; w < kWarps; ++w)
            better(v, i, __uint_as_float(static_cast<uint32_t>(red[w])), static_cast<int>(red[w] >> 32));
        slot[0] = (static_cast<uint64_t>(static_cast<uint32_t>(i)) << 32) | __float_as_uint(v);
        slot[1] = nan_flag;
    }
    cl.sync();
    if (rank == 0 && warp == 0) {
        float v = -INFINITY;
        int i = -1;
        uint32_t f = 0;
        if (lane < s) {
            const uint64_t* rs = cl.map_shared_rank(slot, lane);
            const uint64_t x = rs[0];
            v = __uint_as_float(static_cast<uint32_t>(x));
            i = static_cast<int>(x >> 32);
            f = static_cast<uint32_t>(rs[1]);
        }
        warp_argmax(v, i);
        f = __reduce_or_sync(0xFFFFFFFFu, f);
        if (lane == 0) {
            uint32_t err = f ? ARC_ERR_NAN : 0u;
            if (i < 0) {
                i = 0;
                err |= ARC_ERR_DEGENERATE;
            }
            a.out[row] = i;
            if (err && a.err_word) atomicOr(a.err_word, err);
        }
    }
    cl.sync();
}

}  // namespace arc
