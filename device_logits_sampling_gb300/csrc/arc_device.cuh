// Device primitives for the sm_103a sampler: 16-byte global loads and
// asynchronous global -> shared copies, order-preserving float keys, the
// Splitmix64 generator, fixed-point scaling and warp reductions.
#pragma once

#include <cooperative_groups.h>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

#include "arc_sample.h"

namespace arc {
namespace cg = cooperative_groups;

constexpr int kThreads = 256;              // threads per CTA
constexpr int kWarps = kThreads / 32;
constexpr int kBins = 512;                 // histogram bins per select pass
constexpr int kBinBits = 9;
constexpr int kCand = 256;                 // crossing-bin candidates gathered per row
constexpr int kMaxCluster = 16;

// ------------------------------------------------------------------ PTX
// IEEE max that propagates NaN (max.NaN, sm_80+).
__device__ __forceinline__ float fmax_nan(float a, float b) {
    float r;
    asm("max.NaN.f32 %0, %1, %2;" : "=f"(r) : "f"(a), "f"(b));
    return r;
}

__device__ __forceinline__ float ex2(float x) {
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ uint4 ld_nc_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// ------------------------------------------------------------------ keys
// Order-preserving u32 key of a non-NaN float, reading -0 as +0.
__device__ __forceinline__ uint32_t fkey(float z) {
    const uint32_t b = __float_as_uint(__fadd_rn(z, 0.0f));
    return (b & 0x80000000u) ? ~b : (b | 0x80000000u);
}

__device__ __forceinline__ float key_to_float(uint32_t k) {
    const uint32_t b = (k & 0x80000000u) ? (k & 0x7FFFFFFFu) : ~k;
    return __uint_as_float(b);
}

// ------------------------------------------------------------------ generator
// Splitmix64 (Steele, Lea, Flood 2014): one output for state x.
__device__ __forceinline__ uint64_t splitmix64(uint64_t x) {
    uint64_t z = x + 0x9E3779B97F4A7C15ull;
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// floor(rbits * mass / 2^53) exactly (128-bit product).
__device__ __forceinline__ uint64_t scale_by_u(uint64_t rbits, uint64_t mass) {
    const uint64_t lo = rbits * mass;
    const uint64_t hi = __umul64hi(rbits, mass);
    return (hi << 11) | (lo >> 53);
}

// ------------------------------------------------------------------ element loads
template <int DT>
struct Elem;

template <>
struct Elem<ARC_F32> {
    static constexpr int kVec = 4;    // elements per 16-byte vector
    static constexpr int kBytes = 4;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&z)[4]) {
        z[0] = __uint_as_float(v.x);
        z[1] = __uint_as_float(v.y);
        z[2] = __uint_as_float(v.z);
        z[3] = __uint_as_float(v.w);
    }
    // max of the vector, propagating NaN
    __device__ __forceinline__ static float vmax_nan(const uint4& v) {
        return fmax_nan(fmax_nan(__uint_as_float(v.x), __uint_as_float(v.y)),
                        fmax_nan(__uint_as_float(v.z), __uint_as_float(v.w)));
    }
    __device__ __forceinline__ static float load_scalar(const void* row, int64_t i) {
        return __ldg(reinterpret_cast<const float*>(row) + i);
    }
    // vector v of a slice in global memory holding n elements; elements past
    // n read as -inf; 16-byte load when the slice start is 16-byte aligned
    __device__ __forceinline__ static uint4 global_vec(const void* base, int v, int n, bool aligned) {
        if (aligned && (v + 1) * 4 <= n) return ld_nc_v4(static_cast<const char*>(base) + static_cast<size_t>(v) * 16);
        const uint32_t* p = static_cast<const uint32_t*>(base);
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const int i = v * 4 + e;
            w[e] = (i < n) ? __ldg(p + i) : 0xFF800000u;
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Elem<ARC_BF16> {
    static constexpr int kVec = 8;
    static constexpr int kBytes = 2;
    __device__ __forceinline__ static void unpack(const uint4& v, float (&z)[8]) {
        z[0] = __uint_as_float(v.x << 16);
        z[1] = __uint_as_float(v.x & 0xFFFF0000u);
        z[2] = __uint_as_float(v.y << 16);
        z[3] = __uint_as_float(v.y & 0xFFFF0000u);
        z[4] = __uint_as_float(v.z << 16);
        z[5] = __uint_as_float(v.z & 0xFFFF0000u);
        z[6] = __uint_as_float(v.w << 16);
        z[7] = __uint_as_float(v.w & 0xFFFF0000u);
    }
    // max of the vector, propagating NaN (packed bf16x2 max, exact)
    __device__ __forceinline__ static float vmax_nan(const uint4& v) {
        const __nv_bfloat162 a = *reinterpret_cast<const __nv_bfloat162*>(&v.x);
        const __nv_bfloat162 b = *reinterpret_cast<const __nv_bfloat162*>(&v.y);
        const __nv_bfloat162 c = *reinterpret_cast<const __nv_bfloat162*>(&v.z);
        const __nv_bfloat162 d = *reinterpret_cast<const __nv_bfloat162*>(&v.w);
        const __nv_bfloat162 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        return fmax_nan(__low2float(m), __high2float(m));
    }
    __device__ __forceinline__ static float load_scalar(const void* row, int64_t i) {
        const unsigned short h = __ldg(reinterpret_cast<const unsigned short*>(row) + i);
        return __uint_as_float(static_cast<uint32_t>(h) << 16);
    }
    // vector v of a slice in global memory holding n elements; elements past
    // n read as -inf; 16-byte load when the slice start is 16-byte aligned
    __device__ __forceinline__ static uint4 global_vec(const void* base, int v, int n, bool aligned) {
        if (aligned && (v + 1) * 8 <= n) return ld_nc_v4(static_cast<const char*>(base) + static_cast<size_t>(v) * 16);
        const unsigned short* p = static_cast<const unsigned short*>(base);
        uint32_t w[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
            const int i = v * 8 + 2 * h;
            const uint32_t lo = (i < n) ? __ldg(p + i) : 0xFF80u;
            const uint32_t hi = (i + 1 < n) ? __ldg(p + i + 1) : 0xFF80u;
            w[h] = lo | (hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

template <>
struct Elem<ARC_F16> {
    static constexpr int kVec = 8;
    static constexpr int kBytes = 2;
    __device__ __forceinline__ static float h(uint32_t bits) {  // exact widening
        return __half2float(__ushort_as_half(static_cast<unsigned short>(bits)));
    }
    __device__ __forceinline__ static void unpack(const uint4& v, float (&z)[8]) {
        z[0] = h(v.x & 0xFFFFu);
        z[1] = h(v.x >> 16);
        z[2] = h(v.y & 0xFFFFu);
        z[3] = h(v.y >> 16);
        z[4] = h(v.z & 0xFFFFu);
        z[5] = h(v.z >> 16);
        z[6] = h(v.w & 0xFFFFu);
        z[7] = h(v.w >> 16);
    }
    // max of the vector, propagating NaN (packed half2 max, exact)
    __device__ __forceinline__ static float vmax_nan(const uint4& v) {
        const __half2 a = *reinterpret_cast<const __half2*>(&v.x);
        const __half2 b = *reinterpret_cast<const __half2*>(&v.y);
        const __half2 c = *reinterpret_cast<const __half2*>(&v.z);
        const __half2 d = *reinterpret_cast<const __half2*>(&v.w);
        const __half2 m = __hmax2_nan(__hmax2_nan(a, b), __hmax2_nan(c, d));
        return fmax_nan(__low2float(m), __high2float(m));
    }
    __device__ __forceinline__ static float load_scalar(const void* row, int64_t i) {
        return h(__ldg(reinterpret_cast<const unsigned short*>(row) + i));
    }
    // vector v of a slice in global memory holding n elements; elements past
    // n read as -inf; 16-byte load when the slice start is 16-byte aligned
    __device__ __forceinline__ static uint4 global_vec(const void* base, int v, int n, bool aligned) {
        if (aligned && (v + 1) * 8 <= n) return ld_nc_v4(static_cast<const char*>(base) + static_cast<size_t>(v) * 16);
        const unsigned short* p = static_cast<const unsigned short*>(base);
        uint32_t w[4];
#pragma unroll
        for (int k = 0; k < 4; ++k) {
            const int i = v * 8 + 2 * k;
            const uint32_t lo = (i < n) ? __ldg(p + i) : 0xFC00u;
            const uint32_t hi = (i + 1 < n) ? __ldg(p + i + 1) : 0xFC00u;
            w[k] = lo | (hi << 16);
        }
        return make_uint4(w[0], w[1], w[2], w[3]);
    }
};

// ------------------------------------------------------------------ warp helpers
__device__ __forceinline__ uint64_t shfl_u64(uint64_t v, int src) {
    const uint32_t lo = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), src);
    const uint32_t hi = __shfl_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), src);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t shfl_up_u64(uint64_t v, int d) {
    const uint32_t lo = __shfl_up_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), d);
    const uint32_t hi = __shfl_up_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), d);
    return (static_cast<uint64_t>(hi) << 32) | lo;
}

__device__ __forceinline__ uint64_t warp_sum_u64(uint64_t v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const uint32_t lo = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v), d);
        const uint32_t hi = __shfl_xor_sync(0xFFFFFFFFu, static_cast<uint32_t>(v >> 32), d);
        v += (static_cast<uint64_t>(hi) << 32) | lo;
    }
    return v;
}

__device__ __forceinline__ uint64_t warp_inclusive_u64(uint64_t v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint64_t o = shfl_up_u64(v, d);
        if (lane >= d) v += o;
    }
    return v;
}

// (value, index) max with ties to the smaller index; -1 index means "none".
__device__ __forceinline__ void better(float& v, int& i, float v2, int i2) {
    if (i2 >= 0 && (i < 0 || v2 > v || (v2 == v && i2 < i))) {
        v = v2;
        i = i2;
    }
}

__device__ __forceinline__ void warp_argmax(float& v, int& i) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) {
        const float v2 = __shfl_xor_sync(0xFFFFFFFFu, v, d);
        const int i2 = __shfl_xor_sync(0xFFFFFFFFu, i, d);
        better(v, i, v2, i2);
    }
}

// The patch-table position of a patched id at bit li of the bitmap: patches
// before its word (kept per even word), before it in its word.
__device__ __forceinline__ int patch_word_base(const uint32_t* bm, const uint32_t* wp, int w) {
    return static_cast<int>(wp[w >> 1] + ((w & 1) ? __popc(bm[w - 1]) : 0u));
}
__device__ __forceinline__ int patch_rank(const uint32_t* bm, const uint32_t* wp, int li) {
    return patch_word_base(bm, wp, li >> 5) + __popc(bm[li >> 5] & ((1u << (li & 31)) - 1u));
}

}  // namespace arc
