// C ABI of the GB300 sampler (include/arc_sample.h): argument checks, launch
// geometry, per-device kernel attributes and one launch per call.
#include <atomic>
#include <climits>
#include <cstdint>
#include <cstring>

#include "arc_sample.h"
#include "argmax_kernel.cuh"
#include "sample_kernel.cuh"

namespace {

using namespace arc;

constexpr int kMaxDevices = 64;
constexpr int kSliceBytes = 32 * 1024;        // target bytes of a row per CTA
constexpr int kSmemPerBlock = 232448;         // 227 KB opt-in limit of sm_100-class GPUs
constexpr int kDefaultHist = 1024;
constexpr int kAssumedSMs = 152;

struct Plan {
    int s = 1;
    int L = 0;
    int vmax_off = 0;
    int wsum_off = 0;
    int hist_off_b = 0;
    int rounds_max = 0;
    int hist_cap = 0;
    int smem = 0;
    int64_t grid = 0;
    int F = 0;
};

int elem_bytes(int dtype) { return dtype == ARC_BF16 ? 2 : 4; }

int pow2_at_least(int64_t x) {
    int p = 1;
    while (p < x && p < (1 << 30)) p <<= 1;
    return p;
}

int ceil_log2(int64_t v) {
    int b = 0;
    while ((int64_t{1} << b) < v) ++b;
    return b;
}

int check_common(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype, const int32_t* out) {
    if (logits == nullptr || out == nullptr) return ARC_E_NULL;
    if (dtype != ARC_F32 && dtype != ARC_BF16) return ARC_E_DTYPE;
    if (B <= 0 || V <= 0 || V > INT_MAX || ld < V) return ARC_E_SHAPE;
    if (B > (int64_t{1} << 26)) return ARC_E_SHAPE;
    if (reinterpret_cast<uintptr_t>(logits) % static_cast<uintptr_t>(elem_bytes(dtype)) != 0) return ARC_E_ALIGN;
    return ARC_OK;
}

int check_options(const arc_sample_options* o) {
    if (o == nullptr) return ARC_OK;
    if (o->flags & ~ARC_OPT_STEP_AUTOINC) return ARC_E_OPTION;
    const int c = o->cluster_ctas;
    if (!(c == 0 || c == 1 || c == 2 || c == 4 || c == 8 || c == 16)) return ARC_E_OPTION;
    if (o->max_hist_len < 0 || o->max_hist_len > (1 << 20)) return ARC_E_OPTION;
    if (o->reserved != 0) return ARC_E_OPTION;
    return ARC_OK;
}

// Geometry of the fused kernel.  The row is split over s CTAs (a cluster);
// each CTA keeps its slice, plus per-chunk masses and history patches, in
// shared memory.
int make_plan(int64_t B, int64_t V, int dtype, bool has_hist, const arc_sample_options* o, int num_sms,
              Plan& p) {
    const int es = elem_bytes(dtype);
    const int vec = 16 / es;
    int s;
    if (o != nullptr && o->cluster_ctas != 0) {
        s = o->cluster_ctas;
    } else {
        const int s_min = min(kMaxCluster, pow2_at_least((V * es + kSliceBytes - 1) / kSliceBytes));
        const int s_want = min(kMaxCluster, pow2_at_least((2 * int64_t{num_sms} + B - 1) / B));
        int s_cap = 1;
        while (s_cap < kMaxCluster && V / (2 * s_cap) >= 2048) s_cap <<= 1;
        s = max(s_min, min(s_want, s_cap));
    }
    const int64_t per = (V + s - 1) / s;
    const int64_t L = ((per + vec - 1) / vec) * vec;
    const int64_t nv_max = L / vec;
    const int64_t rounds_max = (nv_max + kThreads - 1) / kThreads;
    // dynamic shared memory: slice | per-vector max | per-(round, warp) masses | history tables
    const int64_t data_bytes = ((nv_max * 16 + 127) / 128) * 128;
    const int64_t vmax_off = data_bytes;
    const int64_t wsum_off = vmax_off + ((nv_max * 4 + 15) / 16) * 16;
    const int64_t hist_off_b = wsum_off + rounds_max * kWarps * 8;
    int64_t smem = hist_off_b;
    int cap = 0;
    if (has_hist) {
        cap = (o != nullptr && o->max_hist_len > 0) ? o->max_hist_len : kDefaultHist;
        const int64_t nwords_max = (rounds_max * kThreads * vec + 31) / 32;
        smem += 2 * nwords_max * 4 + 2 * int64_t{cap} * 4;
    }
    const int64_t limit = kSmemPerBlock - static_cast<int64_t>(sizeof(SampleShared)) - 1024;
    if (smem > limit) return ARC_E_UNSUPPORTED;
    p.s = s;
    p.L = static_cast<int>(L);
    p.vmax_off = static_cast<int>(vmax_off);
    p.wsum_off = static_cast<int>(wsum_off);
    p.hist_off_b = static_cast<int>(hist_off_b);
    p.rounds_max = static_cast<int>(rounds_max);
    p.hist_cap = cap;
    p.smem = static_cast<int>(smem);
    p.grid = B * s;
    p.F = 62 - ceil_log2(V);
    return ARC_OK;
}

int num_sms_of(int dev) {
    static std::atomic<int> cache[kMaxDevices];
    if (dev < 0 || dev >= kMaxDevices) return kAssumedSMs;
    int v = cache[dev].load(std::memory_order_relaxed);
    if (v > 0) return v;
    if (cudaDeviceGetAttribute(&v, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || v <= 0)
        v = kAssumedSMs;
    cache[dev].store(v, std::memory_order_relaxed);
    return v;
}

// Function attributes are set once per (device, kernel): the first call on a
// device must come before any stream capture that contains a call.
template <class K>
cudaError_t prepare(K kernel, int dev, std::atomic<uint64_t>& done) {
    const uint64_t bit = uint64_t{1} << (dev & 63);
    if (done.load(std::memory_order_acquire) & bit) return cudaSuccess;
    cudaError_t e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSmemPerBlock - static_cast<int>(sizeof(SampleShared)) - 1024);
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
    if (e != cudaSuccess) return e;
    done.fetch_or(bit, std::memory_order_acq_rel);
    return cudaSuccess;
}

template <class K, class A>
cudaError_t launch_cluster(K kernel, int64_t grid, int s, int smem, cudaStream_t st, const A& args) {
    cudaLaunchConfig_t cfg;
    std::memset(&cfg, 0, sizeof(cfg));
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(kThreads, 1, 1);
    cfg.dynamicSmemBytes = static_cast<size_t>(smem);
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = static_cast<unsigned>(s);
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, args);
}

std::atomic<uint64_t> g_prep_sample[2][2];
std::atomic<uint64_t> g_prep_argmax[2];

}  // namespace

extern "C" {

int arc_sample_abi_version(void) { return ARC_SAMPLE_ABI_VERSION; }

const char* arc_sample_strerror(int code) {
    switch (code) {
        case ARC_OK: return "ok";
        case ARC_E_NULL: return "a required pointer is NULL";
        case ARC_E_SHAPE: return "bad shape: need B > 0, 0 < V <= 2^31-1 and ld >= V";
        case ARC_E_DTYPE: return "dtype must be ARC_F32 or ARC_BF16";
        case ARC_E_ALIGN: return "logits pointer is not aligned to its element size";
        case ARC_E_UNSUPPORTED: return "a row slice does not fit in shared memory";
        case ARC_E_OPTION: return "bad field in arc_sample_options";
        case ARC_E_CUDA: return "CUDA error while configuring or launching the kernel";
        default: return "unknown error code";
    }
}

int arc_sample_plan(int64_t B, int64_t V, int32_t dtype, int32_t has_history, const arc_sample_options* opts,
                    arc_sample_geometry* geom) {
    if (geom == nullptr) return ARC_E_NULL;
    if (dtype != ARC_F32 && dtype != ARC_BF16) return ARC_E_DTYPE;
    if (B <= 0 || V <= 0 || V > INT_MAX || B > (int64_t{1} << 26)) return ARC_E_SHAPE;
    int rc = check_options(opts);
    if (rc != ARC_OK) return rc;
    Plan p;
    rc = make_plan(B, V, dtype, has_history != 0, opts, kAssumedSMs, p);
    if (rc != ARC_OK) return rc;
    geom->cluster_ctas = p.s;
    geom->threads = kThreads;
    geom->slice_elems = p.L;
    geom->smem_bytes = p.smem;
    geom->grid_ctas = p.grid;
    geom->frac_bits = p.F;
    geom->reserved = 0;
    return ARC_OK;
}

int arc_sample_batch(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype, arc_row_params* params,
                     const int32_t* hist_offsets, const int32_t* hist_ids, int32_t* out, uint32_t* err_word,
                     const arc_sample_options* opts, void* stream) {
    int rc = check_common(logits, B, V, ld, dtype, out);
    if (rc != ARC_OK) return rc;
    if (params == nullptr) return ARC_E_NULL;
    if (hist_offsets != nullptr && hist_ids == nullptr) return ARC_E_NULL;
    if (reinterpret_cast<uintptr_t>(params) % 8 != 0) return ARC_E_ALIGN;
    rc = check_options(opts);
    if (rc != ARC_OK) return rc;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ARC_E_CUDA;
    const bool has_hist = hist_offsets != nullptr;
    Plan p;
    rc = make_plan(B, V, dtype, has_hist, opts, num_sms_of(dev), p);
    if (rc != ARC_OK) return rc;

    SampleArgs a;
    a.logits = logits;
    a.ld = ld;
    a.B = static_cast<int>(B);
    a.V = static_cast<int>(V);
    a.params = params;
    a.hist_off = hist_offsets;
    a.hist_ids = hist_ids;
    a.out = out;
    a.err_word = err_word;
    a.debug = opts ? opts->debug : nullptr;
    a.L = p.L;
    a.vmax_off = p.vmax_off;
    a.wsum_off = p.wsum_off;
    a.hist_off_b = p.hist_off_b;
    a.rounds_max = p.rounds_max;
    a.hist_cap = p.hist_cap;
    a.F = p.F;
    a.flags = opts ? opts->flags : 0u;
    const int es = elem_bytes(dtype);
    a.aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((ld * es) % 16 == 0);

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == ARC_BF16) {
        if (has_hist) {
            e = prepare(sample_kernel<ARC_BF16, true>, dev, g_prep_sample[1][1]);
            if (e == cudaSuccess) e = launch_cluster(sample_kernel<ARC_BF16, true>, p.grid, p.s, p.smem, st, a);
        } else {
            e = prepare(sample_kernel<ARC_BF16, false>, dev, g_prep_sample[1][0]);
            if (e == cudaSuccess) e = launch_cluster(sample_kernel<ARC_BF16, false>, p.grid, p.s, p.smem, st, a);
        }
    } else {
        if (has_hist) {
            e = prepare(sample_kernel<ARC_F32, true>, dev, g_prep_sample[0][1]);
            if (e == cudaSuccess) e = launch_cluster(sample_kernel<ARC_F32, true>, p.grid, p.s, p.smem, st, a);
        } else {
            e = prepare(sample_kernel<ARC_F32, false>, dev, g_prep_sample[0][0]);
            if (e == cudaSuccess) e = launch_cluster(sample_kernel<ARC_F32, false>, p.grid, p.s, p.smem, st, a);
        }
    }
    return e == cudaSuccess ? ARC_OK : ARC_E_CUDA;
}

int arc_sample_greedy(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype, int32_t* out,
                      uint32_t* err_word, void* stream) {
    int rc = check_common(logits, B, V, ld, dtype, out);
    if (rc != ARC_OK) return rc;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ARC_E_CUDA;
    const int es = elem_bytes(dtype);
    const int vec = 16 / es;
    const int sms = num_sms_of(dev);
    // enough CTAs for four per SM, at most 16 per row, at least 2048 logits each
    int s = max(pow2_at_least((V * es + 65535) / 65536), pow2_at_least((4 * int64_t{sms} + B - 1) / B));
    int s_cap = 1;
    while (s_cap < kMaxCluster && V / (2 * s_cap) >= 2048) s_cap <<= 1;
    s = max(1, min(min(s, s_cap), kMaxCluster));
    const int64_t per = (V + s - 1) / s;
    ArgmaxArgs a;
    a.logits = logits;
    a.ld = ld;
    a.V = static_cast<int>(V);
    a.L = static_cast<int>(((per + vec - 1) / vec) * vec);
    a.aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((ld * es) % 16 == 0);
    a.out = out;
    a.err_word = err_word;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (dtype == ARC_BF16) {
        e = prepare(argmax_kernel<ARC_BF16>, dev, g_prep_argmax[1]);
        if (e == cudaSuccess) e = launch_cluster(argmax_kernel<ARC_BF16>, B * s, s, 0, st, a);
    } else {
        e = prepare(argmax_kernel<ARC_F32>, dev, g_prep_argmax[0]);
        if (e == cudaSuccess) e = launch_cluster(argmax_kernel<ARC_F32>, B * s, s, 0, st, a);
    }
    return e == cudaSuccess ? ARC_OK : ARC_E_CUDA;
}

}  // extern "C"
