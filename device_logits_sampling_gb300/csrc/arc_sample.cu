// C ABI of the GB300 sampler (include/arc_sample.h): argument checks, launch
// geometry, per-device kernel attributes and one launch per call.
#include <algorithm>
#include <atomic>
#include <map>
#include <mutex>
#include <tuple>
#include <climits>
#include <cstdint>
#include <cstring>
#include <type_traits>

#include "arc_decode.h"
#include "arc_sample.h"
#include "argmax_kernel.cuh"
#include "kernel_set.cuh"
#include "launch_util.cuh"

namespace {

using namespace arc;

constexpr int kMaxDevices = 64;
constexpr int kDefaultHist = 1024;  // history capacity when max_hist_len is 0
constexpr int kAssumedSMs = 152;

struct Plan {
    bool cluster = false;   // one cluster_kernel launch (a cluster of s CTAs per row)
    int s = 1;              // slices per row
    int L = 0;              // logits per slice
    int hist_cap = 0;
    int scan_smem = 0;      // dynamic shared memory of the scan kernel
    int cmax_off = 0;       // finish kernel layout
    int cs_off = 0;
    int cid_off = 0;
    int cv2_off = 0;
    int cmv_off = -1;
    int cwide_off = -1;
    int clist_off = 0;
    int cand_off = 0;
    int sorted_off = 0;
    int fb_wsum_off = 0;
    int fb_patch_off = 0;
    int fb_rounds = 0;
    int fin_smem = 0;
    int fin_g = 1;          // finish CTAs per row (a cluster when > 1)
    int64_t slices = 0;
    int F = 0;
    size_t ws_bytes = 0;
};

int elem_bytes(int dtype) { return dtype == ARC_F32 ? 4 : 2; }
bool known_dtype(int dtype) { return dtype == ARC_F32 || dtype == ARC_BF16 || dtype == ARC_F16; }

// One call of F on the kernel set of (dtype, history): F receives a value of
// type KernelSet<DT, HIST> (its static members are the calls).
template <class F>
auto with_kernel_set(int dtype, bool hist, F f) {
    if (dtype == ARC_BF16) return hist ? f(KernelSet<ARC_BF16, true>{}) : f(KernelSet<ARC_BF16, false>{});
    if (dtype == ARC_F16) return hist ? f(KernelSet<ARC_F16, true>{}) : f(KernelSet<ARC_F16, false>{});
    return hist ? f(KernelSet<ARC_F32, true>{}) : f(KernelSet<ARC_F32, false>{});
}

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
    if (!known_dtype(dtype)) return ARC_E_DTYPE;
    if (B <= 0 || V <= 0 || V > INT_MAX || ld < V) return ARC_E_SHAPE;
    if (B > (int64_t{1} << 24)) return ARC_E_SHAPE;
    if (reinterpret_cast<uintptr_t>(logits) % static_cast<uintptr_t>(elem_bytes(dtype)) != 0) return ARC_E_ALIGN;
    return ARC_OK;
}

int check_options(const arc_sample_options* o) {
    if (o == nullptr) return ARC_OK;
    if (o->flags & ~(ARC_OPT_STEP_AUTOINC | ARC_OPT_FORCE_BISECTION)) return ARC_E_OPTION;
    if (o->ctas_per_row < 0 || o->ctas_per_row > kMaxRowCtas) return ARC_E_OPTION;
    if (o->max_hist_len < 0 || o->max_hist_len > (1 << 20)) return ARC_E_OPTION;
    if (o->top_n < 0 || o->top_n > ARC_MAX_TOP_N) return ARC_E_OPTION;
    if (o->top_n > 0 && o->top_logprobs == nullptr) return ARC_E_OPTION;
    return ARC_OK;
}

// Geometry: a row is cut into s slices of at most kVpt * kThreads 16-byte
// vectors (one scan CTA each), as few as the row allows: every slice adds 32
// chunk entries to the row's finish, and on the mixed rows at V = 129,280
// more, smaller slices were slower at every batch size measured (20 rows:
// 19.0 us with 61 slices against 11.3 us with 16).  A batch of at most 8 rows
// whose rows fit in clusters of at most 16 CTAs, all resident at once (two
// per SM), takes the one-launch cluster kernel when `allow_cluster` (at 16
// rows and more the two kernels were faster); an explicit ctas_per_row always
// takes the two kernels.
constexpr int kClusterMax = 16;
constexpr int kClusterMaxRows = 8;
constexpr int kFinishClusterMax = 8;
constexpr int64_t kSmemPerSM = 233472;  // shared memory of an SM (228 KB)

int make_plan(int64_t B, int64_t V, int dtype, bool has_hist, const arc_sample_options* o, int num_sms,
              Plan& p, bool allow_cluster = true) {
    const int es = elem_bytes(dtype);
    const int vec = 16 / es;
    const int64_t slice_max = int64_t{kVpt} * kThreads * vec;
    int64_t s;
    const bool automatic = o == nullptr || o->ctas_per_row == 0;
    bool cluster = false;
    if (automatic && allow_cluster && B <= kClusterMaxRows) {
        const int64_t s_min = (V + slice_max - 1) / slice_max;
        const int64_t s_cap = std::max<int64_t>(1, V / 1024);
        // one row: more, smaller slices shorten its scan; several rows: the
        // fewest slices (a smaller finish), measured faster at V = 20,000 and
        // 50,000 for 4 and 8 rows (8.2-9.1 against 9.3-10.4 us)
        const int64_t fs =
            B == 1 ? std::max<int64_t>(s_min, std::min<int64_t>({int64_t{kClusterMax}, s_cap, 2 * int64_t{num_sms}}))
                   : s_min;
        if (fs <= kClusterMax && B * fs <= 2 * int64_t{num_sms}) {
            cluster = true;
            s = fs;
        }
    }
    if (cluster) {
    } else if (!automatic) {
        s = o->ctas_per_row;
    } else {
        s = std::min<int64_t>((V + slice_max - 1) / slice_max, kMaxRowCtas);
    }
    if (s * slice_max < V || s > kMaxRowCtas) return ARC_E_UNSUPPORTED;
    const int64_t per = (V + s - 1) / s;
    const int64_t L = ((per + vec - 1) / vec) * vec;
    s = (V + L - 1) / L;  // no empty slice (fewer CTAs in the cluster when rounding frees one)
    const int cap = has_hist ? ((o != nullptr && o->max_hist_len > 0) ? o->max_hist_len : kDefaultHist) : 0;
    int64_t scan_smem = 0;
    if (has_hist) {
        const int64_t nwords = (int64_t{kVpt} * kThreads * vec + 31) / 32;
        scan_smem = nwords * 4 + (nwords + 1) / 2 * 4 + 2 * int64_t{cap} * 4;
    }
    auto r128 = [](int64_t x) { return ((x + 127) / 128) * 128; };
    const int64_t cmax_bytes = r128(s * kChunks * 4);
    const int64_t cs_bytes = 3 * cmax_bytes;  // masses, max ids, second largest logits
    const int64_t clist_bytes = r128((s * kChunks + kWarps) * 4);
    const int64_t cand_bytes = r128(int64_t{kCandCap} * 8);     // (key, id) as one 64-bit value
    const int64_t stage_bytes = r128(int64_t{kCandCap} * 16);   // in rank order: key, id, mass
    const int64_t nv_row = (V + vec - 1) / vec;
    const int64_t fb_rounds = (nv_row + kThreads - 1) / kThreads;
    const int64_t fb_wsum = r128(fb_rounds * kWarps * 8);
    int64_t fb_patch = 0;
    if (has_hist) {
        const int64_t nwords = (fb_rounds * kThreads * vec + 31) / 32;
        fb_patch = r128(nwords * 4 + (nwords + 1) / 2 * 4 + 2 * int64_t{cap} * 4);
    }
    // the chunk max vectors of a filtered row, when they fit in 16 KB (else
    // the finish reads them from the logits)
    const int64_t cmv_raw = s * kChunks * 16;
    // two finish CTAs per SM when their shared memory allows it (227 KB of the
    // SM's 228 KB usable, 1 KB reserved per CTA)
    const int64_t per_cta_extra = static_cast<int64_t>(sizeof(KernelShared)) + 1024;
    auto fits_two = [&](int64_t dyn) { return 2 * (dyn + per_cta_extra) <= kSmemPerSM; };
    const int64_t fin_base = cmax_bytes + cs_bytes + clist_bytes + cand_bytes + stage_bytes + fb_wsum + fb_patch;
    int64_t cmv_bytes = cmv_raw <= 16384 ? r128(cmv_raw) : 0;
    // the wide entries of large-k rows stay (they give those rows a floor);
    // the max vectors (which only save a re-read) not at the price of the
    // second CTA per SM
    if (fits_two(fin_base + cmv_bytes) && !fits_two(fin_base + 2 * cmv_bytes)) cmv_bytes = 0;
    // and the wide entries of top-k rows with a large k, under the same bound
    const int64_t cwide_bytes = cmv_raw <= 16384 ? r128(cmv_raw) : 0;
    const int64_t fin_smem = fin_base + cmv_bytes + cwide_bytes;
    int64_t limit = kSmemPerBlock - static_cast<int64_t>(sizeof(KernelShared)) - 1024;
    if (cluster) limit -= kSummaryBytes + static_cast<int64_t>(sizeof(ScanShared));
    if (fin_smem > limit || scan_smem > limit) {
        if (cluster) return make_plan(B, V, dtype, has_hist, o, num_sms, p, false);
        return ARC_E_UNSUPPORTED;
    }
    p.cluster = cluster;
    p.s = static_cast<int>(s);
    p.L = static_cast<int>(L);
    p.hist_cap = cap;
    p.scan_smem = static_cast<int>(scan_smem);
    p.cmax_off = 0;
    p.cs_off = static_cast<int>(cmax_bytes);
    p.cid_off = static_cast<int>(2 * cmax_bytes);
    p.cv2_off = static_cast<int>(3 * cmax_bytes);
    p.clist_off = static_cast<int>(cmax_bytes + cs_bytes);
    p.cand_off = static_cast<int>(cmax_bytes + cs_bytes + clist_bytes);
    p.sorted_off = static_cast<int>(cmax_bytes + cs_bytes + clist_bytes + cand_bytes);
    p.fb_wsum_off = static_cast<int>(cmax_bytes + cs_bytes + clist_bytes + cand_bytes + stage_bytes);
    p.fb_patch_off = static_cast<int>(cmax_bytes + cs_bytes + clist_bytes + cand_bytes + stage_bytes + fb_wsum);
    p.fb_rounds = static_cast<int>(fb_rounds);
    p.cmv_off = cmv_bytes ? static_cast<int>(fin_smem - cmv_bytes - cwide_bytes) : -1;
    p.cwide_off = cwide_bytes ? static_cast<int>(fin_smem - cwide_bytes) : -1;
    // every region holds 16-byte vectors or 8-byte words: starts must be 16-byte aligned
    for (const int off : {p.cs_off, p.cid_off, p.cv2_off, p.clist_off, p.cand_off, p.sorted_off,
                          p.fb_wsum_off, p.fb_patch_off, p.cmv_off, p.cwide_off})
        if (off >= 0 && off % 16 != 0) return ARC_E_UNSUPPORTED;
    p.fin_smem = static_cast<int>(fin_smem);
    // finish CTAs per row: while the batch leaves finish slots idle (one or
    // two CTAs per SM, by shared memory), rows of at least 2,048 vectors per
    // CTA get a cluster of up to 8, which splits the threshold bisection of a
    // row over the cluster
    p.fin_g = 1;
    if (!cluster) {
        const int64_t nv_row = (V + vec - 1) / vec;
        const int64_t per_sm = fits_two(fin_smem) ? 2 : 1;
        while (p.fin_g < kFinishClusterMax && B * 2 * p.fin_g <= per_sm * num_sms &&
               nv_row >= int64_t{2} * p.fin_g * 2048)
            p.fin_g *= 2;
    }
    p.slices = B * s;
    p.F = 62 - ceil_log2(V);
    p.ws_bytes = cluster ? 0 : static_cast<size_t>(B * s) * kSummaryBytes;
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

std::atomic<uint64_t> g_prep_argmax[3];

// Scratch of arc_sample_batch_static, for callers that cannot allocate device
// memory: one array per device context, created with the module.  Host code
// sees only a stand-in symbol; its device address is looked up in the current
// context at every call.
__device__ __align__(256) unsigned char g_static_workspace[ARC_STATIC_WORKSPACE_BYTES];

}  // namespace

extern "C" {

int arc_sample_abi_version(void) { return ARC_SAMPLE_ABI_VERSION; }

const char* arc_sample_strerror(int code) {
    switch (code) {
        case ARC_OK: return "ok";
        case ARC_E_NULL: return "a required pointer is NULL";
        case ARC_E_SHAPE: return "bad shape: need B > 0, 0 < V <= 2^31-1 and ld >= V";
        case ARC_E_DTYPE: return "dtype must be ARC_F32, ARC_BF16 or ARC_F16";
        case ARC_E_ALIGN: return "logits pointer is not aligned to its element size";
        case ARC_E_UNSUPPORTED: return "the vocabulary needs more CTAs per row than allowed";
        case ARC_E_OPTION: return "bad field in arc_sample_options";
        case ARC_E_CUDA: return "CUDA error while configuring or launching the kernel";
        case ARC_E_WORKSPACE: return "workspace is NULL or smaller than arc_sample_workspace_bytes()";
        case ARC_E_RING_OVERRUN: return "a commit ring slot was overwritten before it was drained";
        default: return "unknown error code";
    }
}

int arc_sample_plan(int64_t B, int64_t V, int32_t dtype, int32_t has_history, const arc_sample_options* opts,
                    arc_sample_geometry* geom) {
    if (geom == nullptr) return ARC_E_NULL;
    if (!known_dtype(dtype)) return ARC_E_DTYPE;
    if (B <= 0 || V <= 0 || V > INT_MAX || B > (int64_t{1} << 24)) return ARC_E_SHAPE;
    int rc = check_options(opts);
    if (rc != ARC_OK) return rc;
    Plan p;
    rc = make_plan(B, V, dtype, has_history != 0, opts, kAssumedSMs, p);
    if (rc != ARC_OK) return rc;
    geom->ctas_per_row = p.s;
    geom->threads = kThreads;
    geom->slice_elems = p.L;
    geom->smem_bytes = p.fin_smem;
    geom->grid_ctas = p.slices;
    geom->frac_bits = p.F;
    geom->launches = p.cluster ? 1 : 2;
    geom->workspace_bytes = static_cast<int64_t>(p.ws_bytes);
    geom->finish_ctas = p.cluster ? 1 : p.fin_g;
    geom->reserved = 0;
    return ARC_OK;
}

size_t arc_sample_workspace_bytes(int64_t B, int64_t V, int32_t dtype, int32_t has_history,
                                  const arc_sample_options* opts) {
    if (!known_dtype(dtype)) return 0;
    if (B <= 0 || V <= 0 || V > INT_MAX || B > (int64_t{1} << 24)) return 0;
    if (check_options(opts) != ARC_OK) return 0;
    Plan p;
    if (make_plan(B, V, dtype, has_history != 0, opts, kAssumedSMs, p) != ARC_OK) return 0;
    // the plan depends on the SM count only through ctas_per_row; size for the
    // largest automatic choice so one workspace fits every device
    Plan q;
    arc_sample_options big{};
    if (opts != nullptr) big = *opts;
    if (big.ctas_per_row == 0) {
        big.ctas_per_row = kMaxRowCtas;
        if (make_plan(B, V, dtype, has_history != 0, &big, kAssumedSMs, q) == ARC_OK)
            return std::max(p.ws_bytes, q.ws_bytes);
    }
    return p.ws_bytes;
}

}  // extern "C"

namespace {

// arc_sample_batch, with each row's decode-loop commit folded into its finish
// when `commit` is given (arc_sample_batch_commit).
int sample_impl(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype, arc_row_params* params,
                const int32_t* hist_offsets, const int32_t* hist_ids, int32_t* out, uint32_t* err_word,
                void* workspace, size_t workspace_bytes, const arc_sample_options* opts,
                const arc_commit_target* commit, void* stream) {
    int rc = check_common(logits, B, V, ld, dtype, out);
    if (rc != ARC_OK) return rc;
    if (params == nullptr) return ARC_E_NULL;
    if (hist_offsets != nullptr && hist_ids == nullptr) return ARC_E_NULL;
    if (reinterpret_cast<uintptr_t>(params) % 8 != 0) return ARC_E_ALIGN;
    rc = check_options(opts);
    if (rc != ARC_OK) return rc;
    if (workspace == nullptr) return ARC_E_WORKSPACE;
    if (reinterpret_cast<uintptr_t>(workspace) % 16 != 0) return ARC_E_ALIGN;

    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return ARC_E_CUDA;
    const bool has_hist = hist_offsets != nullptr;
    Plan p;
    rc = make_plan(B, V, dtype, has_hist, opts, num_sms_of(dev), p);
    if (rc != ARC_OK) return rc;
    if (p.cluster) {
        // the one-launch cluster kernel, when the device can schedule its clusters
        const int dyn = std::max(p.scan_smem, p.fin_smem);
        const bool fits = with_kernel_set(dtype, has_hist, [&](auto k) { return k.cluster_ok(p.s, dyn, dev); });
        if (!fits) {
            rc = make_plan(B, V, dtype, has_hist, opts, num_sms_of(dev), p, false);
            if (rc != ARC_OK) return rc;
        }
    }
    if (workspace_bytes < p.ws_bytes) return ARC_E_WORKSPACE;
    if (!p.cluster && p.fin_g > 1) {
        // a split finish only when the device can schedule its clusters
        const bool ok =
            with_kernel_set(dtype, has_hist, [&](auto k) { return k.finish_cluster_ok(p.fin_g, p.fin_smem, dev); });
        if (!ok) p.fin_g = 1;
    }

    const int es = elem_bytes(dtype);
    const int aligned = (reinterpret_cast<uintptr_t>(logits) % 16 == 0) && ((ld * es) % 16 == 0);
    ScanArgs sa;
    sa.logits = logits;
    sa.ld = ld;
    sa.B = static_cast<int>(B);
    sa.V = static_cast<int>(V);
    sa.s = p.s;
    sa.L = p.L;
    sa.params = params;
    sa.hist_off = hist_offsets;
    sa.hist_ids = hist_ids;
    sa.summaries = static_cast<unsigned char*>(workspace);
    sa.hist_cap = p.hist_cap;
    sa.aligned = aligned;
    sa.top_n = opts ? opts->top_n : 0;
    FinishArgs fa;
    fa.logits = logits;
    fa.ld = ld;
    fa.B = static_cast<int>(B);
    fa.V = static_cast<int>(V);
    fa.s = p.s;
    fa.L = p.L;
    fa.params = params;
    fa.hist_off = hist_offsets;
    fa.hist_ids = hist_ids;
    fa.out = out;
    fa.err_word = err_word;
    fa.debug = opts ? opts->debug : nullptr;
    fa.top_n = opts ? opts->top_n : 0;
    fa.top_logprobs = (opts && opts->top_n > 0) ? opts->top_logprobs : nullptr;
    fa.summaries = static_cast<const unsigned char*>(workspace);
    fa.hist_cap = p.hist_cap;
    fa.F = p.F;
    fa.flags = opts ? opts->flags : 0u;
    fa.aligned = aligned;
    fa.cmax_off = p.cmax_off;
    fa.cs_off = p.cs_off;
    fa.cid_off = p.cid_off;
    fa.cv2_off = p.cv2_off;
    fa.cmv_off = p.cmv_off;
    fa.cwide_off = p.cwide_off;
    fa.clist_off = p.clist_off;
    fa.cand_off = p.cand_off;
    fa.sorted_off = p.sorted_off;
    fa.fb_wsum_off = p.fb_wsum_off;
    fa.fb_patch_off = p.fb_patch_off;
    fa.fb_rounds = p.fb_rounds;
    fa.commit = commit ? *commit : arc_commit_target{};
    fa.fin_g = p.fin_g;

    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e;
    if (p.cluster) {
        const FusedArgs fu{sa, fa};
        const int dyn = std::max(p.scan_smem, p.fin_smem);
        e = with_kernel_set(dtype, has_hist, [&](auto k) { return k.launch_fused(fu, B, p.s, dyn, st); });
    } else {
        e = with_kernel_set(dtype, has_hist,
                            [&](auto k) { return k.launch_two(sa, fa, p.s, B, p.scan_smem, p.fin_smem, dev, st); });
    }
    return e == cudaSuccess ? ARC_OK : ARC_E_CUDA;
}

}  // namespace

extern "C" {

int arc_sample_batch(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype, arc_row_params* params,
                     const int32_t* hist_offsets, const int32_t* hist_ids, int32_t* out, uint32_t* err_word,
                     void* workspace, size_t workspace_bytes, const arc_sample_options* opts, void* stream) {
    return sample_impl(logits, B, V, ld, dtype, params, hist_offsets, hist_ids, out, err_word, workspace,
                       workspace_bytes, opts, nullptr, stream);
}

int arc_sample_batch_commit(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype,
                            arc_row_params* params, const int32_t* hist_offsets, const int32_t* hist_ids,
                            int32_t* out, uint32_t* err_word, void* workspace, size_t workspace_bytes,
                            const arc_sample_options* opts, const arc_commit_target* commit, void* stream) {
    if (commit == nullptr || commit->next_ids == nullptr || commit->positions == nullptr ||
        commit->ring == nullptr || commit->head == nullptr)
        return ARC_E_NULL;
    if (reinterpret_cast<uintptr_t>(commit->head) % 8 != 0 || reinterpret_cast<uintptr_t>(commit->ring) % 8 != 0)
        return ARC_E_ALIGN;
    if (commit->max_position <= 0 || commit->capacity == 0 || commit->capacity > ARC_RING_MAX_CAPACITY ||
        B > static_cast<int64_t>(commit->capacity))
        return ARC_E_SHAPE;
    return sample_impl(logits, B, V, ld, dtype, params, hist_offsets, hist_ids, out, err_word, workspace,
                       workspace_bytes, opts, commit, stream);
}

int arc_sample_batch_static(const void* logits, int64_t B, int64_t V, int64_t ld, int32_t dtype,
                            arc_row_params* params, const int32_t* hist_offsets, const int32_t* hist_ids,
                            int32_t* out, uint32_t* err_word, const arc_sample_options* opts, void* stream) {
    // the host checks of arc_sample_batch, before any CUDA call
    int rc = check_common(logits, B, V, ld, dtype, out);
    if (rc != ARC_OK) return rc;
    if (params == nullptr) return ARC_E_NULL;
    if (hist_offsets != nullptr && hist_ids == nullptr) return ARC_E_NULL;
    if (reinterpret_cast<uintptr_t>(params) % 8 != 0) return ARC_E_ALIGN;
    rc = check_options(opts);
    if (rc != ARC_OK) return rc;

    // the array's address in the current context (never cached: a device
    // reset or another context loads the module at another address)
    void* addr = nullptr;
    if (cudaGetSymbolAddress(&addr, g_static_workspace) != cudaSuccess || addr == nullptr) return ARC_E_CUDA;
    // a plan that needs more than the array is refused there (ARC_E_WORKSPACE)
    return arc_sample_batch(logits, B, V, ld, dtype, params, hist_offsets, hist_ids, out, err_word, addr,
                            ARC_STATIC_WORKSPACE_BYTES, opts, stream);
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
        e = prepare(argmax_kernel<ARC_BF16>, dev, g_prep_argmax[1], 0);
        if (e == cudaSuccess) e = launch_cluster(argmax_kernel<ARC_BF16>, B * s, s, 0, st, a);
    } else if (dtype == ARC_F16) {
        e = prepare(argmax_kernel<ARC_F16>, dev, g_prep_argmax[2], 0);
        if (e == cudaSuccess) e = launch_cluster(argmax_kernel<ARC_F16>, B * s, s, 0, st, a);
    } else {
        e = prepare(argmax_kernel<ARC_F32>, dev, g_prep_argmax[0], 0);
        if (e == cudaSuccess) e = launch_cluster(argmax_kernel<ARC_F32>, B * s, s, 0, st, a);
    }
    return e == cudaSuccess ? ARC_OK : ARC_E_CUDA;
}

}  // extern "C"
