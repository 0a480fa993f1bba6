// On-device sampling in two kernels, one HBM pass over the logits.
//
// scan_kernel: a row is split into s slices of at most kVpt * kThreads
// 16-byte vectors; one CTA per slice issues all its 16-byte loads first (they
// depend on nothing), applies the history penalties in registers, and writes
// a small summary to the workspace: the slice max and its first id, and per
// 32-vector chunk (256 bf16 / 128 fp32 logits) the chunk max and, for rows
// that need masses, the fp32 sum of 2^((z - chunk max) log2(e) / T).  No CTA
// waits for another and registers stay few, so many CTAs per SM keep HBM busy.
//
// finish_kernel: one CTA per row combines the slice summaries.
//  - greedy rows take the row max;
//  - default rows draw from the chunk masses (exact integer fixed point,
//    rescaled to the row max) with one block scan, and re-read only the chunk
//    that holds the draw;
//  - filtered rows first bound the cutoff from below with the chunk maxima
//    (the k-th largest chunk max for top-k, the min-p threshold, or a mass
//    bound for top-p), gather the few ids at or above that floor from the
//    chunks that can hold them, in id order, into shared memory, and select
//    exactly there by ranking.  When the floor admits too many ids, the
//    general threshold bisection of row_select.cuh runs over the row instead.
#pragma once

#include <climits>

#include "row_select.cuh"

namespace arc {

constexpr int kVpt = 4;                  // 16-byte vectors per thread in a scan CTA
constexpr int kChunks = kVpt * kWarps;   // chunks per slice summary (32-vector chunks)
constexpr int kHdrBytes = 32;
constexpr int kSummaryBytes = kHdrBytes + kChunks * 8;
constexpr int kMaxRowCtas = 128;         // slices per row at most
constexpr int kCandCap = 1024;           // ids the direct selection holds
constexpr int kCandChunks = 256;         // chunks it reads at most
constexpr int kCollectU = 8;             // chunks per warp in flight while gathering
constexpr int kFloorBins = 1024;         // bins of the floor search (10 key bits per pass)

struct ScanArgs {
    const void* logits;
    int64_t ld;
    int B;
    int V;
    int s;  // slices per row
    int L;  // logits per slice (multiple of the vector width)
    const arc_row_params* params;
    const int32_t* hist_off;
    const int32_t* hist_ids;
    unsigned char* summaries;  // [B * s] x kSummaryBytes
    int hist_cap;
    int aligned;    // rows start on 16-byte boundaries: 16-byte loads
};

struct FinishArgs {
    const void* logits;
    int64_t ld;
    int B;
    int V;
    int s;
    int L;
    arc_row_params* params;
    const int32_t* hist_off;
    const int32_t* hist_ids;
    int32_t* out;
    uint32_t* err_word;
    arc_row_debug* debug;
    const unsigned char* summaries;
    int hist_cap;
    int F;
    uint32_t flags;
    int aligned;
    int cmax_off;      // dynamic shared memory: chunk maxima of the row,
    int cs_off;        //   chunk masses,
    int clist_off;     //   candidate chunk list,
    int cand_off;      //   candidates (key, id, mass),
    int fb_wsum_off;   //   per-(round, warp) masses,
    int fb_patch_off;  //   row patch tables
    int fb_rounds;     // rounds of a whole row
};

struct SliceHeader {
    float m;         // slice max (NaN-free), -inf when none
    int am;          // its first id, -1 when none
    uint32_t flags;  // ARC_ERR_NAN | ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP
    int nchunk;      // chunk entries written
    int pad[4];
};

struct FinishScratch {
    uint64_t redu[kWarps];
    uint32_t red32[kWarps];
    int bi[8];
    uint64_t bu[8];
    float bf[8];
    uint32_t ccount;  // candidates gathered
    double bd[2];
};

struct __align__(16) KernelShared {
    union {
        SampleShared fb;              // general selection path
        uint32_t fhist[kFloorBins + kFloorBins / 32];  // floor search (padded)
    };
    FinishScratch st;
};

__device__ __forceinline__ const unsigned char* summary_at(const unsigned char* base, int s, int row, int c) {
    return base + (static_cast<size_t>(row) * s + c) * kSummaryBytes;
}
__device__ __forceinline__ const float2* chunk_table(const unsigned char* sm) {
    return reinterpret_cast<const float2*>(sm + kHdrBytes);
}

// weight of z relative to a reference max mr (chunk or row): ex2((z - mr) c);
// a +inf reference gives [z == +inf]
__device__ __forceinline__ float wrel(float z, float mr, float c) {
    if (mr == INFINITY) return z == INFINITY ? 1.0f : 0.0f;
    return ex2(__fmul_rn(__fsub_rn(z, mr), c));
}

__device__ __forceinline__ uint32_t param_errors(const arc_row_params& P) {
    bool ok = isfinite(P.temperature) && P.temperature >= 0.0f;
    ok &= (P.top_p > 0.0f) && (P.top_p <= 1.0f);
    ok &= (P.min_p >= 0.0f) && (P.min_p <= 1.0f);
    ok &= isfinite(P.repetition_penalty) && P.repetition_penalty > 0.0f;
    ok &= isfinite(P.frequency_penalty) && isfinite(P.presence_penalty);
    ok &= P.flags == 0u;
    return ok ? 0u : ARC_ERR_PARAM;
}

// What a row needs, from its parameters.
struct RowMode {
    bool greedy, topk_on, topp_on, minp_on, filtered, need_mass;
    __device__ __forceinline__ RowMode(const arc_row_params& P, int V) {
        const int k = P.top_k;
        topk_on = k >= 1 && k < V;
        topp_on = P.top_p < 1.0f;
        minp_on = P.min_p > 0.0f;
        greedy = (P.temperature == 0.0f || k == 1);
        filtered = !greedy && (topk_on || topp_on || minp_on);
        // chunk masses: default rows draw from them, top-p over every id takes its total
        need_mass = !greedy && !topk_on && (topp_on || !minp_on);
    }
};

// ------------------------------------------------------------------ history
// Penalties for the ids of [a0, a0 + nvec*VEC) that occur in the row's
// history: a bitmap of those ids, per-word prefix popcounts (rank of an id),
// and per-rank counts and penalised logits.  Returns the number of distinct
// ids; sets ARC_ERR_HIST_ID in *bad for ids outside [0, V).
template <int DT>
__device__ int build_patches(const char* rowp, int V, int a0, int n, int nvec, const arc_row_params& P,
                             const int32_t* ids, int hn, uint32_t* bm, uint32_t* wp, uint32_t* cnt, float* pat,
                             uint32_t* red32, uint32_t* bad) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int a1 = a0 + n;
    const int nwords = (nvec * VEC + 31) / 32;
    for (int w = tid; w < nwords; w += kThreads) bm[w] = 0;
    __syncthreads();
    for (int e = tid; e < hn; e += kThreads) {
        const int id = ids[e];
        if (id < 0 || id >= V)
            atomicOr(bad, ARC_ERR_HIST_ID);
        else if (id >= a0 && id < a1)
            atomicOr(&bm[(id - a0) >> 5], 1u << ((id - a0) & 31));
    }
    __syncthreads();
    const int per = (nwords + kThreads - 1) / kThreads;
    const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
    uint32_t mine = 0;
    for (int w = w0; w < w1; ++w) mine += __popc(bm[w]);
    uint32_t inc = mine;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
        const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
        if (lane >= d) inc += o;
    }
    if (lane == 31) red32[warp] = inc;
    __syncthreads();
    uint32_t wbase = 0, distinct = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) wbase += red32[w];
        distinct += red32[w];
    }
    uint32_t run = wbase + inc - mine;
    for (int w = w0; w < w1; ++w) {
        wp[w] = run;
        run += __popc(bm[w]);
    }
    for (int q = tid; q < static_cast<int>(distinct); q += kThreads) cnt[q] = 0;
    __syncthreads();
    auto rank_of = [&](int li) {
        return static_cast<int>(wp[li >> 5] + __popc(bm[li >> 5] & ((1u << (li & 31)) - 1u)));
    };
    for (int e = tid; e < hn; e += kThreads) {
        const int id = ids[e];
        if (id >= a0 && id < a1) atomicAdd(&cnt[rank_of(id - a0)], 1u);
    }
    __syncthreads();
    const float rep = P.repetition_penalty, fr = P.frequency_penalty, pr = P.presence_penalty;
    for (int e = tid; e < hn; e += kThreads) {
        const int id = ids[e];
        if (id >= a0 && id < a1) {
            const int q = rank_of(id - a0);
            float z = E::load_scalar(rowp, id);
            z = (z > 0.0f) ? __fdiv_rn(z, rep) : __fmul_rn(z, rep);
            z = __fsub_rn(z, __fmul_rn(static_cast<float>(cnt[q]), fr));
            z = __fsub_rn(z, pr);
            pat[q] = z;  // duplicates of an id store the same value
        }
    }
    __syncthreads();
    return static_cast<int>(distinct);
}

template <int VEC>
__device__ __forceinline__ void apply_patches(const uint32_t* bm, const uint32_t* wp, const float* pat, int v,
                                              float (&z)[VEC]) {
    const int l0 = v * VEC;
    const uint32_t word = bm[l0 >> 5];
    const uint32_t bits = (word >> (l0 & 31)) & ((1u << VEC) - 1u);
    if (bits) {
        const int base = static_cast<int>(wp[l0 >> 5]);
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const int li = l0 + e;
            if ((bits >> e) & 1u) z[e] = pat[base + __popc(word & ((1u << (li & 31)) - 1u))];
        }
    }
}

// ------------------------------------------------------------------ small block helpers
__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = fmaxf(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    return v;
}
__device__ __forceinline__ float warp_sum_f(float v) {
#pragma unroll
    for (int d = 16; d > 0; d >>= 1) v = __fadd_rn(v, __shfl_xor_sync(0xFFFFFFFFu, v, d));
    return v;
}

// Block-wide sum of a u64 (all threads get it); uses red[kWarps].
__device__ __forceinline__ uint64_t block_sum_u64(uint64_t v, uint64_t* red) {
    v = warp_sum_u64(v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint64_t t = 0;
    for (int w = 0; w < kWarps; ++w) t += red[w];
    return t;
}

// Block-wide inclusive scan of a u64 in thread order; returns the inclusive
// value and sets total.  Uses red[kWarps].
__device__ __forceinline__ uint64_t block_scan_u64(uint64_t v, uint64_t* red, uint64_t& total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t inc = warp_inclusive_u64(v);
    __syncthreads();
    if (lane == 31) red[warp] = inc;
    __syncthreads();
    uint64_t base = 0;
    total = 0;
    for (int w = 0; w < kWarps; ++w) {
        if (w < warp) base += red[w];
        total += red[w];
    }
    return base + inc;
}

// ------------------------------------------------------------------ scan
// What the scan reads of a row besides its logits.
struct ScanRow {
    arc_row_params P;
    int hbeg, hn;
};

template <bool HIST>
__device__ __forceinline__ ScanRow scan_row_of(const ScanArgs& a, int row) {
    ScanRow r;
    // the finish kernel of an earlier call may have rewritten `step`, never
    // while this kernel runs: plain loads
    r.P = a.params[row];
    r.hbeg = 0;
    r.hn = 0;
    if (HIST && a.hist_off != nullptr) {
        r.hbeg = a.hist_off[row];
        r.hn = a.hist_off[row + 1] - r.hbeg;
    }
    return r;
}

struct ScanShared {
    float redf[kWarps];
    int redi[kWarps];
    uint32_t rednan[kWarps];
    uint32_t red32[kWarps];
    uint32_t sflags;  // history id errors (written only after a barrier past its init)
};

// sum_e 2^((z_e - ref) c) for a finite ref and NaN-free z, two elements per
// packed f32x2 add / multiply (same rounding as the scalar operations)
template <int VEC>
__device__ __forceinline__ float lane_mass_packed(const float (&z)[VEC], float ref, float c) {
    const float2 nr = make_float2(-ref, -ref), c2 = make_float2(c, c);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int e = 0; e < VEC; e += 2) {
        const float2 x = __fmul2_rn(__fadd2_rn(make_float2(z[e], z[e + 1]), nr), c2);
        acc = __fadd2_rn(acc, make_float2(ex2(x.x), ex2(x.y)));
    }
    return __fadd_rn(acc.x, acc.y);
}

// The same with NaN ids weighing nothing and an infinite ref handled.
template <int VEC>
__device__ __forceinline__ float lane_mass_safe(const float (&z)[VEC], float ref, float c) {
    float ls = 0.0f;
#pragma unroll
    for (int e = 0; e < VEC; ++e) ls = __fadd_rn(ls, (z[e] >= -INFINITY) ? wrel(z[e], ref, c) : 0.0f);
    return ls;
}

// One slice, its vectors already in registers (vectors past the slice read
// as -inf): penalties, slice max and first id, chunk table, header.
template <int DT, bool HIST>
__device__ __forceinline__ void scan_slice(const ScanArgs& a, const uint4 (&d)[kVpt], int row, int cidx,
                                           const ScanRow& R, ScanShared& sh, unsigned char* patch_mem) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int a0 = cidx * a.L;
    const int n = min(a0 + a.L, a.V) - a0;  // > 0: the plan makes no empty slice
    const int nv = (n + VEC - 1) / VEC;
    const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;
    const arc_row_params& P = R.P;
    uint32_t rerr = param_errors(P);
    const RowMode md(P, a.V);
    const int hn = R.hn;
    if (HIST && a.hist_off != nullptr) {
        if (hn < 0) rerr |= ARC_ERR_HIST_ID;
        if (hn > a.hist_cap) rerr |= ARC_ERR_HIST_CAP;
    }
    const bool need_data = rerr == 0;
    const bool row_chunks = need_data && !md.greedy;
    const bool mass = row_chunks && md.need_mass;
    const float cT = mass ? __fdiv_rn(1.4426950408889634f, P.temperature) : 0.0f;

    const uint32_t* pbm = nullptr;
    const uint32_t* pwp = nullptr;
    const float* ppat = nullptr;
    bool has_patch = false;
    if (HIST && need_data && hn > 0) {
        if (tid == 0) sh.sflags = 0;
        __syncthreads();
        const int nwords_max = (kVpt * kThreads * VEC + 31) / 32;
        uint32_t* bm = reinterpret_cast<uint32_t*>(patch_mem);
        uint32_t* wp = bm + nwords_max;
        uint32_t* cnt = wp + nwords_max;
        float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
        const int distinct = build_patches<DT>(rowp, a.V, a0, n, nv, P, a.hist_ids + R.hbeg, hn, bm, wp, cnt, pat,
                                               sh.red32, &sh.sflags);
        rerr |= sh.sflags & ARC_ERR_HIST_ID;
        pbm = bm;
        pwp = wp;
        ppat = pat;
        has_patch = distinct > 0;
    }
    auto vals = [&](int j, float (&z)[VEC]) {
        E::unpack(d[j], z);
        if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, j * kThreads + tid, z);
    };
    auto patched = [&](int j) {
        if (!(HIST && has_patch)) return false;
        const int l0 = (j * kThreads + tid) * VEC;
        return ((pbm[l0 >> 5] >> (l0 & 31)) & ((1u << VEC) - 1u)) != 0;
    };

    // per vector: its max with NaN ignored, and (rows that need masses) the
    // lane's weight sum relative to that max; per lane: the best vector
    float vm[kVpt], ls[kVpt];
    float bv = -INFINITY;
    int bj = -1;
    bool nanf = false;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        const int v = j * kThreads + tid;
        float x = -INFINITY, l = 0.0f;
        if (v < nv) {
            float z[VEC];
            vals(j, z);
            x = patched(j) ? z[0] : E::vmax_nan(d[j]);
            if (patched(j)) {
#pragma unroll
                for (int e = 1; e < VEC; ++e) x = fmax_nan(x, z[e]);
            }
            const bool vnan = (x != x);
            if (vnan) {
                nanf = true;
                x = -INFINITY;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (z[e] > x) x = z[e];
            }
            if (x > bv) {
                bv = x;
                bj = j;
            }
            if (mass && x != -INFINITY)
                l = (vnan || x == INFINITY) ? lane_mass_safe<VEC>(z, x, cT) : lane_mass_packed<VEC>(z, x, cT);
        }
        vm[j] = x;
        ls[j] = l;
    }

    // chunk table: per 32-vector chunk its max and, when needed, the fp32 sum of
    // weights relative to it (NaN ids weigh nothing); every entry is written,
    // entries past the slice as (-inf, 0)
    unsigned char* mysum = const_cast<unsigned char*>(summary_at(a.summaries, a.s, row, cidx));
    if (row_chunks) {
        float2* ch = reinterpret_cast<float2*>(mysum + kHdrBytes);
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            const float mj = key_to_float(__reduce_max_sync(0xFFFFFFFFu, fkey(vm[j])));
            float Sj = 0.0f;
            if (mass) {
                const float lr = (vm[j] != -INFINITY) ? __fmul_rn(ls[j], wrel(vm[j], mj, cT)) : 0.0f;
                Sj = warp_sum_f(lr);
            }
            if (lane == 0) ch[j * kWarps + warp] = make_float2(mj, Sj);
        }
    }

    // slice max and its first id: the warp's best key, then the first id of
    // it among the lanes that hold it
    const uint32_t wkey = __reduce_max_sync(0xFFFFFFFFu, fkey(bv));
    uint32_t mine = 0xFFFFFFFFu;
    if (bj >= 0 && fkey(bv) == wkey) {
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            if (j == bj) {
                float z[VEC];
                vals(j, z);
                int e0 = VEC - 1;
#pragma unroll
                for (int e = VEC - 1; e >= 0; --e)
                    if (z[e] == bv) e0 = e;
                mine = static_cast<uint32_t>(a0 + (j * kThreads + tid) * VEC + e0);
            }
        }
    }
    const uint32_t wid = __reduce_min_sync(0xFFFFFFFFu, mine);
    const bool wnan = __any_sync(0xFFFFFFFFu, nanf);
    if (lane == 0) {
        sh.redf[warp] = (wid == 0xFFFFFFFFu) ? -INFINITY : key_to_float(wkey);
        sh.redi[warp] = (wid == 0xFFFFFFFFu) ? -1 : static_cast<int>(wid);
        sh.rednan[warp] = wnan ? ARC_ERR_NAN : 0u;
    }
    __syncthreads();
    if (tid == 0) {
        float mc = -INFINITY;
        int amc = -1;
        uint32_t nanw = 0;
        for (int w = 0; w < kWarps; ++w) {
            better(mc, amc, sh.redf[w], sh.redi[w]);
            nanw |= sh.rednan[w];
        }
        SliceHeader h;
        h.m = mc;
        h.am = amc;
        h.flags = nanw | (rerr & (ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP));
        h.nchunk = row_chunks ? kChunks : 0;
        h.pad[0] = h.pad[1] = h.pad[2] = h.pad[3] = 0;
        *reinterpret_cast<SliceHeader*>(mysum) = h;
    }
}

// One CTA per slice: every 16-byte load of the slice is issued first (they
// depend on nothing), then the row's parameters; registers stay few so that
// many CTAs per SM keep enough bytes in flight.
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, HIST ? 4 : 6) scan_kernel(const ScanArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ ScanShared sh;
    const int tid = threadIdx.x;
    const int row = static_cast<int>(blockIdx.x) / a.s;
    const int cidx = static_cast<int>(blockIdx.x) - row * a.s;
    const int a0 = cidx * a.L;
    const int n = min(a0 + a.L, a.V) - a0;
    const int nv = (n + VEC - 1) / VEC;
    const char* sp = static_cast<const char*>(a.logits) +
                     (static_cast<int64_t>(row) * a.ld + static_cast<int64_t>(a0)) * E::kBytes;
    const uint4 ninf = (DT == ARC_BF16) ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                        : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    uint4 d[kVpt];
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        const int v = j * kThreads + tid;
        d[j] = (v < nv) ? E::global_vec(sp, v, n, a.aligned) : ninf;
    }
    const ScanRow R = scan_row_of<HIST>(a, row);
    scan_slice<DT, HIST>(a, d, row, cidx, R, sh, dyn);
}

// ------------------------------------------------------------------ finish helpers
// Block-wide max of a u32 (all threads get it); uses red[kWarps].
__device__ __forceinline__ uint32_t block_max_u32(uint32_t v, uint32_t* red) {
    v = __reduce_max_sync(0xFFFFFFFFu, v);
    __syncthreads();
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    uint32_t t = 0;
    for (int w = 0; w < kWarps; ++w) t = max(t, red[w]);
    return t;
}

// Floor search over n weighted keys: the lower edge (to 2^12 keys) of the
// largest key x whose entries at or above it weigh at least tgt in total.
// kw(e, key, weight) gives entry e (u32 weights whose sum fits in 32 bits).
// False when all entries weigh less than tgt.  Two passes of 10 key bits
// over a 1024-bin histogram (native 32-bit shared atomics; bin b lives at
// b + b / 32 so that warp 0 scans it without bank conflicts).
template <class KW>
__device__ bool floor_select(int n, KW kw, uint32_t tgt, uint32_t* hist, FinishScratch& SS, uint32_t& edge) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    auto at = [](int b) { return b + (b >> 5); };
    uint32_t prefix = 0;
    uint32_t rem = tgt;
    for (int pass = 0; pass < 2; ++pass) {
        const int shift = pass == 0 ? 22 : 12;
        for (int b = tid; b < kFloorBins + kFloorBins / 32; b += kThreads) hist[b] = 0;
        __syncthreads();
        for (int e = tid; e < n; e += kThreads) {
            uint32_t key, w;
            kw(e, key, w);
            if (w != 0 && (pass == 0 || (key >> 22) == (prefix >> 22)))
                atomicAdd(&hist[at(static_cast<int>((key >> shift) & (kFloorBins - 1)))], w);
        }
        __syncthreads();
        if (warp == 0) {
            // lane l owns bins 1023 - 32 l down to 992 - 32 l: an inclusive scan
            // in lane order walks the bins from the top key down
            uint32_t loc = 0;
#pragma unroll 8
            for (int q = 0; q < 32; ++q) loc += hist[at(kFloorBins - 1 - 32 * lane - q)];
            uint32_t inc = loc;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
                if (lane >= d) inc += o;
            }
            const uint32_t total = __shfl_sync(0xFFFFFFFFu, inc, 31);
            const uint32_t before = inc - loc;
            if (lane == 0) SS.bi[4] = (total < rem) ? -2 : -1;
            __syncwarp();
            if (total >= rem && before < rem && inc >= rem) {
                uint32_t run = before;
                for (int q = 0; q < 32; ++q) {
                    const int b = kFloorBins - 1 - 32 * lane - q;
                    const uint32_t hb = hist[at(b)];
                    if (run + hb >= rem) {
                        SS.bi[4] = b;
                        SS.bu[4] = run;
                        break;
                    }
                    run += hb;
                }
            }
        }
        __syncthreads();
        const int b = SS.bi[4];
        if (b < 0) return false;  // uniform: every thread reads the same slot
        rem -= static_cast<uint32_t>(SS.bu[4]);
        prefix |= static_cast<uint32_t>(b) << shift;
        __syncthreads();  // the histogram and the slots are rewritten next pass
    }
    edge = prefix;
    return true;
}

// ------------------------------------------------------------------ finish
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, 1) finish_kernel(const FinishArgs a) {
    using E = Elem<DT>;
    using Ctx = RowCtx<DT, HIST>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ KernelShared KS;
    FinishScratch& SS = KS.st;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int s = a.s;
    const int nch = s * kChunks;
    const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;
    const arc_row_params P = load_params(a.params + row);
    uint32_t rerr = param_errors(P);
    const RowMode md(P, a.V);
    const bool greedy = md.greedy, filtered = md.filtered, need_mass = md.need_mass;
    const bool topk_on = md.topk_on, topp_on = md.topp_on, minp_on = md.minp_on;
    const float T = P.temperature;
    const int k = P.top_k;
    const float cT = greedy ? 0.0f : __fdiv_rn(1.4426950408889634f, T);
    int hn = 0, hbeg = 0;
    if (HIST && a.hist_off != nullptr) {
        hbeg = a.hist_off[row];
        hn = max(0, a.hist_off[row + 1] - hbeg);
    }
    float* cm = reinterpret_cast<float*>(dyn + a.cmax_off);
    float* cs = reinterpret_cast<float*>(dyn + a.cs_off);

    // slice headers (warp 0) and, for sampled rows, the chunk tables (warps
    // 0-6); meanwhile one thread of warp 7 takes T ln(min_p) in fp64, whose
    // rate on this part is a small fraction of fp32
    const bool minp_row = minp_on && filtered && rerr == 0;
    if (minp_row && tid == kThreads - 32)
        SS.bd[0] = static_cast<double>(T) * log(static_cast<double>(P.min_p));
    if (!greedy && tid < kThreads - 32) {
        constexpr int kLd = 4;  // chunk entries in flight per thread
        constexpr int kStride = kThreads - 32;
        for (int g0 = tid; g0 < nch; g0 += kLd * kStride) {
            float2 e[kLd];
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int gi = g0 + u * kStride;
                e[u] = (gi < nch) ? chunk_table(summary_at(a.summaries, s, row, gi / kChunks))[gi % kChunks]
                                  : make_float2(0.0f, 0.0f);
            }
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int gi = g0 + u * kStride;
                if (gi < nch) {
                    cm[gi] = e[u].x;
                    cs[gi] = e[u].y;
                }
            }
        }
    }
    if (warp == 0) {
        float v = -INFINITY;
        int i = -1;
        uint32_t f = 0;
        for (int c = lane; c < s; c += 32) {
            const SliceHeader* h = reinterpret_cast<const SliceHeader*>(summary_at(a.summaries, s, row, c));
            better(v, i, h->m, h->am);
            f |= h->flags;
        }
        warp_argmax(v, i);
        f = __reduce_or_sync(0xFFFFFFFFu, f);
        if (lane == 0) {
            SS.bf[0] = v;
            SS.bi[0] = i;
            SS.bi[1] = static_cast<int>(f);
        }
    }
    __syncthreads();
    const float m = SS.bf[0];
    const int am = SS.bi[0];
    const uint32_t rflags = static_cast<uint32_t>(SS.bi[1]);
    const bool row_nan = (rflags & ARC_ERR_NAN) != 0;
    rerr |= rflags & (ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP | ARC_ERR_TIMEOUT);
    uint32_t err = rerr | (rflags & ARC_ERR_NAN);
    int mode;
    int token = -2;
    if (rerr != 0) {
        mode = -1;
        token = -1;
    } else {
        mode = greedy ? 0 : (filtered ? 2 : 1);
        if (am < 0) {
            token = 0;
            err |= ARC_ERR_DEGENERATE;
        } else if (greedy) {
            token = am;
        }
    }
    uint32_t kap_k = 0, kap_r = 0;
    int iot_k = a.V, iot_r = a.V;
    uint64_t mass_k = 0, mass_r = 0, target = 0, rbits = 0;
    int passes = 1;
    const float scale = __uint_as_float(static_cast<uint32_t>(127 + a.F) << 23);
    auto fixq = [&](float w) { return __float2ull_rn(__fmul_rn(w, scale)); };
    // a chunk's fixed-point mass, rescaled from its own max to the row max
    auto chunk_q = [&](int e) -> uint64_t {
        const float mj = cm[e], Sj = cs[e];
        if (mj == -INFINITY || Sj == 0.0f) return 0;
        return fixq(__fmul_rn(Sj, wrel(mj, m, cT)));
    };
    const int cper = (nch + kThreads - 1) / kThreads;  // chunk entries per thread, in id order
    const int ce0 = min(nch, tid * cper), ce1 = min(nch, ce0 + cper);

    if (token == -2) {
        rbits = splitmix64(P.seed ^ (static_cast<uint64_t>(row) << 32) ^ P.step) >> 11;
        if (mode == 1) {
            // total mass and the chunk that holds the draw, in one block scan
            uint64_t loc = 0;
            for (int e = ce0; e < ce1; ++e) loc += chunk_q(e);
            if (tid == 0) SS.bi[2] = -1;
            uint64_t total;
            const uint64_t incl = block_scan_u64(loc, SS.redu, total);
            mass_r = total;
            target = scale_by_u(rbits, total);
            const uint64_t before = incl - loc;
            if (before <= target && target < incl) {
                uint64_t run = before;
                for (int e = ce0; e < ce1; ++e) {
                    const uint64_t q = chunk_q(e);
                    if (q > 0 && run + q > target) {
                        SS.bi[2] = e;
                        SS.bu[2] = run;
                        break;
                    }
                    run += q;
                }
            }
            __syncthreads();
            const int hit = SS.bi[2];
            const uint64_t hit_before = SS.bu[2];
            if (hit < 0) {
                err |= kErrInternal;
                token = am;
            } else if (warp == 0) {
                // re-read the chunk (32 vectors) and walk it
                const int c = hit / kChunks, jr = hit % kChunks;
                const int jround = jr / kWarps, w = jr % kWarps;
                const float mj = cm[hit];
                const float r = wrel(mj, m, cT);
                const int ca0 = c * a.L;
                const int cn = min(ca0 + a.L, a.V) - ca0;
                const int v = jround * kThreads + w * 32 + lane;
                const int cnv = (cn + VEC - 1) / VEC;
                float z[VEC];
                float ls = 0.0f;
                if (v < cnv) {
                    E::unpack(E::global_vec(rowp + static_cast<int64_t>(ca0) * E::kBytes, v, cn, a.aligned), z);
                }
                if (HIST && hn > 0) {
                    // penalties of this chunk's ids, counted from the history 32 ids at a time
                    int cnts[VEC];
#pragma unroll
                    for (int q = 0; q < VEC; ++q) cnts[q] = 0;
                    const int idb = ca0 + v * VEC;
                    for (int h0 = 0; h0 < hn; h0 += 32) {
                        const int hid = (h0 + lane < hn) ? __ldg(a.hist_ids + hbeg + h0 + lane) : -1;
                        for (int t = 0; t < 32; ++t) {
                            const int x = __shfl_sync(0xFFFFFFFFu, hid, t) - idb;
#pragma unroll
                            for (int q = 0; q < VEC; ++q) cnts[q] += (x == q) ? 1 : 0;
                        }
                    }
                    if (v < cnv) {
#pragma unroll
                        for (int q = 0; q < VEC; ++q) {
                            const int id = idb + q;
                            const int cnt = cnts[q];
                            if (cnt > 0 && id < a.V) {
                                float zz = z[q];
                                zz = (zz > 0.0f) ? __fdiv_rn(zz, P.repetition_penalty)
                                                 : __fmul_rn(zz, P.repetition_penalty);
                                zz = __fsub_rn(zz, __fmul_rn(static_cast<float>(cnt), P.frequency_penalty));
                                zz = __fsub_rn(zz, P.presence_penalty);
                                z[q] = zz;
                            }
                        }
                    }
                }
                if (v < cnv && mj != -INFINITY) {
#pragma unroll
                    for (int q = 0; q < VEC; ++q) {
                        const float wq = (z[q] >= -INFINITY) ? wrel(z[q], mj, cT) : 0.0f;
                        ls = __fadd_rn(ls, wq);
                    }
                }
                const uint64_t f = fixq(__fmul_rn(ls, r));
                const uint64_t inc = warp_inclusive_u64(f);
                const uint64_t Q = shfl_u64(inc, 31);
                uint64_t tres = target - hit_before;
                if (Q == 0) {
                    token = -3;  // no lane carries mass: take the row's first max below
                } else {
                    if (tres >= Q) tres = Q - 1;  // rounding gap between the chunk total and its lanes
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, inc > tres);
                    const int l = __ffs(bal) - 1;
                    int eidx = -1;
                    if (lane == l) {
                        const uint64_t t2 = tres - (inc - f);
                        float part = 0.0f;
                        for (int q = 0; q < VEC; ++q) {
                            const float wq = (z[q] >= -INFINITY) ? wrel(z[q], mj, cT) : 0.0f;
                            part = __fadd_rn(part, wq);
                            if (fixq(__fmul_rn(part, r)) > t2) {
                                eidx = q;
                                break;
                            }
                        }
                        if (eidx < 0) eidx = VEC - 1;
                    }
                    eidx = __shfl_sync(0xFFFFFFFFu, eidx, l);
                    token = ca0 + (jround * kThreads + w * 32 + l) * VEC + eidx;
                }
                if (lane == 0) SS.bi[3] = token;
            }
            __syncthreads();
            if (hit >= 0) token = SS.bi[3];
            if (token == -3) token = am;
        } else {
            // ---------------------------------------------------------- filtered rows
            float zm = -INFINITY;  // min-p: z >= zm survives
            if (minp_on) {
                if (tid == 0) SS.bf[1] = __double2float_ru(static_cast<double>(m) + SS.bd[0]);
                __syncthreads();
                zm = SS.bf[1];
            }
            uint64_t S_all = 0;  // top-p over every id: the chunk tables' total mass
            if (need_mass) {
                uint64_t loc = 0;
                for (int e = ce0; e < ce1; ++e) loc += chunk_q(e);
                S_all = block_sum_u64(loc, SS.redu);
            }
            // history patches of the whole row (both selection paths read them)
            const uint32_t* pbm = nullptr;
            const uint32_t* pwp = nullptr;
            const float* ppat = nullptr;
            bool has_patch = false;
            if (HIST && hn > 0) {
                const int nwords_max = (a.fb_rounds * kThreads * VEC + 31) / 32;
                uint32_t* bm = reinterpret_cast<uint32_t*>(dyn + a.fb_patch_off);
                uint32_t* wp = bm + nwords_max;
                uint32_t* cnt = wp + nwords_max;
                float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
                __syncthreads();
                if (tid == 0) KS.st.bi[7] = 0;
                const int nv_row = (a.V + VEC - 1) / VEC;
                const int distinct = build_patches<DT>(rowp, a.V, 0, a.V, nv_row, P, a.hist_ids + hbeg, hn, bm, wp,
                                                       cnt, pat, SS.red32,
                                                       reinterpret_cast<uint32_t*>(&KS.st.bi[7]));
                pbm = bm;
                pwp = wp;
                ppat = pat;
                has_patch = distinct > 0;
            }

            // floor zf: every survivor has z >= zf
            bool fast = true;
            float zf = -INFINITY;
            if (topk_on) {
                // every chunk holds an id >= its max, so k chunk maxima >= x
                // put the k-th largest logit at or above x
                uint32_t edge = 0;
                fast = floor_select(
                    nch,
                    [&](int e, uint32_t& key, uint32_t& w) {
                        const float x = cm[e];
                        key = fkey(x);
                        w = (x > -INFINITY) ? 1u : 0u;
                    },
                    static_cast<uint32_t>(k), KS.fhist, SS, edge);
                if (fast) zf = Ctx::lo_float(edge);
            } else if (minp_on) {
                zf = zm;
            } else {
                // top-p alone: the chunk maxima at or above x already carry
                // at least the target mass
                if (tid == 0) SS.bu[5] = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(S_all)));
                __syncthreads();
                uint64_t tgt = SS.bu[5];
                if (tgt == 0) tgt = 1;
                // masses in units of 2^sh rounded down, the target rounded up:
                // the bound stays valid and every sum fits in 32 bits
                const int sh = max(0, a.F - 19);
                const uint32_t tgt32 = static_cast<uint32_t>((tgt + (uint64_t{1} << sh) - 1) >> sh);
                uint32_t edge = 0;
                fast = floor_select(
                    nch,
                    [&](int e, uint32_t& key, uint32_t& w) {
                        const float x = cm[e];
                        key = fkey(x);
                        w = (x > -INFINITY) ? static_cast<uint32_t>(fixq(wrel(x, m, cT)) >> sh) : 0u;
                    },
                    tgt32, KS.fhist, SS, edge);
                if (fast) zf = Ctx::lo_float(edge);
            }
            fast = fast && zf > -INFINITY;

            // candidate chunks: max >= zf, in id order
            int* clist = reinterpret_cast<int*>(dyn + a.clist_off);
            int nclist = 0;
            if (fast) {
                uint64_t loc = 0;
                for (int e = ce0; e < ce1; ++e) loc += (cm[e] >= zf) ? 1u : 0u;
                uint64_t total;
                const uint64_t incl = block_scan_u64(loc, SS.redu, total);
                int pos = static_cast<int>(incl - loc);
                for (int e = ce0; e < ce1; ++e)
                    if (cm[e] >= zf) clist[pos++] = e;
                nclist = static_cast<int>(total);
                fast = nclist <= kCandChunks;
                __syncthreads();
            }

            // gather the ids >= zf of those chunks, in id order: (key, id, mass)
            uint32_t* ck = reinterpret_cast<uint32_t*>(dyn + a.cand_off);
            int* ci = reinterpret_cast<int*>(ck + kCandCap);
            uint64_t* cw = reinterpret_cast<uint64_t*>(ci + kCandCap);
            const bool infm = (m == INFINITY);
            auto weight_of = [&](float z) -> float {
                return infm ? (z == m ? 1.0f : 0.0f) : ex2(__fmul_rn(__fsub_rn(z, m), cT));
            };
            int nc = 0;
            if (fast) {
                // warp w takes list entries w, w + 8, ...; kCollectU of its chunks'
                // 16-byte vectors are in flight per lane; slots come from one counter
                const int Lv = a.L / VEC;
                if (tid == 0) SS.ccount = 0;
                __syncthreads();
                for (int r0 = warp; r0 < nclist; r0 += kWarps * kCollectU) {
                    uint4 raw[kCollectU];
                    int vrow[kCollectU];
#pragma unroll
                    for (int u = 0; u < kCollectU; ++u) {
                        const int li = r0 + u * kWarps;
                        vrow[u] = -1;
                        raw[u] = make_uint4(0u, 0u, 0u, 0u);
                        if (li < nclist) {
                            const int gi = clist[li];
                            const int c = gi / kChunks, jj = gi % kChunks;
                            const int vs = jj * 32 + lane;
                            const int sa0 = c * a.L;
                            const int sn = min(sa0 + a.L, a.V) - sa0;
                            if (vs < (sn + VEC - 1) / VEC) {
                                raw[u] = E::global_vec(rowp + static_cast<int64_t>(sa0) * E::kBytes, vs, sn, a.aligned);
                                vrow[u] = c * Lv + vs;
                            }
                        }
                    }
#pragma unroll
                    for (int u = 0; u < kCollectU; ++u) {
                        if (r0 + u * kWarps >= nclist) break;  // uniform over the warp
                        float z[VEC];
                        int cnt = 0;
                        if (vrow[u] >= 0) {
                            E::unpack(raw[u], z);
                            if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, vrow[u], z);
#pragma unroll
                            for (int e = 0; e < VEC; ++e) cnt += (z[e] >= zf) ? 1 : 0;
                        }
                        int inc = cnt;
#pragma unroll
                        for (int dd = 1; dd < 32; dd <<= 1) {
                            const int o = __shfl_up_sync(0xFFFFFFFFu, inc, dd);
                            if (lane >= dd) inc += o;
                        }
                        const int tot = __shfl_sync(0xFFFFFFFFu, inc, 31);
                        if (tot == 0) continue;
                        uint32_t base = 0;
                        if (lane == 31) base = atomicAdd(&SS.ccount, static_cast<uint32_t>(tot));
                        base = __shfl_sync(0xFFFFFFFFu, base, 31);
                        int pos = static_cast<int>(base) + inc - cnt;
                        if (cnt > 0) {
#pragma unroll
                            for (int e = 0; e < VEC; ++e) {
                                if (z[e] >= zf) {
                                    if (pos < kCandCap) {
                                        ck[pos] = fkey(z[e]);
                                        ci[pos] = vrow[u] * VEC + e;
                                        cw[pos] = fixq(weight_of(z[e]));
                                    }
                                    ++pos;
                                }
                            }
                        }
                    }
                }
                __syncthreads();
                nc = static_cast<int>(SS.ccount);
                fast = nc <= kCandCap;
            }

            if (fast) {
                // ------------------------------------------------------ direct selection
                // candidates sit in gather order: ties are broken by id
                Surv K{-INFINITY, INT_MAX};
                if (topk_on) {
                    // K: the first k ids by (z desc, id asc)
                    if (tid == 0) SS.bi[5] = -1;
                    __syncthreads();
                    for (int i = tid; i < nc; i += kThreads) {
                        const uint32_t ki = ck[i];
                        const int ii = ci[i];
                        int rk = 0;
                        for (int j = 0; j < nc; ++j) {
                            const uint32_t kj = ck[j];
                            rk += (kj > ki || (kj == ki && ci[j] < ii)) ? 1 : 0;
                        }
                        if (rk == k - 1) SS.bi[5] = i;
                    }
                    __syncthreads();
                    const int wi = SS.bi[5];
                    if (wi < 0) {
                        err |= kErrInternal;
                    } else {
                        const uint32_t kw = ck[wi];
                        const int iw = ci[wi];
                        int later = 0;
                        for (int i = tid; i < nc; i += kThreads) later |= (ck[i] == kw && ci[i] > iw) ? 1 : 0;
                        later = __syncthreads_or(later);
                        K = Surv{key_to_float(kw), later ? iw + 1 : INT_MAX};
                    }
                    kap_k = (K.zt == -INFINITY && K.ge_form()) ? 0u : fkey(K.zt);
                    iot_k = K.ge_form() ? a.V : K.iota;
                    // ids outside K get key 0 (no real logit has it)
                    uint64_t loc = 0;
                    for (int i = tid; i < nc; i += kThreads) {
                        if (!K.test(key_to_float(ck[i]), ci[i]))
                            ck[i] = 0u;
                        else
                            loc += cw[i];
                    }
                    mass_k = block_sum_u64(loc, SS.redu);
                } else {
                    mass_k = S_all;
                }
                bool found = false;
                float zp = -INFINITY;
                if (topp_on) {
                    // largest key whose mass at or above it reaches ceil(p * mass_k)
                    if (tid == 0) SS.bu[5] = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(mass_k)));
                    __syncthreads();
                    uint64_t tgt = SS.bu[5];
                    if (tgt == 0) tgt = 1;
                    uint32_t best = 0;
                    for (int i = tid; i < nc; i += kThreads) {
                        const uint32_t ki = ck[i];
                        if (ki == 0u) continue;
                        uint64_t mge = 0;
                        for (int j = 0; j < nc; ++j) mge += (ck[j] >= ki) ? cw[j] : 0u;
                        if (mge >= tgt) best = max(best, ki);
                    }
                    best = block_max_u32(best, SS.red32);
                    found = best != 0u;
                    if (found) zp = key_to_float(best);
                }
                if (topp_on && !found && !minp_on && !topk_on) err |= kErrInternal;  // the floor guarantees it
                const float zx = found ? fmaxf(zp, zm) : zm;
                const Surv R = (zx > K.zt) ? Surv{zx, INT_MAX} : K;
                kap_r = (R.zt == -INFINITY && R.ge_form()) ? 0u : fkey(R.zt);
                iot_r = R.ge_form() ? a.V : R.iota;
                // survivors' mass, then the draw in id order: each survivor sums
                // the survivors with smaller ids
                auto surv_q = [&](int i) -> uint64_t {
                    const uint32_t ki = ck[i];
                    return (ki != 0u && R.test(key_to_float(ki), ci[i])) ? cw[i] : 0u;
                };
                uint64_t loc = 0;
                for (int i = tid; i < nc; i += kThreads) loc += surv_q(i);
                if (tid == 0) SS.bi[6] = -1;
                mass_r = block_sum_u64(loc, SS.redu);
                target = scale_by_u(rbits, mass_r);
                for (int i = tid; i < nc; i += kThreads) {
                    const uint64_t qi = surv_q(i);
                    if (qi == 0) continue;
                    const int ii = ci[i];
                    uint64_t before = 0;
                    for (int j = 0; j < nc; ++j) before += (ci[j] < ii) ? surv_q(j) : 0u;
                    if (before <= target && target < before + qi) SS.bi[6] = ii;
                }
                __syncthreads();
                token = SS.bi[6];
                if (token < 0) {
                    token = am;
                    err |= kErrInternal;
                }
            } else {
                // ------------------------------------------------------ general path
                __syncthreads();
                cg::cluster_group cl = cg::this_cluster();
                Ctx X(KS.fb, cl);
                X.s = 1;
                X.rank = 0;
                X.row = row;
                X.tid = tid;
                X.lane = lane;
                X.warp = warp;
                X.a0 = 0;
                X.a1 = a.V;
                X.n = a.V;
                X.nv = (a.V + VEC - 1) / VEC;
                X.nvf = a.V / VEC;
                X.rounds = (X.nv + kThreads - 1) / kThreads;
                X.data = reinterpret_cast<const unsigned char*>(rowp);
                X.src_global = true;
                X.src_aligned = a.aligned != 0;
                X.vmax = cm;
                X.vps = a.L / VEC;
                X.cps = kChunks;
                X.Wsum = reinterpret_cast<uint64_t*>(dyn + a.fb_wsum_off);
                X.par = 0;
                X.passes = 0;
                X.epoch = 1;
                X.ghist_zeroed = -1;
                X.cand_zeroed = -1;
                X.has_patch = has_patch;
                X.row_nan = row_nan;
                X.bm = pbm;
                X.wp = pwp;
                X.patch = ppat;
                X.m = m;
                X.c = cT;
                X.scale = scale;
                X.infm = infm;
                for (int b = tid; b < kBins; b += kThreads) KS.fb.ghist[b] = 0;
                if (tid == 0) {
                    KS.fb.ccount = 0;
                    KS.fb.flags = 0;
                }
                __syncthreads();
                const uint32_t Km = fkey(m);
                Surv K{-INFINITY, INT_MAX};
                if (topk_on) {
                    K = select_topk(X, k, Km, err);
                    kap_k = (K.zt == -INFINITY && K.ge_form()) ? 0u : fkey(K.zt);
                    iot_k = K.ge_form() ? a.V : K.iota;
                }
                Surv R = K;
                bool wsum_is_R = false;
                if (topp_on) {
                    if (tid == 0)
                        SS.bf[2] = __double2float_rd(static_cast<double>(m) +
                                                     static_cast<double>(T) * log((1.0 - static_cast<double>(P.top_p)) /
                                                                                  (2.0 * static_cast<double>(a.V))));
                    __syncthreads();
                    const float zb = SS.bf[2];
                    const float zfloor = fmaxf(zm, K.zt);
                    float zlo = fmaxf(zb, zfloor);
                    Window W = Ctx::make_window(fkey(zlo), Km);
                    const int mk = mass_mode(X, K);
                    if (topk_on) {
                        pass_mass<Ctx, true>(X, mk, K, W);
                        X.publish_wsum_total(0);
                        X.push_hist();
                        X.xsync();
                        mass_k = X.xscan(0, ~0ull).total;
                        X.xnext();
                    } else {
                        // K is every id: its mass is the chunk tables' total
                        pass_hist<Ctx, true>(X, W, K);
                        X.push_hist();
                        X.xsync();
                        mass_k = S_all;
                    }
                    if (tid == 0) SS.bu[5] = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(mass_k)));
                    __syncthreads();
                    uint64_t tgt = SS.bu[5];
                    if (tgt == 0) tgt = 1;
                    float zp = -INFINITY;
                    bool found = select_mass(X, W, K, tgt, zp);
                    if (!found && zlo > zfloor) {
                        zlo = zfloor;
                        W = Ctx::make_window(fkey(zlo), Km);
                        pass_hist<Ctx, true>(X, W, K);
                        X.push_hist();
                        X.xsync();
                        found = select_mass(X, W, K, tgt, zp);
                    }
                    const float zx = found ? fmaxf(zp, zm) : zm;
                    if (zx > K.zt)
                        R = Surv{zx, INT_MAX};
                    else
                        wsum_is_R = topk_on;  // Wsum holds K's masses only when top-k ran
                } else if (minp_on && zm > K.zt) {
                    R = Surv{zm, INT_MAX};
                }
                kap_r = (R.zt == -INFINITY && R.ge_form()) ? 0u : fkey(R.zt);
                iot_r = R.ge_form() ? a.V : R.iota;
                const int mr = mass_mode(X, R);
                if (!wsum_is_R) pass_mass<Ctx, false>(X, mr, R, Window{0u, 0u, 0});
                X.publish_wsum_total(0);
                X.xsync();
                mass_r = X.xscan(0, ~0ull).total;
                target = scale_by_u(rbits, mass_r);
                X.xnext();
                int tok = X.walk(
                    target, [&](const float(&z)[VEC], int g0) { return X.vec_mass(mr, z, g0, R); },
                    [&](const float(&z)[VEC], int g0, uint64_t tt) { return X.vec_mass_walk(mr, z, g0, R, tt); });
                if (tok < 0) {
                    tok = am;
                    err |= kErrInternal;
                }
                token = tok;
                passes = 1 + X.passes;
            }
        }
    }

    // -------------------------------------------------------------- results
    if (tid == 0) {
        a.out[row] = token;
        if (err != 0 && a.err_word) atomicOr(a.err_word, err);
        if (a.debug) {
            arc_row_debug& dbg = a.debug[row];
            dbg.mode = mode;
            dbg.err = err;
            dbg.token = token;
            dbg.passes = passes;
            dbg.kappa_k = kap_k;
            dbg.iota_k = iot_k;
            dbg.kappa_r = kap_r;
            dbg.iota_r = iot_r;
            dbg.max_z = m;
            dbg.frac_bits = a.F;
            dbg.rbits = rbits;
            dbg.mass_k = mass_k;
            dbg.mass_r = mass_r;
            dbg.target = target;
        }
        if (a.flags & ARC_OPT_STEP_AUTOINC) a.params[row].step = P.step + 1;
    }
}

}  // namespace arc
