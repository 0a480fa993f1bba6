// On-device sampling in two kernels, one HBM pass over the logits.
//
// scan_kernel: a row is split into s slices of at most kVpt * kThreads
// 16-byte vectors; one CTA per slice issues all its 16-byte loads first (they
// depend on nothing), applies the history penalties in registers, and writes
// a small summary to the workspace: per warp the max of its vectors (with its
// first id for greedy rows and rows with a history), and per 32-vector chunk
// (256 bf16 / 128 fp32 logits) the chunk max, for rows that need masses the
// fp32 sum of 2^((z - chunk max) log2(e) / T), and for filtered rows where
// the max lies and the largest max of the chunk's other vectors.  No CTA
// waits for another, no warp for another (rows with history excepted), and
// registers stay at 32, so 8 CTAs per SM keep HBM busy.
//
// finish_kernel: one CTA per row combines the slice summaries.
//  - greedy rows take the row max;
//  - default rows draw from the chunk masses (exact integer fixed point,
//    rescaled to the row max) with one block scan, and re-read only the chunk
//    that holds the draw;
//  - filtered rows first bound the cutoff from below with the chunk maxima
//    (the k-th largest chunk max for top-k, the min-p threshold, or a mass
//    bound for top-p), gather the few ids at or above that floor from the
//    chunks that can hold them into shared memory, and select exactly there
//    by ranking.  When the floor admits too many ids, the general threshold
//    bisection of row_select.cuh runs over the row instead.
#pragma once

#include <climits>

#include "commit_row.cuh"
#include "row_select.cuh"

namespace arc {

constexpr int kVpt = 4;                  // 16-byte vectors per thread in a scan CTA
constexpr int kChunks = kVpt * kWarps;   // chunks per slice summary (32-vector chunks)
constexpr int kHdrBytes = kWarps * 16;   // per-warp records of a slice
constexpr int kEntryBytes = kChunks * 16;  // chunk entries of a slice
constexpr int kWideK = 64;               // top-k rows with larger k record more per chunk (see WideEntry)
// a slice summary: warp records, chunk entries, and (filtered rows) the raw
// 16-byte vector holding each chunk's max
constexpr int kSummaryBytes = kHdrBytes + 3 * kEntryBytes;
constexpr int kMaxRowCtas = 128;         // slices per row at most
constexpr int kCandCap = 2048;           // ids the direct selection holds
constexpr int kRankMax = 256;            // candidates ranked by counting; more are sorted

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
    int top_n;      // > 0: every row records chunk masses, maxima and max vectors
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
    int top_n;                       // > 0: write the row's top-n log-probabilities
    arc_top_logprob* top_logprobs;   //   [B][top_n]
    const unsigned char* summaries;
    int hist_cap;
    int F;
    uint32_t flags;
    int aligned;
    int cmax_off;      // dynamic shared memory: chunk maxima of the row,
    int cs_off;        //   chunk masses,
    int cid_off;       //   chunk max vectors,
    int cv2_off;       //   chunk second vector maxima,
    int cmv_off;       //   chunk max vectors (-1: read from the logits instead),
    int cwide_off;     //   wide entries of top-k rows with large k (-1: none),
    int clist_off;     //   per-warp candidate chunk lists,
    int cand_off;      //   candidates (key, id, mass),
    int sorted_off;    //   the candidates in (key desc, id asc) order,
    int fb_wsum_off;   //   per-(round, warp) masses,
    int fb_patch_off;  //   row patch tables
    int fb_rounds;     // rounds of a whole row
    int fin_g;         // finish CTAs per row (a cluster when > 1)
    arc_commit_target commit;  // decode-loop commit of each row after its token (ring NULL: none)
};

// One warp's share of a slice, as the scan kernel summarises it: each warp
// writes its own record, so the scan needs no barrier between its warps.
struct __align__(16) WarpRecord {
    float m;         // max of the warp's vectors (NaN-free), -inf when none
    int am;          // its first id, -1 when none, kAmUnknown when left open
    uint32_t flags;  // ARC_ERR_NAN | ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP
    int pad;
};
static_assert(sizeof(WarpRecord) * kWarps == kHdrBytes, "slice record size");

struct FinishScratch {
    uint64_t redu[kWarps];
    uint32_t red32[kWarps];
    int bi[8];
    uint64_t bu[8];
    float bf[8];
    uint32_t ccount;  // candidates gathered
    uint32_t nwhole;  // chunks listed for a whole read
    int draw_bin;              // draw over many survivors: the id range holding the target,
    uint32_t draw_n;           //   its survivors,
    uint64_t draw_base;        //   the mass of the ranges before it
    unsigned long long chead;  // decode-loop commit: the ring head this call read,
    int32_t cpos;              //   the row's position
    uint32_t cown;             //   and owner tag
    uint32_t fc[2][kWarps][4];  // floor search partial counts
    double bd[2];
};

struct __align__(16) KernelShared {
    SampleShared fb;  // general selection path
    FinishScratch st;
};

__device__ __forceinline__ const unsigned char* summary_at(const unsigned char* base, int s, int row, int c) {
    return base + (static_cast<size_t>(row) * s + c) * kSummaryBytes;
}
// One 32-vector chunk of a slice, as the scan kernel summarises it.
struct __align__(16) ChunkEntry {
    float m;   // chunk max (NaN ignored), -inf when the chunk holds no number
    float S;   // rows that need masses: fp32 sum of 2^((z - m) log2(e) / T), else 0
    int lane;  // filtered rows: the vector (lane) of the chunk holding the max first, else -1
    float u2;  // filtered rows: the largest max of the chunk's other vectors, else +inf
};
static_assert(sizeof(ChunkEntry) == 16, "chunk entry size");

__device__ __forceinline__ const ChunkEntry* chunk_table(const unsigned char* sm) {
    return reinterpret_cast<const ChunkEntry*>(sm + kHdrBytes);
}
__device__ __forceinline__ const uint4* max_vectors(const unsigned char* sm) {
    return reinterpret_cast<const uint4*>(sm + kHdrBytes + kEntryBytes);
}
// Top-k rows with k > kWideK: the third and fourth largest vector maxima of a
// chunk and the lanes of its second and third, so that the k-th largest of
// the four maxima per chunk bounds the k-th logit from below and a chunk
// whose fourth is below that floor is read as at most three known vectors.
struct __align__(16) WideEntry {
    float u3, u4;
    int lane2, lane3;  // -1 when none
};
static_assert(sizeof(WideEntry) == 16, "wide entry size");
__device__ __forceinline__ const WideEntry* wide_entries(const unsigned char* sm) {
    return reinterpret_cast<const WideEntry*>(sm + kHdrBytes + 2 * kEntryBytes);
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
    // the rank of word w's first bit is kept for even w only (half the
    // table): an odd word adds its even neighbour's bit count
    uint32_t run = wbase + inc - mine;
    for (int w = w0; w < w1; ++w) {
        if (!(w & 1)) wp[w >> 1] = run;
        run += __popc(bm[w]);
    }
    for (int q = tid; q < static_cast<int>(distinct); q += kThreads) cnt[q] = 0;
    __syncthreads();
    auto rank_of = [&](int li) { return patch_rank(bm, wp, li); };
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
        const int base = patch_word_base(bm, wp, l0 >> 5);
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
// value and sets total.  Uses red[kWarps]; `fresh`: every earlier reader of
// red is already behind a barrier, so the leading one is skipped.
__device__ __forceinline__ uint64_t block_scan_u64(uint64_t v, uint64_t* red, uint64_t& total, bool fresh = false) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const uint64_t inc = warp_inclusive_u64(v);
    if (!fresh) __syncthreads();
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
// Row-level facts every CTA of a row needs, decided once per CTA by warp 0
// while the slice's loads are in flight.
enum : uint32_t {
    kRowArgmax = 1u,  // greedy rows and rows with invalid parameters: slice max and first id
    kRowChunks = 2u,  // chunk table
    kRowMass = 4u,    // chunk masses
    kRowFiltered = 8u,  // chunk max vectors and second vector maxima
};
constexpr int kAmUnknown = INT_MAX;  // slice record of a row whose first max id the scan leaves open

struct ScanShared {
    uint32_t red32[kWarps];
    uint32_t sflags;  // history id errors (written only after a barrier past its init)
};

// What the scan does for a row, decoded by every thread from its parameter
// record: no barrier, no validation.  Rows with invalid parameters are
// rejected by the finish kernel, which reads nothing the scan wrote for them
// but the error flags; only a history length outside [0, cap] must keep the
// scan from building penalties.
struct ScanRowInfo {
    uint32_t bits;
    uint32_t rerr;  // history length errors
    float cT;       // log2(e) / T for rows that need masses
    arc_row_params P;
    int hbeg, hn;
};

// The row's parameter record through the non-coherent path (the finish kernel
// of an earlier call may have rewritten `step`, never while this kernel
// runs): the first two words (temperature, top_k, top_p, min_p), or all six
// for rows with history.  Volatile, so that these loads go out before the
// slice's.
template <bool HIST>
__device__ __forceinline__ void params_words_nc(const arc_row_params* p, uint64_t (&w)[6]) {
    const uint64_t* q = reinterpret_cast<const uint64_t*>(p);
#pragma unroll
    for (int i = 0; i < 6; ++i) {
        if (i < 2 || HIST)
            asm volatile("ld.global.nc.u64 %0, [%1];" : "=l"(w[i]) : "l"(q + i));
        else
            w[i] = 0;
    }
}

template <bool HIST>
__device__ __forceinline__ ScanRowInfo scan_row_info(const ScanArgs& a, int row, const uint64_t (&pw)[6]) {
    ScanRowInfo R;
    R.P = params_from_words(pw);
    const RowMode md(R.P, a.V);  // reads temperature, top_k, top_p and min_p only
    R.rerr = 0;
    R.hbeg = 0;
    R.hn = 0;
    if (HIST && a.hist_off != nullptr) {
        R.hbeg = a.hist_off[row];
        R.hn = a.hist_off[row + 1] - R.hbeg;
        if (R.hn < 0) R.rerr |= ARC_ERR_HIST_ID;
        if (R.hn > a.hist_cap) R.rerr |= ARC_ERR_HIST_CAP;
    }
    if (R.rerr != 0 || md.greedy) {
        R.bits = kRowArgmax;
    } else {
        R.bits = kRowChunks | (md.need_mass ? kRowMass : 0u) | (md.filtered ? kRowFiltered : 0u);
        if (HIST) R.bits |= kRowArgmax;  // penalised rows keep their first max id
    }
    // top-n log-probabilities: the masses at the row's temperature (1 for a
    // greedy row) and the chunk maxima and max vectors of every row
    if (a.top_n > 0 && R.rerr == 0) R.bits |= kRowChunks | kRowMass | kRowFiltered;
    const float Tm = R.P.temperature > 0.0f ? R.P.temperature : 1.0f;
    R.cT = (R.bits & kRowMass) ? __fdiv_rn(1.4426950408889634f, Tm) : 0.0f;
    return R;
}

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

// The same for 8 bf16 logits held raw in a 16-byte vector: z - ref by
// mixed-precision subtraction (the bf16 operand is exact, one rounding, as
// unpacking then subtracting), then the same products, powers and sums.
__device__ __forceinline__ float lane_mass_bf16(const uint4& v, float ref, float c) {
    float t[8];
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i)
        asm("{\n\t.reg .b16 lo, hi;\n\tmov.b32 {lo, hi}, %2;\n\t"
            "sub.rn.f32.bf16 %0, lo, %3;\n\tsub.rn.f32.bf16 %1, hi, %3;\n\t}"
            : "=f"(t[2 * i]), "=f"(t[2 * i + 1])
            : "r"(w[i]), "f"(ref));
    const float2 c2 = make_float2(c, c);
    float2 acc = make_float2(0.0f, 0.0f);
#pragma unroll
    for (int e = 0; e < 8; e += 2) {
        const float2 x = __fmul2_rn(make_float2(t[e], t[e + 1]), c2);
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

// Warp max of a NaN-free float.
__device__ __forceinline__ float warp_max_nonan(float v) {
    float r;
    asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(r) : "f"(v));
    return r;
}

// NV warp sums at once (NV a power of two <= 32): lane l ends with the sum
// over the warp of v[l / (32 / NV)] (lanes 0, 32/NV, 2*32/NV, ... hold sums
// 0, 1, 2, ...).  Each halving step keeps the half of the values that the
// lane's bit selects and adds the partner's copy of it.
template <int NV>
__device__ __forceinline__ float warp_sum_n(const float (&v)[NV], int lane) {
    float a[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) a[i] = v[i];
    int d = 16;
#pragma unroll
    for (int h = NV / 2; h >= 1; h /= 2, d /= 2) {
        const bool up = (lane & d) != 0;
#pragma unroll
        for (int i = 0; i < h; ++i) {
            const float keep = up ? a[i + h] : a[i];
            const float send = up ? a[i] : a[i + h];
            a[i] = __fadd_rn(keep, __shfl_xor_sync(0xFFFFFFFFu, send, d));
        }
    }
    float b = a[0];
#pragma unroll
    for (; d > 0; d /= 2) b = __fadd_rn(b, __shfl_xor_sync(0xFFFFFFFFu, b, d));
    return b;
}

// The j-th of a thread's vectors, for a j the compiler cannot see.
__device__ __forceinline__ uint4 pick(const uint4 (&d)[kVpt], int j) {
    uint4 r = d[0];
#pragma unroll
    for (int i = 1; i < kVpt; ++i)
        if (j == i) r = d[i];
    return r;
}

// One slice, its vectors already in registers (vectors past the slice read
// as -inf): penalties, chunk table, per-warp records.
template <int DT, bool HIST>
__device__ __forceinline__ void scan_slice(const ScanArgs& a, const uint4 (&d)[kVpt], int row, int cidx,
                                           const ScanRowInfo& R, ScanShared& sh, unsigned char* patch_mem,
                                           unsigned char* mysum) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    constexpr int kSumLanes = 32 / kVpt;  // lane kSumLanes * j holds chunk j's mass
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int a0 = cidx * a.L;
    const int n = min(a0 + a.L, a.V) - a0;  // > 0: the plan makes no empty slice
    const int nv = (n + VEC - 1) / VEC;
    const uint32_t bits = R.bits;
    uint32_t rerr = R.rerr;

    const uint32_t* pbm = nullptr;
    const uint32_t* pwp = nullptr;
    const float* ppat = nullptr;
    bool has_patch = false;
    if (HIST && rerr == 0 && R.hn > 0) {
        if (threadIdx.x == 0) sh.sflags = 0;
        __syncthreads();
        const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;
        const int nwords_max = (kVpt * kThreads * VEC + 31) / 32;
        uint32_t* bm = reinterpret_cast<uint32_t*>(patch_mem);
        uint32_t* wp = bm + nwords_max;
        uint32_t* cnt = wp + (nwords_max + 1) / 2;
        float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
        const int distinct = build_patches<DT>(rowp, a.V, a0, n, nv, R.P, a.hist_ids + R.hbeg, R.hn, bm, wp, cnt,
                                               pat, sh.red32, &sh.sflags);
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

    // vector maxima with NaN ignored (-inf for vectors past the slice, which
    // were loaded as -inf); NaN is rare: one test for the thread's vectors
    float xs[kVpt];
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        if (j * kThreads + tid < nv && patched(j)) {
            float z[VEC];
            vals(j, z);
            float x = z[0];
#pragma unroll
            for (int e = 1; e < VEC; ++e) x = fmax_nan(x, z[e]);
            xs[j] = x;
        } else {
            xs[j] = E::vmax_nan(d[j]);
        }
    }
    uint32_t vn = 0;  // vectors holding a NaN
    bool anynan = false;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) anynan |= (xs[j] != xs[j]);
    if (anynan) {
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            if (xs[j] != xs[j]) {
                vn |= 1u << j;
                float z[VEC];
                vals(j, z);
                float x = -INFINITY;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (z[e] > x) x = z[e];
                xs[j] = x;
            }
        }
    }
    const bool wnan = __any_sync(0xFFFFFFFFu, vn != 0);

    float wm = -INFINITY;
    int wam = -1;
    if (bits & kRowChunks) {
        // per 32-vector chunk (the warp's vectors j): the chunk max; rows that
        // need masses: the fp32 sum of weights relative to it (NaN ids weigh
        // nothing); filtered rows: the vector holding the max first and the
        // largest max of the other vectors, so that a chunk with one vector at
        // or above a later floor is re-read as that one 16-byte vector.  Lane
        // 8j writes entry j.  Every entry is written; entries past the slice
        // hold no number.
        float mj[kVpt];
#pragma unroll
        for (int j = 0; j < kVpt; ++j) mj[j] = warp_max_nonan(xs[j]);
        float S = 0.0f;
        if (bits & kRowMass) {
            const float cT = R.cT;
            float sl[kVpt];
            bool plain = DT == ARC_BF16 && !(HIST && has_patch) && !wnan;
#pragma unroll
            for (int j = 0; j < kVpt; ++j) plain &= mj[j] < INFINITY;
            if (plain) {
                // the common case, decided once for the warp: every lane by the
                // raw-vector formula; -inf logits (padding included) weigh 0, and a
                // chunk with no number takes any finite reference
#pragma unroll
                for (int j = 0; j < kVpt; ++j) sl[j] = lane_mass_bf16(d[j], fmaxf(mj[j], -3.0e38f), cT);
            } else {
#pragma unroll
                for (int j = 0; j < kVpt; ++j) {
                    float l = 0.0f;
                    if (xs[j] != -INFINITY) {  // then mj[j] >= xs[j] > -inf
                        float z[VEC];
                        vals(j, z);
                        l = (((vn >> j) & 1u) || mj[j] == INFINITY) ? lane_mass_safe<VEC>(z, mj[j], cT)
                                                                    : lane_mass_packed<VEC>(z, mj[j], cT);
                    }
                    sl[j] = l;
                }
            }
            S = warp_sum_n<kVpt>(sl, lane);
        }
        // entry j as soon as its fields are known, by lane 8j (which holds the
        // chunk's mass): nothing per chunk stays live across the loop
        ChunkEntry* ch = reinterpret_cast<ChunkEntry*>(mysum + kHdrBytes);
        uint4* mvec = reinterpret_cast<uint4*>(mysum + kHdrBytes + kEntryBytes);
        WideEntry* wide = reinterpret_cast<WideEntry*>(mysum + kHdrBytes + 2 * kEntryBytes);
        const bool filtered = (bits & kRowFiltered) != 0;
        const bool wide_row = filtered && R.P.top_k > kWideK && R.P.top_k < a.V;
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            int fl = -1;
            float u2 = INFINITY;
            if (filtered) {
                const unsigned holders = __ballot_sync(0xFFFFFFFFu, xs[j] == mj[j] && xs[j] > -INFINITY);
                fl = holders ? __ffs(holders) - 1 : -1;
                u2 = warp_max_nonan(lane == fl ? -INFINITY : xs[j]);
                // the max's vector as loaded (history patches are applied by
                // the reader), so that a chunk with one vector at or above a
                // later floor needs no second read of the logits
                if (lane == fl) mvec[j * kWarps + warp] = d[j];
            }
            if (lane == kSumLanes * j) {
                ChunkEntry ce;
                ce.m = mj[j];
                ce.S = S;
                ce.lane = fl;
                ce.u2 = u2;
                ch[j * kWarps + warp] = ce;
            }
        }
        if (wide_row) {
            // per chunk: the vectors holding the largest and second largest
            // maxima (by position), then the third and fourth largest maxima
#pragma unroll
            for (int j = 0; j < kVpt; ++j) {
                const float x = xs[j];
                const unsigned h1 = __ballot_sync(0xFFFFFFFFu, x == mj[j] && x > -INFINITY);
                const int fl = h1 ? __ffs(h1) - 1 : -1;
                const float u2 = warp_max_nonan(lane == fl ? -INFINITY : x);
                const unsigned h2 = __ballot_sync(0xFFFFFFFFu, lane != fl && x == u2 && u2 > -INFINITY);
                const int fl2 = h2 ? __ffs(h2) - 1 : -1;
                const float u3 = warp_max_nonan((lane == fl || lane == fl2) ? -INFINITY : x);
                const unsigned h3 = __ballot_sync(0xFFFFFFFFu, lane != fl && lane != fl2 && x == u3 && u3 > -INFINITY);
                const int fl3 = h3 ? __ffs(h3) - 1 : -1;
                const float u4 = warp_max_nonan((lane == fl || lane == fl2 || lane == fl3) ? -INFINITY : x);
                if (lane == 0) wide[j * kWarps + warp] = WideEntry{u3, u4, fl2, fl3};
            }
        }
        wm = mj[0];
#pragma unroll
        for (int j = 1; j < kVpt; ++j) wm = fmaxf(wm, mj[j]);
        wam = wm > -INFINITY ? kAmUnknown : -1;
    }
    if (bits & kRowArgmax) {
        // the warp's max and its first id: the best key, then the first id of
        // it among the lanes that hold it
        float bv = -INFINITY;
        int bj = -1;
#pragma unroll
        for (int j = 0; j < kVpt; ++j)
            if (xs[j] > bv) {
                bv = xs[j];
                bj = j;
            }
        const float wv = warp_max_nonan(bv);
        // ids of a warp run vector-major: the holder with the smallest
        // (vector, lane) has the first id of wv, in its first element equal to it
        const uint32_t code = (bj >= 0 && bv == wv) ? static_cast<uint32_t>(bj * 32 + lane) : 0xFFFFFFFFu;
        const uint32_t wc = __reduce_min_sync(0xFFFFFFFFu, code);
        int wid = -1;
        if (wc != 0xFFFFFFFFu) {
            const int jw = static_cast<int>(wc >> 5), lw = static_cast<int>(wc & 31u);
            if (lane == lw) {
                const uint4 dv = pick(d, jw);
                float z[VEC];
                E::unpack(dv, z);
                if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, jw * kThreads + tid, z);
                int e0 = VEC - 1;
#pragma unroll
                for (int e = VEC - 1; e >= 0; --e)
                    if (z[e] == wv) e0 = e;
                wid = a0 + (jw * kThreads + tid) * VEC + e0;
            }
            wid = __shfl_sync(0xFFFFFFFFu, wid, lw);
        }
        wm = (wid < 0) ? -INFINITY : wv;
        wam = wid;
    }
    if (lane == 0) {
        WarpRecord r;
        r.m = wm;
        r.am = wam;
        r.flags = (wnan ? ARC_ERR_NAN : 0u) | (rerr & (ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP));
        r.pad = 0;
        reinterpret_cast<WarpRecord*>(mysum)[warp] = r;
    }
}

// One slice of one row: the row's parameter words and every 16-byte load of
// the slice are issued first (they depend on nothing); the warps share
// nothing and meet at no barrier (rows with history excepted), and registers
// stay few so that many CTAs per SM keep enough bytes in flight.  The summary
// goes to `mysum` (the workspace, or this CTA's shared memory in the cluster
// kernel).
template <int DT, bool HIST>
__device__ __forceinline__ void scan_cta(const ScanArgs& a, int row, int cidx, ScanShared& sh, unsigned char* dyn,
                                         unsigned char* mysum) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    const int tid = threadIdx.x;
    const int a0 = cidx * a.L;
    const int n = min(a0 + a.L, a.V) - a0;
    const int nv = (n + VEC - 1) / VEC;
    const char* sp = static_cast<const char*>(a.logits) +
                     (static_cast<int64_t>(row) * a.ld + static_cast<int64_t>(a0)) * E::kBytes;
    const uint4 ninf = (DT == ARC_BF16)  ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                       : (DT == ARC_F16) ? make_uint4(0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u, 0xFC00FC00u)
                                         : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
    uint64_t pw[6];
    params_words_nc<HIST>(a.params + row, pw);
    uint4 d[kVpt];
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        const int v = j * kThreads + tid;
        if (a.aligned && (j + 1) * kThreads * VEC <= n)  // the whole round inside the slice
            d[j] = ld_nc_v4(sp + static_cast<size_t>(v) * 16);
        else
            d[j] = (v < nv) ? E::global_vec(sp, v, n, a.aligned) : ninf;
    }
    const ScanRowInfo R = scan_row_info<HIST>(a, row, pw);
    scan_slice<DT, HIST>(a, d, row, cidx, R, sh, dyn, mysum);
}

// One CTA per slice (grid: slices x rows, rows past 65,535 folded into z).
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, HIST ? 4 : 8) scan_kernel(const ScanArgs a) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ ScanShared sh;
    // the finish kernel may be scheduled once every scan CTA is running; it
    // waits (griddepcontrol.wait) for this grid to complete before reading
    // the summaries
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
    const int row = static_cast<int>(blockIdx.z * gridDim.y + blockIdx.y);
    if (row >= a.B) return;  // the whole CTA, before any barrier
    const int cidx = static_cast<int>(blockIdx.x);
    scan_cta<DT, HIST>(a, row, cidx, sh, dyn,
                       const_cast<unsigned char*>(summary_at(a.summaries, a.s, row, cidx)));
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

// Histogram words of floor_hist (256 bins, padded); the caller zeroes them
// before a barrier that precedes the call.
constexpr int kFloorHistWords = 256 + 256 / 8;

// Floor search, one pass: entries binned by (m - x) in steps of 1/8 over the
// 32 logit units below the row max m (256 bins, 32-bit shared atomics), then
// every warp finds the first bin at which the running weight reaches tgt.  The
// floor lies below that bin: every entry counted is at or above it, so the
// bound holds.  False when the window holds less than tgt (the exact
// search below then decides).
template <class KW>
__device__ bool floor_hist(int n, KW kw, float m, uint32_t tgt, uint32_t* hist, float& zf) {
    const int tid = threadIdx.x, lane = tid & 31;
    constexpr int kHB = 256;
    static_assert(kHB + kHB / 8 == kFloorHistWords, "floor histogram size");
    constexpr float kStep = 8.0f;  // bins per logit unit
    // bin b at b + b / 8: a warp reads its lanes' 8-bin runs without bank conflicts
    auto at = [](int b) { return b + (b >> 3); };
    for (int e = tid; e < n; e += kThreads) {
        float x;
        uint32_t w;
        kw(e, x, w);
        const float d = __fmul_rn(__fsub_rn(m, x), kStep);  // >= 0; NaN-free
        if (w != 0u && d < static_cast<float>(kHB)) atomicAdd(&hist[at(static_cast<int>(d))], w);
    }
    __syncthreads();
    // every warp finds the same bin itself (no second barrier)
    {
        uint32_t loc = 0;
#pragma unroll
        for (int q = 0; q < kHB / 32; ++q) loc += hist[at(lane * (kHB / 32) + q)];
        uint32_t inc = loc;
#pragma unroll
        for (int d = 1; d < 32; d <<= 1) {
            const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
            if (lane >= d) inc += o;
        }
        int bin = -1;
        if (inc >= tgt && inc - loc < tgt) {
            uint32_t run = inc - loc;
#pragma unroll
            for (int q = 0; q < kHB / 32; ++q) {
                run += hist[at(lane * (kHB / 32) + q)];
                if (bin < 0 && run >= tgt) bin = lane * (kHB / 32) + q;
            }
        }
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, bin >= 0);
        bin = bal ? __shfl_sync(0xFFFFFFFFu, bin, __ffs(bal) - 1) : -1;
        // entries of bins 0..b satisfy m - x < (b + 1) / 8 up to the rounding of
        // m - x, below 3e-5 of a bin for the 256 bins: a thousandth of a bin
        // of margin, the edge rounded down
        zf = (bin < 0) ? -INFINITY : __fsub_rd(m, (static_cast<float>(bin) + 1.001f) / kStep);
    }
    return zf > -INFINITY;
}

// Floor search by the whole CTA, exact to 2^12 keys: the largest key x whose
// entries at or above it weigh at least tgt in total, two key bits per step
// from the top (three candidate prefixes counted per step, one barrier per
// step).  kw(e, key, weight) gives entry e; the weights' sum must fit in 32
// bits.  False when all entries weigh less than tgt.  The fallback of
// floor_hist: entries are re-read every step rather than held in registers.
template <class KW>
__device__ bool floor_block(int n, KW kw, uint32_t tgt, FinishScratch& SS, uint32_t& edge) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    uint32_t tot = 0;
    for (int e = tid; e < n; e += kThreads) {
        uint32_t key, w;
        kw(e, key, w);
        tot += w;
    }
    tot = __reduce_add_sync(0xFFFFFFFFu, tot);
    if (lane == 0) SS.fc[0][warp][0] = tot;
    __syncthreads();
    uint32_t all = 0;
    for (int v = 0; v < kWarps; ++v) all += SS.fc[0][v][0];
    if (all < tgt) return false;  // uniform
    uint32_t p = 0;
    int par = 1;
#pragma unroll 1
    for (int b = 30; b >= 12; b -= 2, par ^= 1) {
        const uint32_t t1 = p | (1u << b), t2 = p | (2u << b), t3 = p | (3u << b);
        uint32_t c1 = 0, c2 = 0, c3 = 0;
        for (int e = tid; e < n; e += kThreads) {
            uint32_t key, w;
            kw(e, key, w);
            c1 += (key >= t1) ? w : 0u;
            c2 += (key >= t2) ? w : 0u;
            c3 += (key >= t3) ? w : 0u;
        }
        c1 = __reduce_add_sync(0xFFFFFFFFu, c1);
        c2 = __reduce_add_sync(0xFFFFFFFFu, c2);
        c3 = __reduce_add_sync(0xFFFFFFFFu, c3);
        if (lane == 0) {
            SS.fc[par][warp][0] = c1;
            SS.fc[par][warp][1] = c2;
            SS.fc[par][warp][2] = c3;
        }
        __syncthreads();  // (the other parity slot is rewritten only after the next barrier)
        uint32_t s1 = 0, s2 = 0, s3 = 0;
        for (int v = 0; v < kWarps; ++v) {
            s1 += SS.fc[par][v][0];
            s2 += SS.fc[par][v][1];
            s3 += SS.fc[par][v][2];
        }
        p = (s3 >= tgt) ? t3 : ((s2 >= tgt) ? t2 : ((s1 >= tgt) ? t1 : p));
    }
    edge = p;
    return true;
}

// ------------------------------------------------------------------ finish
// First id of the row max m (NaN ignored) for a row whose scan left it open
// (rows without history): the first chunk, in id order, whose max is m,
// re-read by the calling thread alone.  Only error and rounding fallbacks
// need it.
template <int DT>
__device__ __noinline__ int first_max_id(const FinishArgs& a, const char* rowp, const float* cm, int nch, float m) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    const uint32_t km = fkey(m);
    for (int g = 0; g < nch; ++g) {
        if (!(cm[g] > -INFINITY) || fkey(cm[g]) != km) continue;
        const int c = g / kChunks, jr = g % kChunks;
        const int ca0 = c * a.L, cn = min(ca0 + a.L, a.V) - ca0;
        const int v0 = (jr / kWarps) * kThreads + (jr % kWarps) * 32;
        for (int i = v0 * VEC; i < min(cn, (v0 + 32) * VEC); ++i)
            if (E::load_scalar(rowp, ca0 + i) == m) return ca0 + i;
    }
    return 0;
}

// What the steps of one row's finish share, and what they report.
struct RowState {
    float m;         // row max of the penalised logits
    int am;          // its first id (kAmUnknown: not recorded by the scan)
    float cT;        // log2(e) / T
    float scale;     // 2^F: fixed-point unit of a weight
    float zm;        // min-p threshold (z >= zm survives), -inf when off
    bool row_nan, infm;
    uint64_t rbits;  // the row's 53 random bits
    uint64_t S_all;  // chunk tables' total mass (rows that need it)
    uint32_t err;
    uint32_t kap_k, kap_r;
    int iot_k, iot_r;
    uint64_t mass_k, mass_r, target;
    int token, passes;
};

// The selection context of one row held by one CTA, read from global memory.
template <int DT, bool HIST>
__device__ __forceinline__ void setup_row_ctx(RowCtx<DT, HIST>& X, const FinishArgs& a, int row, const char* rowp,
                                              float* cm, const uint32_t* pbm, const uint32_t* pwp, const float* ppat,
                                              bool has_patch, bool row_nan, float m, float c, float scale, bool infm,
                                              unsigned char* dyn, int g = 1, int rank = 0) {
    constexpr int VEC = Elem<DT>::kVec;
    // a cluster of g CTAs splits the row into g parts of whole 32-vector runs
    const int nv_row = (a.V + VEC - 1) / VEC;
    int v0 = 0, v1 = nv_row;
    if (g > 1) {
        const int per = ((nv_row + g - 1) / g + 31) & ~31;
        v0 = min(nv_row, rank * per);
        v1 = min(nv_row, v0 + per);
    }
    X.s = g;
    X.rank = rank;
    X.row = row;
    X.tid = threadIdx.x;
    X.lane = threadIdx.x & 31;
    X.warp = threadIdx.x >> 5;
    X.v0 = v0;
    X.a0 = v0 * VEC;
    X.a1 = min(a.V, v1 * VEC);
    X.n = max(0, X.a1 - X.a0);
    X.nv = v1 - v0;
    X.nvf = X.n / VEC;
    X.rounds = (X.nv + kThreads - 1) / kThreads;
    X.data = reinterpret_cast<const unsigned char*>(rowp) + static_cast<int64_t>(X.a0) * Elem<DT>::kBytes;
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
    X.c = c;
    X.scale = scale;
    X.infm = infm;
}

// Exact selection over the row in global memory by multi-way threshold
// bisection (row_select.cuh), skipping every 32-vector chunk whose max lies
// below a pass's threshold: the path for rows whose floor admits too many
// ids.  Inlined: out of line, the row state, parameters and mode it takes by
// reference would live in local memory for the whole kernel.
template <int DT, bool HIST>
__device__ __forceinline__ void finish_general(const FinishArgs& a, const arc_row_params& P, const RowMode& md, int row,
                                            const char* rowp, float* cm, const uint32_t* pbm, const uint32_t* pwp,
                                            const float* ppat, bool has_patch, KernelShared& KS, unsigned char* dyn,
                                            RowState& st, int g, int rank) {
    using E = Elem<DT>;
    using Ctx = RowCtx<DT, HIST>;
    constexpr int VEC = E::kVec;
    FinishScratch& SS = KS.st;
    const int tid = threadIdx.x;
    const float T = P.temperature;
    const float m = st.m, zm = st.zm;
    __syncthreads();
    cg::cluster_group cl = cg::this_cluster();
    Ctx X(KS.fb, cl);
    setup_row_ctx<DT, HIST>(X, a, row, rowp, cm, pbm, pwp, ppat, has_patch, st.row_nan, m, st.cT, st.scale, st.infm,
                            dyn, g, rank);
    for (int b = tid; b < kBins; b += kThreads) KS.fb.ghist[b] = 0;
    if (tid == 0) {
        KS.fb.ccount = 0;
        KS.fb.flags = 0;
    }
    // every CTA of the row has cleared what the others add into (a cluster
    // barrier when the row is split)
    X.xsync();
    const uint32_t Km = fkey(m);
    uint32_t err = st.err;
    Surv K{-INFINITY, INT_MAX};
    if (md.topk_on) {
        // every chunk max and every second vector max of a chunk is an id at or
        // above itself: the k-th largest of them bounds the k-th largest logit
        // from below and narrows the first histogram window
        float zhint = -INFINITY;
        if (isfinite(m)) {
            const float* cu2 = reinterpret_cast<const float*>(dyn + a.cv2_off);
            const int nch = a.s * kChunks;
            uint32_t* fh = reinterpret_cast<uint32_t*>(KS.fb.lhist);
            for (int b = tid; b < kFloorHistWords; b += kThreads) fh[b] = 0u;
            __syncthreads();
            float zh = -INFINITY;
            floor_hist(2 * nch,
                       [&](int e, float& x, uint32_t& w) {
                           x = e < nch ? cm[e] : cu2[e - nch];
                           w = (x > -INFINITY && x < INFINITY) ? 1u : 0u;
                           if (w == 0u) x = m;
                       },
                       m, static_cast<uint32_t>(P.top_k), fh, zh);
            zhint = zh;
            __syncthreads();
        }
        K = select_topk(X, P.top_k, Km, err, zhint);
        st.kap_k = (K.zt == -INFINITY && K.ge_form()) ? 0u : fkey(K.zt);
        st.iot_k = K.ge_form() ? a.V : K.iota;
    }
    Surv R = K;
    bool wsum_is_R = false;
    if (md.topp_on) {
        // below zb the whole row holds at most (1 - p) / 2 of the top mass
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
        if (md.topk_on) {
            pass_mass<Ctx, true>(X, mk, K, W);
            X.publish_wsum_total(0);
            X.push_hist();
            X.xsync();
            st.mass_k = X.xscan(0, ~0ull).total;
            X.xnext();
        } else {
            // K is every id: its mass is the chunk tables' total
            pass_hist<Ctx, true>(X, W, K);
            X.push_hist();
            X.xsync();
            st.mass_k = st.S_all;
        }
        if (tid == 0) SS.bu[5] = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(st.mass_k)));
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
            wsum_is_R = md.topk_on;  // Wsum holds K's masses only when top-k ran
    } else if (md.minp_on && zm > K.zt) {
        R = Surv{zm, INT_MAX};
    }
    st.kap_r = (R.zt == -INFINITY && R.ge_form()) ? 0u : fkey(R.zt);
    st.iot_r = R.ge_form() ? a.V : R.iota;
    const int mr = mass_mode(X, R);
    if (!wsum_is_R) pass_mass<Ctx, false>(X, mr, R, Window{0u, 0u, 0});
    X.publish_wsum_total(0);
    X.xsync();
    st.mass_r = X.xscan(0, ~0ull).total;
    st.target = scale_by_u(st.rbits, st.mass_r);
    // the CTA whose part holds the target walks it; the others learn the token
    const typename Ctx::Scan sc = X.xscan(0, st.target);
    X.xnext();
    int tok = -1;
    if (sc.first == X.rank)
        tok = X.walk(
            st.target - sc.before_me, [&](const float(&z)[VEC], int g0) { return X.vec_mass(mr, z, g0, R); },
            [&](const float(&z)[VEC], int g0, uint64_t tt) { return X.vec_mass_walk(mr, z, g0, R, tt); });
    if (X.s > 1) {
        if (tid == 0) X.S.slot[X.par][0] = static_cast<uint64_t>(static_cast<uint32_t>(tok));
        X.xsync();
        tok = sc.first >= 0 ? static_cast<int>(static_cast<uint32_t>(X.xread(sc.first, 0))) : -1;
        X.xnext();
        X.xsync();  // no CTA leaves while another may still read its shared memory
    }
    if (tok < 0) {
        tok = st.am != kAmUnknown ? st.am : first_max_id<DT>(a, rowp, cm, a.s * kChunks, m);
        err |= kErrInternal;
    }
    st.token = tok;
    st.passes = 1 + X.passes;
    st.err = err;
}

// Top-n log-probabilities of one row (a.top_n > 0), after its token: the n
// ids first in (z desc, id asc) order of the penalised logits and their
// log-softmax at the row's temperature (1 for a greedy row).  The ids come
// from the direct selection's floor (the n-th largest chunk max) and gather;
// a row whose floor admits more ids than the selection holds takes the exact
// top-k bisection with k = n.  ln(S) is the fp64 log of the chunk tables'
// fixed-point total at the same temperature.
template <int DT, bool HIST>
__device__ __noinline__ void top_n_row(const FinishArgs& a, int row, const arc_row_params& P, bool valid,
                                      const char* rowp, float m, bool row_nan, float cT, float scale, bool want_mv,
                                      int hbeg, int hn, KernelShared& KS, unsigned char* dyn) {
    using E = Elem<DT>;
    using Ctx = RowCtx<DT, HIST>;
    constexpr int VEC = E::kVec;
    FinishScratch& SS = KS.st;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int n = a.top_n;
    arc_top_logprob* out = a.top_logprobs + static_cast<size_t>(row) * n;
    const int nch = a.s * kChunks;
    float* cm = reinterpret_cast<float*>(dyn + a.cmax_off);
    const float* cs = reinterpret_cast<const float*>(dyn + a.cs_off);
    const int* cln = reinterpret_cast<const int*>(dyn + a.cid_off);
    const float* cu2 = reinterpret_cast<const float*>(dyn + a.cv2_off);
    const uint4* cmv = reinterpret_cast<const uint4*>(dyn + a.cmv_off);
    __syncthreads();  // the row's selection is done with the shared scratch
    if (!valid || !(m > -INFINITY)) {
        // invalid parameters: (-1, -inf); no finite or +inf logit: every id
        // ties at -inf, listed in id order
        for (int j = tid; j < n; j += kThreads) out[j] = arc_top_logprob{(valid && j < a.V) ? j : -1, -INFINITY};
        return;
    }
    const bool infm = m == INFINITY;
    const float Tm = P.temperature > 0.0f ? P.temperature : 1.0f;
    // the total mass: chunk masses rescaled to the row max, in units of 2^-F
    {
        const int cper = (nch + kThreads - 1) / kThreads;
        uint64_t loc = 0;
        for (int e = tid * cper; e < min(nch, tid * cper + cper); ++e) {
            const float mj = cm[e], Sj = cs[e];
            if (mj != -INFINITY && Sj != 0.0f) loc += __float2ull_rn(__fmul_rn(__fmul_rn(Sj, wrel(mj, m, cT)), scale));
        }
        const uint64_t tot = block_sum_u64(loc, SS.redu);
        if (tid == 0) SS.bd[0] = log(static_cast<double>(tot)) - static_cast<double>(a.F) * 0.69314718055994530942;
    }
    // history patches of the whole row
    const uint32_t* pbm = nullptr;
    const uint32_t* pwp = nullptr;
    const float* ppat = nullptr;
    bool has_patch = false;
    if (HIST && hn > 0) {
        const int nwords_max = (a.fb_rounds * kThreads * VEC + 31) / 32;
        uint32_t* bm = reinterpret_cast<uint32_t*>(dyn + a.fb_patch_off);
        uint32_t* wp = bm + nwords_max;
        uint32_t* cnt = wp + (nwords_max + 1) / 2;
        float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
        __syncthreads();
        if (tid == 0) SS.bi[7] = 0;
        const int distinct = build_patches<DT>(rowp, a.V, 0, a.V, (a.V + VEC - 1) / VEC, P, a.hist_ids + hbeg, hn, bm,
                                               wp, cnt, pat, SS.red32, reinterpret_cast<uint32_t*>(&SS.bi[7]));
        pbm = bm;
        pwp = wp;
        ppat = pat;
        has_patch = distinct > 0;
    }
    uint64_t* cc = reinterpret_cast<uint64_t*>(dyn + a.cand_off);
    for (int b = tid; b < kFloorHistWords; b += kThreads) reinterpret_cast<uint32_t*>(KS.fb.lhist)[b] = 0u;
    if (tid == 0) SS.ccount = 0;
    __syncthreads();
    // floor: the n-th largest chunk max (every chunk max is an id at or above it)
    float zf = -INFINITY;
    bool fast = false;
    if (!infm) {
        auto wt = [&](float x) -> uint32_t { return x > -INFINITY ? 1u : 0u; };
        fast = floor_hist(nch, [&](int e, float& x, uint32_t& w) { x = cm[e]; w = wt(x); }, m,
                          static_cast<uint32_t>(n), reinterpret_cast<uint32_t*>(KS.fb.lhist), zf);
        if (!fast) {
            uint32_t edge = 0;
            fast = floor_block(nch, [&](int e, uint32_t& key, uint32_t& w) { key = fkey(cm[e]); w = wt(cm[e]); },
                               static_cast<uint32_t>(n), SS, edge);
            if (fast) zf = Ctx::lo_float(edge);
        }
        fast = fast && zf > -INFINITY;
    }
    auto emit = [&](const float (&z)[VEC], int vrow, float thr) {
        int cnt = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) cnt += (z[e] >= thr) ? 1 : 0;
        if (cnt > 0) {
            uint32_t pos = atomicAdd(&SS.ccount, static_cast<uint32_t>(cnt));
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if (z[e] >= thr) {
                    if (pos < static_cast<uint32_t>(kCandCap))
                        cc[pos] = (static_cast<uint64_t>(fkey(z[e])) << 32) |
                                  (0xFFFFFFFFu - static_cast<uint32_t>(vrow * VEC + e));
                    ++pos;
                }
            }
        }
    };
    if (fast) {
        // ids >= zf from the chunks whose max reaches it: one vector (the max's)
        // when the other vectors lie below zf, else all 32, one per lane
        const int Lv = a.L / VEC;
        const int wcap = (nch + kWarps - 1) / kWarps;
        for (int g = warp * wcap; g < min(nch, warp * wcap + wcap); ++g) {
            if (!(cm[g] >= zf)) continue;  // (warp-uniform)
            const int c = g / kChunks;
            const int sn = min((c + 1) * a.L, a.V) - c * a.L;
            const char* sb = rowp + static_cast<int64_t>(c) * a.L * E::kBytes;
            const bool single = cu2[g] < zf && cln[g] >= 0;
            const int vs = (g % kChunks) * 32 + (single ? cln[g] : lane);
            if (single && lane != 0) continue;
            float z[VEC];
            if (vs * VEC < sn) {
                E::unpack(single && want_mv ? cmv[g] : E::global_vec(sb, vs, sn, a.aligned), z);
                if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, c * Lv + vs, z);
                emit(z, c * Lv + vs, zf);
            }
        }
        __syncthreads();
        fast = SS.ccount <= static_cast<uint32_t>(kCandCap);
    }
    if (!fast) {
        // exact: the top-k set for k = n by threshold bisection, then its ids
        __syncthreads();
        cg::cluster_group cl = cg::this_cluster();
        Ctx X(KS.fb, cl);
        setup_row_ctx<DT, HIST>(X, a, row, rowp, cm, pbm, pwp, ppat, has_patch, row_nan, m, cT, scale, infm, dyn);
        for (int b = tid; b < kBins; b += kThreads) KS.fb.ghist[b] = 0;
        if (tid == 0) {
            KS.fb.ccount = 0;
            KS.fb.flags = 0;
            SS.ccount = 0;
        }
        __syncthreads();
        uint32_t err = 0;
        const Surv K = select_topk(X, n, fkey(m), err);
        __syncthreads();
        X.batched_pass([&](int v) { return X.may_hold(v, K.zt); },
                       [&](int, int v, const float(&z)[VEC]) {
                           float zk[VEC];
#pragma unroll
                           for (int e = 0; e < VEC; ++e)  // (the row's tail vector pads past V with -inf)
                               zk[e] = (v * VEC + e < a.V && K.test(z[e], v * VEC + e)) ? z[e] : NAN;
                           emit(zk, v, -INFINITY);
                       },
                       [](int) {});
        __syncthreads();
    }
    // rank by (key desc, id asc); the first n are written, the rest padded
    const int nc = min(static_cast<int>(SS.ccount), kCandCap);
    const double lnS = SS.bd[0];
    for (int i = tid; i < nc; i += kThreads) {
        const uint64_t vi = cc[i];
        int rk = 0;
#pragma unroll 8
        for (int j = 0; j < nc; ++j) rk += (cc[j] > vi) ? 1 : 0;
        if (rk < n) {
            const float z = key_to_float(static_cast<uint32_t>(vi >> 32));
            const int id = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(vi));
            float lp;
            if (infm)
                lp = z == INFINITY ? static_cast<float>(-lnS) : -INFINITY;
            else if (z == -INFINITY)
                lp = -INFINITY;
            else
                lp = static_cast<float>((static_cast<double>(z) - static_cast<double>(m)) / static_cast<double>(Tm) - lnS);
            out[rk] = arc_top_logprob{id, lp};
        }
    }
    for (int j = nc + tid; j < n; j += kThreads) out[j] = arc_top_logprob{-1, -INFINITY};
}

// The direct selection after the ranking, over the candidates in sorted order
// (sk, sid, sm: keys, ids, fixed-point masses): K = the first nk, the top-p
// cutoff, min-p, the survivors' mass and the draw in id order.  Thread t holds
// sorted positions [POS t, POS t + POS): POS = 4 covers 1,024 candidates, 8
// covers 2,048 (kept apart, so that the common case carries no extra work).
// Bitonic sort of v[0, n2) (n2 a power of two), descending, by the whole
// CTA, v[nc, n2) padded with zeros first.  Out of line: the counting rank of
// few candidates keeps its registers.
static __device__ __noinline__ void bitonic_desc(uint64_t* v, int nc, int n2) {
    const int tid = threadIdx.x;
    for (int i = nc + tid; i < n2; i += kThreads) v[i] = 0;
    __syncthreads();
    for (int size = 2; size <= n2; size <<= 1) {
        for (int ls = __ffs(size) - 2; ls >= 0; --ls) {  // stride 2^ls
            const int stride = 1 << ls;
            for (int i = tid; i < (n2 >> 1); i += kThreads) {
                const int lo = ((i >> ls) << (ls + 1)) | (i & (stride - 1)), hi = lo + stride;
                const uint64_t x = v[lo], y = v[hi];
                if ((x < y) == ((lo & size) == 0)) {  // descending where lo & size == 0
                    v[lo] = y;
                    v[hi] = x;
                }
            }
            __syncthreads();
        }
    }
}

// The draw over many survivors in id order (sorted_select): their masses by
// id range (kThreads ranges in id order, each bin's 64-bit sum as two 32-bit
// words with exact carry), the range holding the target, then that range's
// survivors in id order.  Out of line: the common few-survivor draw keeps its
// registers.
static __device__ __noinline__ void draw_by_id_range(const FinishArgs& a, uint64_t target, FinishScratch& SS,
                                                     const int* sid, const uint64_t* sm, int nsv, uint32_t* bins,
                                                     uint32_t* scratch) {
    const int tid = threadIdx.x;
    auto range_of = [&](int id) {
        return static_cast<int>((static_cast<uint64_t>(id) * kThreads) / static_cast<uint64_t>(a.V));
    };
    bins[2 * tid] = 0u;
    bins[2 * tid + 1] = 0u;
    if (tid == 0) SS.draw_n = 0;
    __syncthreads();
    for (int pp = tid; pp < nsv; pp += kThreads) {
        const uint64_t mp = sm[pp];
        uint32_t* h = &bins[2 * range_of(sid[pp])];
        const uint32_t lo = static_cast<uint32_t>(mp), hi = static_cast<uint32_t>(mp >> 32);
        const uint32_t old = atomicAdd(h, lo);
        const uint32_t carry = (old + lo < old) ? 1u : 0u;
        if (hi + carry) atomicAdd(h + 1, hi + carry);
    }
    __syncthreads();
    const uint64_t mine = (static_cast<uint64_t>(bins[2 * tid + 1]) << 32) | bins[2 * tid];
    uint64_t tot_r;
    const uint64_t inc = block_scan_u64(mine, SS.redu, tot_r);
    if (tid == 0) SS.draw_bin = -1;
    __syncthreads();
    if (mine != 0 && inc - mine <= target && target < inc) {
        SS.draw_bin = tid;
        SS.draw_base = inc - mine;
    }
    __syncthreads();
    const int rb = SS.draw_bin;
    const uint64_t base = SS.draw_base;
    // the range's survivors by sorted position (at most nsv <= 2,048)
    for (int pp = tid; pp < nsv; pp += kThreads) {
        if (range_of(sid[pp]) == rb) scratch[atomicAdd(&SS.draw_n, 1u)] = static_cast<uint32_t>(pp);
    }
    __syncthreads();
    const int nr = static_cast<int>(SS.draw_n);
    for (int i = tid; i < nr; i += kThreads) {
        const int ip = sid[scratch[i]];
        const uint64_t mp = sm[scratch[i]];
        uint64_t before = base;
        for (int j = 0; j < nr; ++j) before += (sid[scratch[j]] < ip) ? sm[scratch[j]] : 0u;
        if (mp != 0 && before <= target && target < before + mp) SS.bi[6] = ip;
    }
}

template <int POS>
__device__ __forceinline__ void sorted_select(const FinishArgs& a, const arc_row_params& P, const RowMode& md,
                                              RowState& st, FinishScratch& SS, const uint32_t* sk, const int* sid,
                                              const uint64_t* sm, int nk, float zm, const Surv& K, uint32_t* bins,
                                                     uint32_t* scratch) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
        // thread t holds sorted positions [POS t, POS t + POS), read once as
        // 16-byte vectors (kCandCap = POS kThreads: always inside the arrays)
        static_assert(POS % 4 == 0 && POS * kThreads <= kCandCap, "sorted positions per thread");
        const int p0 = POS * tid;
        uint32_t tk[POS];
        int ti[POS];
        uint64_t tm[POS];
#pragma unroll
        for (int h = 0; h < POS / 4; ++h) {
            const uint4 kv = reinterpret_cast<const uint4*>(sk)[(POS / 4) * tid + h];
            const int4 iv = reinterpret_cast<const int4*>(sid)[(POS / 4) * tid + h];
            const ulonglong2 m0 = reinterpret_cast<const ulonglong2*>(sm)[(POS / 2) * tid + 2 * h];
            const ulonglong2 m1 = reinterpret_cast<const ulonglong2*>(sm)[(POS / 2) * tid + 2 * h + 1];
            tk[4 * h] = kv.x, tk[4 * h + 1] = kv.y, tk[4 * h + 2] = kv.z, tk[4 * h + 3] = kv.w;
            ti[4 * h] = iv.x, ti[4 * h + 1] = iv.y, ti[4 * h + 2] = iv.z, ti[4 * h + 3] = iv.w;
            tm[4 * h] = m0.x, tm[4 * h + 1] = m0.y, tm[4 * h + 2] = m1.x, tm[4 * h + 3] = m1.y;
        }
        uint64_t lk = 0;
#pragma unroll
        for (int q = 0; q < POS; ++q) lk += (p0 + q < nk) ? tm[q] : 0u;
        uint64_t tot_k;
        // (the barrier after the ranking follows every earlier use of SS.redu)
        const uint64_t inc_k = block_scan_u64(lk, SS.redu, tot_k, /*fresh=*/true);
        st.mass_k = md.topk_on ? tot_k : st.S_all;
        bool found = false;
        float zp = -INFINITY;
        if (md.topp_on) {
            // first sorted position whose running mass reaches ceil(p * mass_k)
            if (tid == 0)
                SS.bu[5] = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(st.mass_k)));
            __syncthreads();
            const uint64_t tgt = max(SS.bu[5], uint64_t{1});
            uint64_t run = inc_k - lk;
            if (run < tgt && inc_k >= tgt) {
#pragma unroll
                for (int q = 0; q < POS; ++q) {
                    const uint64_t mq = (p0 + q < nk) ? tm[q] : 0u;
                    if (mq != 0 && run < tgt && run + mq >= tgt) SS.bi[5] = p0 + q;
                    run += mq;
                }
            }
            __syncthreads();
            if (SS.bi[5] >= 0) {
                found = true;
                zp = key_to_float(sk[SS.bi[5]]);
            }
            if (!found && !md.minp_on && !md.topk_on) st.err |= kErrInternal;  // the floor guarantees it
        }
        const float zx = found ? fmaxf(zp, zm) : zm;
        const Surv R = (zx > K.zt) ? Surv{zx, INT_MAX} : K;
        st.kap_r = (R.zt == -INFINITY && R.ge_form()) ? 0u : fkey(R.zt);
        st.iot_r = R.ge_form() ? a.V : R.iota;
        // survivors: a prefix [0, ns) of the sorted order
        int nsv = nk;
        if (!(zx > K.zt)) {
            // R is K: its positions are [0, nk) and its mass the scan's total
            st.mass_r = tot_k;
        } else {
            // the survivors' mass and their count, in one reduction
            uint64_t lr = 0;
            int first_out = nk;
#pragma unroll
            for (int q = POS - 1; q >= 0; --q) {
                const int pp = p0 + q;
                if (pp < nk) {
                    if (R.test(key_to_float(tk[q]), ti[q]))
                        lr += tm[q];
                    else
                        first_out = pp;
                }
            }
            lr = warp_sum_u64(lr);
            first_out = static_cast<int>(__reduce_min_sync(0xFFFFFFFFu, static_cast<unsigned>(first_out)));
            if (lane == 0) {
                SS.fc[1][warp][0] = static_cast<uint32_t>(lr);
                SS.fc[1][warp][1] = static_cast<uint32_t>(lr >> 32);
                SS.fc[1][warp][2] = static_cast<uint32_t>(first_out);
            }
            __syncthreads();
            uint64_t mr = 0;
            for (int v = 0; v < kWarps; ++v) {
                mr += (static_cast<uint64_t>(SS.fc[1][v][1]) << 32) | SS.fc[1][v][0];
                nsv = min(nsv, static_cast<int>(SS.fc[1][v][2]));
            }
            st.mass_r = mr;
        }
        st.target = scale_by_u(st.rbits, st.mass_r);
        if (nsv <= kRankMax) {
            // the draw in id order: each survivor sums the survivors with smaller ids
            for (int pp = tid; pp < nsv; pp += kThreads) {
                const int ip = sid[pp];
                const uint64_t mp = sm[pp];
                uint64_t before = 0;
#pragma unroll 8
                for (int qq = 0; qq < nsv; ++qq) before += (sid[qq] < ip) ? sm[qq] : 0u;
                if (mp != 0 && before <= st.target && st.target < before + mp) SS.bi[6] = ip;
            }
        } else {
            draw_by_id_range(a, st.target, SS, sid, sm, nsv, bins, scratch);
        }
}

// One row's finish by one CTA.  sum_at(c) is slice c's summary (the
// workspace, or another CTA's shared memory in the cluster kernel); wait()
// returns once every summary of the row is complete and visible; loaded()
// runs after the summaries have been copied on chip (every thread of the CTA
// calls both).
// The decode-loop commit of this CTA's row as record head[0] + row (the
// commit of arc_decode.h, one row per CTA), in two parts.  commit_arrive, in
// the prologue: read head[0] (and the row's position and owner), then arrive
// on head[1] with an acquire-release
// atomic; the CTA that arrives last has seen every other arrival, hence every
// read of head[0], so it advances head[0] by B and leaves head[1] at 0 for the
// next call.  commit_publish, after the token: the row's checks, writes and
// record (no fence, no atomic but the fault bits).
__device__ __forceinline__ void commit_arrive(const FinishArgs& a, int row, FinishScratch& SS) {
    unsigned long long* head = reinterpret_cast<unsigned long long*>(a.commit.head);
    unsigned long long h, n;
    // the row's position and owner tag load with the head (no kernel of the
    // call writes them before the commit)
    SS.cpos = a.commit.positions[row];
    SS.cown = a.commit.owners ? a.commit.owners[row] : 0u;
    asm volatile("ld.relaxed.gpu.global.u64 %0, [%1];" : "=l"(h) : "l"(head) : "memory");
    asm volatile("atom.acq_rel.gpu.global.add.u64 %0, [%1], 1;" : "=l"(n) : "l"(head + 1) : "memory");
    if (n == static_cast<unsigned long long>(a.B) - 1ull) {
        asm volatile("st.relaxed.gpu.global.u64 [%0], 0;" ::"l"(head + 1) : "memory");
        asm volatile("st.relaxed.gpu.global.u64 [%0], %1;" ::"l"(head), "l"(h + static_cast<unsigned long long>(a.B))
                     : "memory");
    }
    SS.chead = h;
}
__device__ __forceinline__ void commit_publish(const FinishArgs& a, int row, int32_t tok, const FinishScratch& SS) {
    const arc_commit_target& c = a.commit;
    const uint32_t bad = commit_row_read(tok, SS.cpos, SS.cown, row, SS.chead + static_cast<unsigned long long>(row),
                                         a.V, c.next_ids, c.positions, c.max_position, c.ring, c.capacity);
    if (bad != 0 && c.fault_word != nullptr) atomicOr(c.fault_word, bad);
}

template <int DT, bool HIST, class SumAt, class Wait, class Loaded>
__device__ __forceinline__ void finish_row(const FinishArgs& a, int row, KernelShared& KS, unsigned char* dyn,
                                           SumAt sum_at, Wait wait, Loaded loaded, int g, int rank) {
    using E = Elem<DT>;
    using Ctx = RowCtx<DT, HIST>;
    constexpr int VEC = E::kVec;
    FinishScratch& SS = KS.st;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int s = a.s;
    const int nch = s * kChunks;
    const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;
    float* cm = reinterpret_cast<float*>(dyn + a.cmax_off);
    float* cs = reinterpret_cast<float*>(dyn + a.cs_off);
    int* cln = reinterpret_cast<int*>(dyn + a.cid_off);
    float* cu2 = reinterpret_cast<float*>(dyn + a.cv2_off);
    // plain loads, issued before the wait below: only this CTA writes its
    // row's record (`step`, at the very end)
    uint64_t pw[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) pw[i] = reinterpret_cast<const uint64_t*>(a.params + row)[i];
    const arc_row_params P = params_from_words(pw);
    int hn = 0, hbeg = 0;
    if (HIST && a.hist_off != nullptr) {
        hbeg = a.hist_off[row];
        hn = max(0, a.hist_off[row + 1] - hbeg);
    }
    // min-p: T ln(min_p) in fp64 (slow on this part), by the thread that uses
    // it, while the scan still runs
    double tl = 0.0;
    if (tid == 0 && P.min_p > 0.0f && P.min_p <= 1.0f && isfinite(P.temperature) && P.temperature > 0.0f &&
        !(P.top_k == 1))
        tl = static_cast<double>(P.temperature) * log(static_cast<double>(P.min_p));
    // the finish needs the chunk max vectors (filtered rows)
    const bool want_mv = a.cmv_off >= 0 && param_errors(P) == 0 && (RowMode(P, a.V).filtered || a.top_n > 0);
    // a top-k row with a large k: the wide entries too
    const bool want_wide = a.cwide_off >= 0 && param_errors(P) == 0 && RowMode(P, a.V).filtered &&
                           P.top_k > kWideK && P.top_k < a.V;
    // the decode-loop commit's ring index: read (and the head advanced) while
    // the scan still runs; the head is no kernel's but the commit's
    const bool leader = rank == 0;  // the CTA that writes the row's results
    if (a.commit.ring != nullptr && leader && tid == 0) commit_arrive(a, row, SS);
    // the summaries are complete and visible after this (the parameters and
    // history above are not written by the scan)
    wait();

    // the warp records (warp 0) and the chunk tables (warps 1-7) load while
    // the parameters do: nothing here waits for them
    if (warp == 0) {
        float v = -INFINITY;
        int i = -1;
        uint32_t f = 0;
        const int nrec = s * kWarps;
        auto rec = [&](int q) {
            return reinterpret_cast<const WarpRecord*>(sum_at(q / kWarps))[q % kWarps];
        };
        constexpr int kLdR = 4;  // records in flight per lane
        WarpRecord r[kLdR];
#pragma unroll
        for (int u = 0; u < kLdR; ++u)
            if (lane + 32 * u < nrec) r[u] = rec(lane + 32 * u);
#pragma unroll
        for (int u = 0; u < kLdR; ++u) {
            if (lane + 32 * u < nrec) {
                better(v, i, r[u].m, r[u].am);
                f |= r[u].flags;
            }
        }
        for (int q = lane + 32 * kLdR; q < nrec; q += 32) {
            const WarpRecord x = rec(q);
            better(v, i, x.m, x.am);
            f |= x.flags;
        }
        warp_argmax(v, i);
        f = __reduce_or_sync(0xFFFFFFFFu, f);
        if (lane == 0) {
            SS.bf[0] = v;
            SS.bi[0] = i;
            SS.bi[1] = static_cast<int>(f);
            // min-p: the smallest float z with z - m >= T ln(min_p)
            SS.bf[1] = __double2float_ru(static_cast<double>(v) + tl);
        }
    } else {
        constexpr int kLd = 4;  // chunk entries in flight per thread
        constexpr int kStride = kThreads - 32;
        for (int g0 = tid - 32; g0 < nch; g0 += kLd * kStride) {
            ChunkEntry e[kLd];
            uint4 mv[kLd];
            WideEntry we[kLd];
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int gi = g0 + u * kStride;
                if (gi < nch) {
                    const unsigned char* sm = sum_at(gi / kChunks);
                    e[u] = chunk_table(sm)[gi % kChunks];
                    if (want_mv) mv[u] = max_vectors(sm)[gi % kChunks];
                    if (want_wide) we[u] = wide_entries(sm)[gi % kChunks];
                }
            }
#pragma unroll
            for (int u = 0; u < kLd; ++u) {
                const int gi = g0 + u * kStride;
                if (gi < nch) {
                    cm[gi] = e[u].m;
                    cs[gi] = e[u].S;
                    cln[gi] = e[u].lane;
                    cu2[gi] = e[u].u2;
                    if (want_mv) reinterpret_cast<uint4*>(dyn + a.cmv_off)[gi] = mv[u];
                    if (want_wide) reinterpret_cast<WideEntry*>(dyn + a.cwide_off)[gi] = we[u];
                }
            }
        }
    }
    // the floor histogram and the candidate counter start at zero (filtered
    // rows), cleared while the summaries load
    for (int b = tid; b < kFloorHistWords; b += kThreads) reinterpret_cast<uint32_t*>(KS.fb.lhist)[b] = 0u;
    if (tid == 0) {
        SS.ccount = 0;  // candidates gathered (filtered rows)
        SS.nwhole = 0;
    }
    uint32_t rerr = param_errors(P);
    const RowMode md(P, a.V);
    const float T = P.temperature;
    const int k = P.top_k;
    __syncthreads();
    loaded();

    RowState st;
    st.m = SS.bf[0];
    st.am = SS.bi[0];
    const uint32_t rflags = static_cast<uint32_t>(SS.bi[1]);
    st.row_nan = (rflags & ARC_ERR_NAN) != 0;
    st.cT = (md.greedy && a.top_n == 0) ? 0.0f : __fdiv_rn(1.4426950408889634f, T > 0.0f ? T : 1.0f);
    st.scale = __uint_as_float(static_cast<uint32_t>(127 + a.F) << 23);
    st.infm = (st.m == INFINITY);
    st.zm = md.minp_on ? SS.bf[1] : -INFINITY;
    st.rbits = 0;
    st.S_all = 0;
    st.kap_k = st.kap_r = 0;
    st.iot_k = st.iot_r = a.V;
    st.mass_k = st.mass_r = st.target = 0;
    st.passes = 1;
    rerr |= rflags & (ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP | ARC_ERR_TIMEOUT);
    st.err = rerr | (rflags & ARC_ERR_NAN);
    int mode;
    st.token = -2;
    if (rerr != 0) {
        mode = -1;
        st.token = -1;
    } else {
        mode = md.greedy ? 0 : (md.filtered ? 2 : 1);
        if (st.am < 0) {
            st.token = 0;
            st.err |= ARC_ERR_DEGENERATE;
        } else if (md.greedy) {
            st.token = st.am;
        }
    }
    const float m = st.m, cT = st.cT;
    // the row max's first id where a fallback needs it
    auto max_id = [&]() { return st.am != kAmUnknown ? st.am : first_max_id<DT>(a, rowp, cm, nch, m); };
    auto fixq = [&](float w) { return __float2ull_rn(__fmul_rn(w, st.scale)); };
    // a chunk's fixed-point mass, rescaled from its own max to the row max
    auto chunk_q = [&](int e) -> uint64_t {
        const float mj = cm[e], Sj = cs[e];
        if (mj == -INFINITY || Sj == 0.0f) return 0;
        return fixq(__fmul_rn(Sj, wrel(mj, m, cT)));
    };
    const int cper = (nch + kThreads - 1) / kThreads;  // chunk entries per thread, in id order
    const int ce0 = min(nch, tid * cper), ce1 = min(nch, ce0 + cper);

    if (st.token == -2) {
        st.rbits = splitmix64(P.seed ^ (static_cast<uint64_t>(row) << 32) ^ P.step) >> 11;
        if (mode == 1) {
            // ---------------------------------------------------------- default rows
            // total mass and the chunk that holds the draw, in one block scan
            uint64_t loc = 0;
            for (int e = ce0; e < ce1; ++e) loc += chunk_q(e);
            if (tid == 0) SS.bi[2] = -1;
            uint64_t total;
            const uint64_t incl = block_scan_u64(loc, SS.redu, total);
            st.mass_r = total;
            st.target = scale_by_u(st.rbits, total);
            const uint64_t before = incl - loc;
            if (before <= st.target && st.target < incl) {
                uint64_t run = before;
                for (int e = ce0; e < ce1; ++e) {
                    const uint64_t q = chunk_q(e);
                    if (q > 0 && run + q > st.target) {
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
                st.err |= kErrInternal;
                st.token = max_id();
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
                uint64_t tres = st.target - hit_before;
                int token = -3;  // no lane carries mass: take the row's first max below
                if (Q != 0) {
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
            if (hit >= 0) st.token = SS.bi[3];
            if (st.token == -3) st.token = max_id();
        } else {
            // ---------------------------------------------------------- filtered rows
            const float zm = st.zm;
            if (md.need_mass) {  // top-p over every id: the chunk tables' total mass
                uint64_t loc = 0;
                for (int e = ce0; e < ce1; ++e) loc += chunk_q(e);
                st.S_all = block_sum_u64(loc, SS.redu);
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
                uint32_t* cnt = wp + (nwords_max + 1) / 2;
                float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
                __syncthreads();
                if (tid == 0) SS.bi[7] = 0;
                const int nv_row = (a.V + VEC - 1) / VEC;
                const int distinct = build_patches<DT>(rowp, a.V, 0, a.V, nv_row, P, a.hist_ids + hbeg, hn, bm, wp,
                                                       cnt, pat, SS.red32, reinterpret_cast<uint32_t*>(&SS.bi[7]));
                pbm = bm;
                pwp = wp;
                ppat = pat;
                has_patch = distinct > 0;
            }

            // floor zf: every survivor has z >= zf
            float zf = -INFINITY;
            bool fast = true;
            if (md.topk_on || !md.minp_on) {
                uint32_t tgt;
                int sh = 0;
                if (md.topk_on) {
                    // every chunk holds an id >= its max, so k chunk maxima >= x put
                    // the k-th largest logit at or above x
                    tgt = static_cast<uint32_t>(k);
                } else {
                    // top-p alone: the chunk maxima at or above x already carry at
                    // least the target mass (masses in units of 2^sh rounded down,
                    // the target rounded up: the bound holds and sums fit in 32 bits)
                    if (tid == 0)
                        SS.bu[5] = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(st.S_all)));
                    __syncthreads();
                    const uint64_t t64 = max(SS.bu[5], uint64_t{1});
                    sh = max(0, a.F - 19);
                    tgt = static_cast<uint32_t>((t64 + (uint64_t{1} << sh) - 1) >> sh);
                }
                auto wt = [&](float x) -> uint32_t {
                    return !(x > -INFINITY) ? 0u
                                            : (md.topk_on ? 1u : static_cast<uint32_t>(fixq(wrel(x, m, cT)) >> sh));
                };
                // wide top-k rows: the four largest vector maxima of every chunk
                // (distinct ids), so that a k beyond the chunk count still has a floor
                const int nv_floor = want_wide ? 4 * nch : nch;
                const WideEntry* cw = reinterpret_cast<const WideEntry*>(dyn + a.cwide_off);
                auto val = [&](int e) -> float {
                    if (e < nch) return cm[e];
                    if (e < 2 * nch) return cu2[e - nch];
                    return e < 3 * nch ? cw[e - 2 * nch].u3 : cw[e - 3 * nch].u4;
                };
                fast = isfinite(m) &&
                       floor_hist(nv_floor,
                                  [&](int e, float& x, uint32_t& w) {
                                      x = val(e);
                                      w = (x < INFINITY) ? wt(x) : 0u;
                                      if (w == 0u) x = m;
                                  },
                                  m, tgt, reinterpret_cast<uint32_t*>(KS.fb.lhist), zf);
                if (!fast) {
                    auto kw = [&](int e, uint32_t& key, uint32_t& w) {
                        const float x = val(e);
                        key = fkey(x < INFINITY ? x : -INFINITY);
                        w = (x < INFINITY) ? wt(x) : 0u;
                    };
                    uint32_t edge = 0;
                    fast = floor_block(nv_floor, kw, tgt, SS, edge);
                    if (fast) zf = Ctx::lo_float(edge);
                }
            } else {
                zf = zm;
            }
            // (the candidate counter was cleared with the summaries)
            fast = fast && zf > -INFINITY && !(a.flags & ARC_OPT_FORCE_BISECTION);

            // gather the ids >= zf as (key, id): every thread takes a contiguous run
            // of chunk entries; a chunk whose other vectors lie below zf ("single")
            // gives the ids of its max's vector, taken from the summary, and any
            // other chunk at or above zf is listed; after one barrier the warps read
            // the listed chunks from the logits, 32 vectors (one per lane) each
            // candidates as one 64-bit value: key << 32 | (2^32 - 1 - id), so
            // that a larger value ranks first by (z desc, id asc)
            uint64_t* cc = reinterpret_cast<uint64_t*>(dyn + a.cand_off);
            auto weight_of = [&](float z) -> float {
                return st.infm ? (z == m ? 1.0f : 0.0f) : ex2(__fmul_rn(__fsub_rn(z, m), cT));
            };
            int nc = 0;
            if (fast) {
                const int Lv = a.L / VEC;
                int* whole = reinterpret_cast<int*>(dyn + a.clist_off);  // listed chunks
                // the ids of a vector >= zf take slots from one shared counter
                auto emit = [&](const float (&z)[VEC], int vrow) {
                    int cnt = 0;
#pragma unroll
                    for (int e = 0; e < VEC; ++e) cnt += (z[e] >= zf) ? 1 : 0;
                    if (cnt > 0) {
                        uint32_t pos = atomicAdd(&SS.ccount, static_cast<uint32_t>(cnt));
#pragma unroll
                        for (int e = 0; e < VEC; ++e) {
                            if (z[e] >= zf) {
                                if (pos < static_cast<uint32_t>(kCandCap))
                                    cc[pos] = (static_cast<uint64_t>(fkey(z[e])) << 32) |
                                              (0xFFFFFFFFu - static_cast<uint32_t>(vrow * VEC + e));
                                ++pos;
                            }
                        }
                    }
                };
                const WideEntry* cw = reinterpret_cast<const WideEntry*>(dyn + a.cwide_off);
                for (int g = ce0; g < ce1; ++g) {
                    if (!(cm[g] >= zf)) continue;
                    const int c = g / kChunks;
                    if (want_wide && cu2[g] >= zf && cw[g].u4 < zf && cln[g] >= 0) {
                        // at most three vectors hold ids >= zf: the max's (from the
                        // summary), the second's and, when its max reaches zf, the third's
                        const WideEntry wg = cw[g];
                        const int sn = min((c + 1) * a.L, a.V) - c * a.L;
                        const char* sb = rowp + static_cast<int64_t>(c) * a.L * E::kBytes;
                        const int vb = (g % kChunks) * 32;
                        const int v1 = vb + cln[g], v2 = vb + wg.lane2, v3 = wg.u3 >= zf ? vb + wg.lane3 : -1;
                        uint4 r1 = want_mv ? reinterpret_cast<const uint4*>(dyn + a.cmv_off)[g]
                                           : E::global_vec(sb, v1, sn, a.aligned);
                        const uint4 r2 = E::global_vec(sb, v2, sn, a.aligned);
                        uint4 r3 = r2;
                        if (v3 >= vb) r3 = E::global_vec(sb, v3, sn, a.aligned);
                        float z[VEC];
                        E::unpack(r1, z);
                        if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, c * Lv + v1, z);
                        emit(z, c * Lv + v1);
                        E::unpack(r2, z);
                        if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, c * Lv + v2, z);
                        emit(z, c * Lv + v2);
                        if (v3 >= vb) {
                            E::unpack(r3, z);
                            if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, c * Lv + v3, z);
                            emit(z, c * Lv + v3);
                        }
                    } else if (cu2[g] < zf && cln[g] >= 0) {
                        const int vs = (g % kChunks) * 32 + cln[g];
                        const int sn = min((c + 1) * a.L, a.V) - c * a.L;
                        float z[VEC];
                        E::unpack(want_mv ? reinterpret_cast<const uint4*>(dyn + a.cmv_off)[g]
                                          : E::global_vec(rowp + static_cast<int64_t>(c) * a.L * E::kBytes, vs, sn,
                                                          a.aligned),
                                  z);
                        if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, c * Lv + vs, z);
                        emit(z, c * Lv + vs);
                    } else {
                        whole[atomicAdd(&SS.nwhole, 1u)] = g;
                    }
                }
                __syncthreads();
                const int nw = static_cast<int>(SS.nwhole);
                // a listed chunk holds at least two ids >= zf (its max and its
                // second vector max): a list that cannot fit is not read
                if (nw > 0 && SS.ccount + 2u * static_cast<uint32_t>(nw) <= static_cast<uint32_t>(kCandCap)) {
                    // warp w reads listed chunks w, w + 8, ...: up to four in flight per lane
                    constexpr int kU = 4;
                    for (int i0 = warp; i0 < nw; i0 += kU * kWarps) {
                        const uint32_t got = *reinterpret_cast<volatile const uint32_t*>(&SS.ccount);
                        if (__shfl_sync(0xFFFFFFFFu, got, 0) > static_cast<uint32_t>(kCandCap)) break;
                        uint4 raw[kU];
                        int vr[kU];
#pragma unroll
                        for (int u = 0; u < kU; ++u) {
                            const int i = i0 + u * kWarps;
                            vr[u] = -1;
                            if (i < nw) {
                                const int g = whole[i];
                                const int c = g / kChunks;
                                const int vs = (g % kChunks) * 32 + lane;
                                const int sn = min((c + 1) * a.L, a.V) - c * a.L;
                                if (vs * VEC < sn) {  // padding vectors past the slice hold no id
                                    raw[u] = E::global_vec(rowp + static_cast<int64_t>(c) * a.L * E::kBytes, vs, sn,
                                                           a.aligned);
                                    vr[u] = c * Lv + vs;
                                }
                            }
                        }
#pragma unroll
                        for (int u = 0; u < kU; ++u) {
                            if (vr[u] >= 0) {
                                float z[VEC];
                                E::unpack(raw[u], z);
                                if (HIST && has_patch) apply_patches<VEC>(pbm, pwp, ppat, vr[u], z);
                                emit(z, vr[u]);
                            }
                        }
                    }
                    __syncthreads();
                } else if (nw > 0) {
                    SS.ccount = kCandCap + 1;  // (every thread stores the same value)
                    __syncthreads();
                }
                nc = static_cast<int>(SS.ccount);
                fast = nc <= kCandCap;
            }

            if (fast) {
                // ------------------------------------------------------ direct selection
                // every candidate in (key desc, id asc) order into sorted arrays:
                // few are ranked by counting, more by a bitonic sort of the
                // 64-bit values (padded with zeros, which rank last)
                uint32_t* sk = reinterpret_cast<uint32_t*>(dyn + a.sorted_off);
                int* sid = reinterpret_cast<int*>(sk + kCandCap);
                uint64_t* sm = reinterpret_cast<uint64_t*>(sid + kCandCap);
                if (nc <= kRankMax) {
                    for (int i = tid; i < nc; i += kThreads) {
                        const uint64_t vi = cc[i];
                        int rk = 0;
#pragma unroll 8
                        for (int j = 0; j < nc; ++j) rk += (cc[j] > vi) ? 1 : 0;
                        const uint32_t ki = static_cast<uint32_t>(vi >> 32);
                        sk[rk] = ki;
                        sid[rk] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(vi));
                        sm[rk] = fixq(weight_of(key_to_float(ki)));
                    }
                } else {
                    int n2 = kRankMax;
                    while (n2 < nc) n2 <<= 1;
                    bitonic_desc(cc, nc, n2);
                    for (int i = tid; i < nc; i += kThreads) {
                        const uint64_t vi = cc[i];
                        const uint32_t ki = static_cast<uint32_t>(vi >> 32);
                        sk[i] = ki;
                        sid[i] = static_cast<int>(0xFFFFFFFFu - static_cast<uint32_t>(vi));
                        sm[i] = fixq(weight_of(key_to_float(ki)));
                    }
                }
                if (tid == 0) {
                    SS.bi[5] = -1;
                    SS.bi[6] = -1;
                }
                __syncthreads();
                // K: sorted positions [0, nk)
                int nk = nc;
                Surv K{-INFINITY, INT_MAX};
                if (md.topk_on) {
                    nk = min(k, nc);
                    if (nk < k) st.err |= kErrInternal;  // the floor guarantees k ids
                    const bool later = nk < nc && sk[nk] == sk[nk - 1];
                    K = Surv{key_to_float(sk[nk - 1]), later ? sid[nk - 1] + 1 : INT_MAX};
                    st.kap_k = fkey(K.zt);
                    st.iot_k = K.ge_form() ? a.V : K.iota;
                }
                if (md.topk_on && !md.topp_on && !md.minp_on) {
                    // top-k alone: the survivors are K = positions [0, nk); each
                    // survivor's thread sums the K masses with smaller ids and all of
                    // them (the total, hence the target), so no scan runs
                    st.kap_r = st.kap_k;
                    st.iot_r = st.iot_k;
                    for (int pp = tid; pp < nk; pp += kThreads) {
                        const int ip = sid[pp];
                        uint64_t before = 0, tot = 0;
#pragma unroll 8
                        for (int qq = 0; qq < nk; ++qq) {
                            const uint64_t mq = sm[qq];
                            tot += mq;
                            before += (sid[qq] < ip) ? mq : 0u;
                        }
                        const uint64_t target = scale_by_u(st.rbits, tot);
                        const uint64_t mp = sm[pp];
                        if (mp != 0 && before <= target && target < before + mp) SS.bi[6] = ip;
                        st.mass_k = st.mass_r = tot;  // thread 0 (position 0) reports them
                        st.target = target;
                    }
                } else {
                    if (nc <= 4 * kThreads)
                        sorted_select<4>(a, P, md, st, SS, sk, sid, sm, nk, zm, K,
                                         reinterpret_cast<uint32_t*>(KS.fb.lhist), reinterpret_cast<uint32_t*>(cc));
                    else
                        sorted_select<8>(a, P, md, st, SS, sk, sid, sm, nk, zm, K,
                                         reinterpret_cast<uint32_t*>(KS.fb.lhist), reinterpret_cast<uint32_t*>(cc));
                }
                __syncthreads();
                st.token = SS.bi[6];
                if (st.token < 0) {
                    st.token = max_id();
                    st.err |= kErrInternal;
                }
            } else {
                finish_general<DT, HIST>(a, P, md, row, rowp, cm, pbm, pwp, ppat, has_patch, KS, dyn, st, g, rank);
            }
        }
    }

    if (!leader) return;  // a helper CTA of a split row: its part is done
    if (a.top_n > 0)
        top_n_row<DT, HIST>(a, row, P, mode >= 0, rowp, m, st.row_nan, cT, st.scale, want_mv, hbeg, hn, KS, dyn);

    // -------------------------------------------------------------- results
    if (tid == 0) {
        a.out[row] = st.token;
        if (st.err != 0 && a.err_word) atomicOr(a.err_word, st.err);
        if (a.debug) {
            arc_row_debug& dbg = a.debug[row];
            dbg.mode = mode;
            dbg.err = st.err;
            dbg.token = st.token;
            dbg.passes = st.passes;
            dbg.kappa_k = st.kap_k;
            dbg.iota_k = st.iot_k;
            dbg.kappa_r = st.kap_r;
            dbg.iota_r = st.iot_r;
            dbg.max_z = m;
            dbg.frac_bits = a.F;
            dbg.rbits = st.rbits;
            dbg.mass_k = st.mass_k;
            dbg.mass_r = st.mass_r;
            dbg.target = st.target;
        }
        if (a.flags & ARC_OPT_STEP_AUTOINC) a.params[row].step = P.step + 1;
        if (a.commit.ring != nullptr) commit_publish(a, row, st.token, SS);
    }
}

// One CTA per row, launched behind scan_kernel (programmatic dependent launch);
// when the batch leaves SMs idle, a cluster of a.fin_g CTAs per row: every CTA
// takes the row's decisions from the same summaries, a row that needs the
// threshold bisection splits its passes over the cluster, and CTA 0 writes
// the results.
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, 2) finish_kernel(const __grid_constant__ FinishArgs a) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ KernelShared KS;
    const int g = a.fin_g;
    const int row = static_cast<int>(blockIdx.x) / g;
    const int rank = static_cast<int>(blockIdx.x) - row * g;  // the CTA's rank in its cluster
    finish_row<DT, HIST>(
        a, row, KS, dyn, [&](int c) { return summary_at(a.summaries, a.s, row, c); },
        [] { asm volatile("griddepcontrol.wait;" ::: "memory"); }, [] {}, g, rank);
}

struct FusedArgs {
    ScanArgs scan;
    FinishArgs fin;
};

// Small batches in one launch: a thread-block cluster of s CTAs per row
// (s <= 16).  Every CTA scans its slice into its own shared memory; after a
// cluster barrier (release / acquire at cluster scope) CTA 0 of the cluster
// reads the s summaries through distributed shared memory and finishes the
// row, while the others wait at a second cluster barrier until those reads
// are done, then exit.  No workspace, no second launch, no global round trip
// for the summaries.
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, 2) cluster_kernel(const __grid_constant__ FusedArgs f) {
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ KernelShared KS;
    __shared__ ScanShared sh;
    __shared__ __align__(16) unsigned char mysum[kSummaryBytes];
    cg::cluster_group cl = cg::this_cluster();
    const int s = static_cast<int>(cl.num_blocks());
    const int rank = static_cast<int>(cl.block_rank());
    const int row = static_cast<int>(blockIdx.x) / s;
    scan_cta<DT, HIST>(f.scan, row, rank, sh, dyn, mysum);
    if (rank != 0) {
        cl.sync();  // the summaries are complete
        cl.sync();  // CTA 0 has copied them
        return;
    }
    // (the scan's shared memory is dead here: the finish reuses dyn)
    finish_row<DT, HIST>(
        f.fin, row, KS, dyn, [&](int c) { return static_cast<const unsigned char*>(cl.map_shared_rank(mysum, c)); },
        [&] { cl.sync(); }, [&] { cl.sync(); }, 1, 0);
}

}  // namespace arc
