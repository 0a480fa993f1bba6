// On-device sampling in two kernels, one HBM pass over the logits.
//
// scan_kernel: a row is split into s slices of at most kVpt * kThreads
// 16-byte vectors; one CTA per slice loads its slice into registers (all its
// 16-byte loads in flight at once), applies the history penalties, and
// writes a small summary to the workspace: the slice max and its first id,
// and per 32-vector chunk (256 bf16 / 128 fp32 logits) the chunk max and, for
// rows that need masses, the fp32 sum of 2^((z - chunk max) log2(e) / T).
// No CTA waits for another; registers stay few, so many CTAs per SM keep HBM
// busy.
//
// finish_kernel: one CTA per row combines the slice summaries.  Greedy rows
// take the row max.  Default rows draw from the chunk masses (exact integer
// fixed point, rescaled to the row max) and re-read only the 256-logit chunk
// that holds the draw.  Filtered rows run the exact top-k / top-p / min-p
// selection of row_select.cuh over the row read back from L2, skipping every
// chunk whose max lies below the current threshold.
#pragma once

#include <climits>

#include "row_select.cuh"

namespace arc {

constexpr int kVpt = 4;                  // 16-byte vectors per thread in a scan CTA
constexpr int kChunks = kVpt * kWarps;   // chunks per slice summary (32-vector chunks)
constexpr int kHdrBytes = 32;
constexpr int kSummaryBytes = kHdrBytes + kChunks * 8;
constexpr int kMaxRowCtas = 128;         // slices per row at most

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
    int patch_off;  // dynamic shared memory offset of the slice patch tables
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
    int bi[8];
    uint64_t bu[8];
    float bf[8];
};

struct __align__(16) KernelShared {
    SampleShared fb;
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
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads) scan_kernel(const ScanArgs a) {
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ float redf[kWarps];
    __shared__ int redi[kWarps];
    __shared__ uint32_t red32[kWarps];
    __shared__ uint32_t sflags;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x / a.s;
    const int cidx = blockIdx.x - row * a.s;
    const int a0 = cidx * a.L;
    const int n = max(0, min(a0 + a.L, a.V) - a0);
    const int nv = (n + VEC - 1) / VEC;
    const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;
    const char* slice = rowp + static_cast<int64_t>(a0) * E::kBytes;

    const arc_row_params P = load_params(a.params + row);
    uint32_t rerr = param_errors(P);
    const RowMode md(P, a.V);
    int hn = 0, hbeg = 0;
    if (HIST && a.hist_off != nullptr) {
        hbeg = a.hist_off[row];
        hn = a.hist_off[row + 1] - hbeg;
        if (hn < 0) rerr |= ARC_ERR_HIST_ID;
        if (hn > a.hist_cap) rerr |= ARC_ERR_HIST_CAP;
    }
    const bool need_data = rerr == 0;

    uint4 d[kVpt];
    const uint4 ninf = (DT == ARC_BF16) ? make_uint4(0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u, 0xFF80FF80u)
                                        : make_uint4(0xFF800000u, 0xFF800000u, 0xFF800000u, 0xFF800000u);
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        const int v = j * kThreads + tid;
        d[j] = (need_data && v < nv) ? E::global_vec(slice, v, n, a.aligned) : ninf;
    }
    if (tid == 0) sflags = 0;
    __syncthreads();

    const uint32_t* pbm = nullptr;
    const uint32_t* pwp = nullptr;
    const float* ppat = nullptr;
    bool has_patch = false;
    if (HIST && need_data && hn > 0) {
        const int nwords_max = (kVpt * kThreads * VEC + 31) / 32;
        uint32_t* bm = reinterpret_cast<uint32_t*>(dyn + a.patch_off);
        uint32_t* wp = bm + nwords_max;
        uint32_t* cnt = wp + nwords_max;
        float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
        const int distinct =
            build_patches<DT>(rowp, a.V, a0, n, nv, P, a.hist_ids + hbeg, hn, bm, wp, cnt, pat, red32, &sflags);
        rerr |= sflags & ARC_ERR_HIST_ID;
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

    // slice max and its first id; per-vector maxima for the chunk table
    float vm[kVpt];
    float bv = -INFINITY;
    int bi = -1;
    bool nanf = false;
#pragma unroll
    for (int j = 0; j < kVpt; ++j) {
        const int v = j * kThreads + tid;
        float x = -INFINITY;
        if (need_data && v < nv) {
            if (patched(j)) {
                float z[VEC];
                vals(j, z);
                x = z[0];
#pragma unroll
                for (int e = 1; e < VEC; ++e) x = fmax_nan(x, z[e]);
            } else {
                x = E::vmax_nan(d[j]);
            }
            if (x != x) {
                nanf = true;
                float z[VEC];
                vals(j, z);
                x = -INFINITY;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (z[e] > x) x = z[e];
            }
            if (x > bv) {
                float z[VEC];
                vals(j, z);
                int e0 = VEC - 1;
#pragma unroll
                for (int e = VEC - 1; e >= 0; --e)
                    if (z[e] == x) e0 = e;
                bv = x;
                bi = a0 + v * VEC + e0;
            }
        }
        vm[j] = x;
    }

    // chunk table: per 32-vector chunk its max and, when needed, the fp32 sum of
    // weights relative to it (NaN ids weigh nothing)
    const int rounds = (nv + kThreads - 1) / kThreads;
    unsigned char* mysum = const_cast<unsigned char*>(summary_at(a.summaries, a.s, row, cidx));
    const bool row_chunks = need_data && !md.greedy;
    if (row_chunks) {
        const float cT = __fdiv_rn(1.4426950408889634f, P.temperature);
        const bool slice_nan = __syncthreads_or(nanf) != 0;
        float2* ch = reinterpret_cast<float2*>(mysum + kHdrBytes);
#pragma unroll
        for (int j = 0; j < kVpt; ++j) {
            if (j < rounds) {
                const float mj = warp_max_f(vm[j]);
                float ls = 0.0f;
                if (md.need_mass && j * kThreads + tid < nv && mj != -INFINITY) {
                    float z[VEC];
                    vals(j, z);
#pragma unroll
                    for (int e = 0; e < VEC; ++e) {
                        const float w = (slice_nan && !(z[e] >= -INFINITY)) ? 0.0f : wrel(z[e], mj, cT);
                        ls = __fadd_rn(ls, w);
                    }
                }
                const float Sj = md.need_mass ? warp_sum_f(ls) : 0.0f;
                if (lane == 0) ch[j * kWarps + warp] = make_float2(mj, Sj);
            }
        }
    }

    warp_argmax(bv, bi);
    const bool wnan = __any_sync(0xFFFFFFFFu, nanf);
    if (lane == 0) {
        redf[warp] = bv;
        redi[warp] = bi;
        if (wnan) atomicOr(&sflags, ARC_ERR_NAN);
    }
    __syncthreads();
    if (tid == 0) {
        float mc = -INFINITY;
        int amc = -1;
        for (int w = 0; w < kWarps; ++w) better(mc, amc, redf[w], redi[w]);
        SliceHeader h;
        h.m = mc;
        h.am = amc;
        h.flags = (sflags & ARC_ERR_NAN) | (rerr & (ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP));
        h.nchunk = row_chunks ? rounds * kWarps : 0;
        h.pad[0] = h.pad[1] = h.pad[2] = h.pad[3] = 0;
        *reinterpret_cast<SliceHeader*>(mysum) = h;
    }
}

// ------------------------------------------------------------------ finish
template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads) finish_kernel(const FinishArgs a) {
    using E = Elem<DT>;
    using Ctx = RowCtx<DT, HIST>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ KernelShared KS;
    FinishScratch& SS = KS.st;
    FinishScratch& KSb = KS.st;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row = blockIdx.x;
    const int s = a.s;
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

    // row max, first id and flags over the slices
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
            KSb.bf[0] = v;
            KSb.bi[0] = i;
            KSb.bi[1] = static_cast<int>(f);
        }
    }
    __syncthreads();
    const float m = KSb.bf[0];
    const int am = KSb.bi[0];
    const uint32_t rflags = static_cast<uint32_t>(KSb.bi[1]);
    const bool row_nan = (rflags & ARC_ERR_NAN) != 0;
    rerr |= rflags & (ARC_ERR_HIST_ID | ARC_ERR_HIST_CAP);
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

    if (token == -2) {
        rbits = splitmix64(P.seed ^ (static_cast<uint64_t>(row) << 32) ^ P.step) >> 11;
        auto summary_of = [&](const FinishArgs& aa, int r, int c) { return summary_at(aa.summaries, s, r, c); };
        auto chunks_of = [&](const unsigned char* sm) { return chunk_table(sm); };
        // total mass from the chunk tables: sum over chunks of fix(S_j * 2^((m_j - m) c))
        auto chunk_q = [&](int gi) -> uint64_t {
            const int c = gi / kChunks, j = gi % kChunks;
            const float2 e = chunks_of(summary_of(a, row, c))[j];
            if (e.x == -INFINITY || e.y == 0.0f) return 0;
            const float r = wrel(e.x, m, cT);
            return fixq(__fmul_rn(e.y, r));
        };
        const int nch_row = s * kChunks;
        auto chunk_valid = [&](int gi) {
            const int c = gi / kChunks, j = gi % kChunks;
            const SliceHeader* h = reinterpret_cast<const SliceHeader*>(summary_of(a, row, c));
            return j < h->nchunk;
        };
        uint64_t S_all = 0;
        if (need_mass) {
            uint64_t acc = 0;
            for (int gi = tid; gi < nch_row; gi += kThreads)
                if (chunk_valid(gi)) acc += chunk_q(gi);
            S_all = block_sum_u64(acc, SS.redu);
        }
        if (mode == 1) {
            mass_r = S_all;
            target = scale_by_u(rbits, mass_r);
            // crossing chunk: id-order scan over the chunk masses, 256 at a time
            uint64_t run = 0;
            int hit = -1;
            uint64_t hit_before = 0, hit_q = 0;
            for (int g0 = 0; g0 < nch_row && hit < 0; g0 += kThreads) {
                const int gi = g0 + tid;
                const uint64_t q = (gi < nch_row && chunk_valid(gi)) ? chunk_q(gi) : 0;
                uint64_t tot;
                const uint64_t inc = block_scan_u64(q, SS.redu, tot);
                const bool cross = (run + inc > target) && (run + inc - q <= target) && q > 0;
                if (cross) {
                    KSb.bi[2] = gi;
                    KSb.bu[2] = run + inc - q;
                    KSb.bu[3] = q;
                }
                __syncthreads();
                if (run + tot > target) {
                    hit = KSb.bi[2];
                    hit_before = KSb.bu[2];
                    hit_q = KSb.bu[3];
                }
                run += tot;
                __syncthreads();
            }
            if (hit < 0) {
                err |= kErrInternal;
                token = am;
            } else if (warp == 0) {
                // re-read the chunk (32 vectors) and walk it
                const int c = hit / kChunks, jr = hit % kChunks;
                const int jround = jr / kWarps, w = jr % kWarps;
                const float2 e = __ldcg(chunks_of(summary_of(a, row, c)) + jr);
                const float mj = e.x;
                const float r = wrel(mj, m, cT);
                const int ca0 = c * a.L;
                const int cn = max(0, min(ca0 + a.L, a.V) - ca0);
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
                if (v < cnv) {
                    if (mj != -INFINITY) {
#pragma unroll
                        for (int q = 0; q < VEC; ++q) {
                            const float wq = (row_nan && !(z[q] >= -INFINITY)) ? 0.0f : wrel(z[q], mj, cT);
                            ls = __fadd_rn(ls, wq);
                        }
                    }
                }
                const uint64_t f = fixq(__fmul_rn(ls, r));
                const uint64_t inc = warp_inclusive_u64(f);
                const uint64_t Q = shfl_u64(inc, 31);
                uint64_t tres = target - hit_before;
                if (Q == 0) {
                    token = -3;  // no lane carries mass: take the chunk's max below
                } else {
                    if (tres >= Q) tres = Q - 1;  // rounding gap between the chunk total and its lanes
                    const unsigned bal = __ballot_sync(0xFFFFFFFFu, inc > tres);
                    const int l = __ffs(bal) - 1;
                    int eidx = -1;
                    if (lane == l) {
                        const uint64_t t2 = tres - (inc - f);
                        float part = 0.0f;
                        for (int q = 0; q < VEC; ++q) {
                            const float wq = (row_nan && !(z[q] >= -INFINITY)) ? 0.0f : wrel(z[q], mj, cT);
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
                if (lane == 0) KSb.bi[3] = token;
            }
            __syncthreads();
            if (hit >= 0) token = KSb.bi[3];
            if (token == -3) token = am;
            (void)hit_q;
            passes = 1;
        } else {
            // filtered rows: exact selection over the row in global memory,
            // skipping the chunks whose max lies below each pass's threshold
            float* cmax = reinterpret_cast<float*>(dyn + a.cmax_off);
            for (int gi = tid; gi < nch_row; gi += kThreads)
                cmax[gi] = chunk_valid(gi) ? chunk_table(summary_of(a, row, gi / kChunks))[gi % kChunks].x : -INFINITY;
            float zm = -INFINITY;
            if (lane == 0 && minp_on)
                zm = __double2float_ru(static_cast<double>(m) + static_cast<double>(T) * log(static_cast<double>(P.min_p)));
            zm = __shfl_sync(0xFFFFFFFFu, zm, 0);
            {
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
                X.vmax = cmax;
                X.vps = a.L / VEC;
                X.cps = kChunks;
                X.Wsum = reinterpret_cast<uint64_t*>(dyn + a.fb_wsum_off);
                X.par = 0;
                X.passes = 0;
                X.epoch = 1;
                X.ghist_zeroed = -1;
                X.cand_zeroed = -1;
                X.has_patch = false;
                X.row_nan = row_nan;
                X.bm = X.wp = nullptr;
                X.patch = nullptr;
                X.m = m;
                X.c = cT;
                X.scale = scale;
                X.infm = (m == INFINITY);
                for (int b = tid; b < kBins; b += kThreads) KS.fb.ghist[b] = 0;
                if (tid == 0) {
                    KS.fb.ccount = 0;
                    KS.fb.flags = 0;
                }
                __syncthreads();
                if (HIST && hn > 0) {
                    const int nwords_max = (a.fb_rounds * kThreads * VEC + 31) / 32;
                    uint32_t* bm = reinterpret_cast<uint32_t*>(dyn + a.fb_patch_off);
                    uint32_t* wp = bm + nwords_max;
                    uint32_t* cnt = wp + nwords_max;
                    float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
                    uint32_t badf = 0;
                    const int distinct = build_patches<DT>(rowp, a.V, 0, a.V, X.nv, P, a.hist_ids + hbeg, hn, bm, wp,
                                                           cnt, pat, KS.fb.wred32, &KS.fb.flags);
                    (void)badf;
                    X.bm = bm;
                    X.wp = wp;
                    X.patch = pat;
                    X.has_patch = distinct > 0;
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
                    float zb = -INFINITY;
                    if (lane == 0)
                        zb = __double2float_rd(static_cast<double>(m) +
                                               static_cast<double>(T) * log((1.0 - static_cast<double>(P.top_p)) /
                                                                            (2.0 * static_cast<double>(a.V))));
                    zb = __shfl_sync(0xFFFFFFFFu, zb, 0);
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
                    uint64_t tgt = 1;
                    if (lane == 0)
                        tgt = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(mass_k)));
                    tgt = shfl_u64(tgt, 0);
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
