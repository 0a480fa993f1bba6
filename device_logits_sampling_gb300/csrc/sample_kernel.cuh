// Fused per-row sampling kernel: one thread-block cluster of s CTAs per row.
//
// Each CTA bulk-copies (TMA, cp.async.bulk) its contiguous slice of the row
// into shared memory once; every later look at the row -- max, top-k select,
// top-p select, masses, the inverse-CDF walk -- runs out of shared memory.
// Pass 1 also caches each 16-byte vector's max, so later threshold passes
// skip vectors that cannot hold a survivor without reading them.
//
// CTAs of a row combine partial results through distributed shared memory
// (DSMEM).  Every decision is computed redundantly and identically by all
// CTAs from the same exchanged data, so control flow, and with it the
// sequence of cluster barriers, is uniform across the cluster.
//
// Thresholds are found by multi-way threshold bisection on the order-
// preserving u32 key of the logit: a 512-bin histogram of the keys in a window
// below the row max (each CTA adds its non-zero bins into every CTA's cluster
// histogram with DSMEM atomics; one cluster barrier) locates the bin that
// crosses the target count (top-k) or mass (top-p); the few ids in that bin
// are then gathered into every CTA and ranked exactly.  Bins that hold too
// many ids are bisected further, 9 bits per pass.
//
// Masses are fixed-point integers (units of 2^-F of the max weight), so sums
// are exact, associative and identical in every pass, CTA and cluster size.
#pragma once

#include <climits>

#include "arc_device.cuh"

namespace arc {

struct SampleArgs {
    const void* logits;
    int64_t ld;  // row stride, elements
    int B;
    int V;
    arc_row_params* params;
    const int32_t* hist_off;
    const int32_t* hist_ids;
    int32_t* out;
    uint32_t* err_word;
    arc_row_debug* debug;
    int L;           // slice elements per CTA (multiple of the vector width)
    int vmax_off;    // dynamic shared memory offsets: per-vector max,
    int wsum_off;    //   per-(round, warp) masses,
    int hist_off_b;  //   history patch tables
    int rounds_max;  // rounds of the largest slice
    int hist_cap;    // history entries per row (patch table capacity)
    int F;           // fixed-point fraction bits
    uint32_t flags;  // ARC_OPT_*
    int aligned;     // rows start on 16-byte boundaries: bulk copies allowed
};

struct __align__(16) SampleShared {
    uint64_t bar[kPieces];
    uint64_t lhist[kBins];  // this CTA's histogram
    uint64_t ghist[kBins];  // the cluster's histogram (every CTA adds into it)
    uint64_t cval[kCand];   // gathered candidates: id or mass
    uint32_t ckey[kCand];   //   and key
    uint64_t slot[2][8];    // exchange ring
    uint64_t wred[kWarps];
    uint64_t bcast_u[4];
    int bcast_i[4];
    uint32_t wred32[kWarps];
    uint32_t ccount;        // candidates pushed into this CTA
    uint32_t flags;
};

constexpr uint32_t kErrInternal = ARC_ERR_INTERNAL;

// Survivor predicate on the penalised logit z at id `idx`:
// survive iff z > zt || (z == zt && idx < iota); iota == INT_MAX means z >= zt.
struct Surv {
    float zt;
    int iota;
    __device__ __forceinline__ bool ge_form() const { return iota == INT_MAX; }
    __device__ __forceinline__ bool test(float z, int idx) const {
        return z > zt || (z == zt && idx < iota);
    }
};

// How a mass pass tests its domain: every id (the row has no NaN), z >= zt,
// or the full (z, id) predicate.
enum MassMode { kAll = 0, kGe = 1, kTie = 2 };

struct Window {
    uint32_t klo, khi;
    int sh;
};

template <int DT, bool HIST>
struct RowCtx {
    using E = Elem<DT>;
    static constexpr int VEC = E::kVec;

    SampleShared& S;
    cg::cluster_group cl;
    int s, rank, row, tid, lane, warp;
    int a0, a1, n, nv, nvf, rounds;
    const unsigned char* data;
    float* vmax;
    uint64_t* Wsum;
    // history patches
    const uint32_t* bm;
    const uint32_t* wp;
    const float* patch;
    bool has_patch;
    bool row_nan;
    // weights: w = ex2((z - m) * c), or [z == m] when m = +inf
    float m, c, scale;
    bool infm;
    int par;           // exchange ring parity
    int passes;
    int epoch;         // cluster barriers so far
    int ghist_zeroed;  // epoch at which the cluster histogram was last cleared
    int cand_zeroed;   // epoch at which the candidate count was last cleared

    __device__ RowCtx(SampleShared& S_, cg::cluster_group cl_) : S(S_), cl(cl_) {}

    // ---------------------------------------------------------------- loads
    __device__ __forceinline__ bool vec_patched(int v) const {
        if (!(HIST && has_patch)) return false;
        const int l0 = v * VEC;
        return ((bm[l0 >> 5] >> (l0 & 31)) & ((1u << VEC) - 1u)) != 0;
    }

    __device__ __forceinline__ void load(int v, float (&z)[VEC]) const {
        const uint4 raw = reinterpret_cast<const uint4*>(data)[v];
        E::unpack(raw, z);
        if (HIST && has_patch) {
            const int l0 = v * VEC;
            const uint32_t word = bm[l0 >> 5];
            const uint32_t bits = (word >> (l0 & 31)) & ((1u << VEC) - 1u);
            if (bits) {
                const int base = static_cast<int>(wp[l0 >> 5]);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int li = l0 + e;
                    if ((bits >> e) & 1u) z[e] = patch[base + __popc(word & ((1u << (li & 31)) - 1u))];
                }
            }
        }
    }

    __device__ __forceinline__ float weight(float z) const {
        return infm ? (z == m ? 1.0f : 0.0f) : ex2(__fmul_rn(__fsub_rn(z, m), c));
    }

    __device__ __forceinline__ uint64_t fix(float w) const { return __float2ull_rn(__fmul_rn(w, scale)); }

    __device__ __forceinline__ static bool in_domain(int mode, const Surv& d, float z, int idx) {
        return mode == kAll ? true : (mode == kGe ? (z >= d.zt) : d.test(z, idx));
    }

    // fixed-point mass of the survivors of one vector: fp32 sum in id order,
    // rounded once
    __device__ __forceinline__ uint64_t vec_mass(int mode, const float (&z)[VEC], int g0, const Surv& d) const {
        float sum = 0.0f;
        if (mode == kAll) {
#pragma unroll
            for (int e = 0; e < VEC; ++e) sum = __fadd_rn(sum, weight(z[e]));
        } else {
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (in_domain(mode, d, z[e], g0 + e)) sum = __fadd_rn(sum, weight(z[e]));
        }
        return fix(sum);
    }

    // first element of the vector whose running fixed-point mass exceeds t
    __device__ __forceinline__ int vec_mass_walk(int mode, const float (&z)[VEC], int g0, const Surv& d,
                                                 uint64_t t) const {
        float sum = 0.0f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            if (in_domain(mode, d, z[e], g0 + e)) sum = __fadd_rn(sum, weight(z[e]));
            if (fix(sum) > t) return e;
        }
        return -1;
    }

    // ---------------------------------------------------------------- cluster exchange
    __device__ __forceinline__ void xsync() {
        cl.sync();
        epoch++;
    }
    __device__ __forceinline__ uint64_t xread(int r, int i) const {
        return cl.map_shared_rank(&S.slot[par][0], r)[i];
    }
    __device__ __forceinline__ void xnext() { par ^= 1; }

    struct Scan {
        uint64_t total, before_me;
        int first;
        uint64_t before_first;
    };
    // Sum over the cluster of slot value i, this CTA's exclusive prefix and the
    // first rank whose inclusive prefix exceeds t (-1 if none).
    __device__ __forceinline__ Scan xscan(int i, uint64_t t) const {
        const uint64_t x = (lane < s) ? xread(lane, i) : 0;
        const uint64_t inc = warp_inclusive_u64(x);
        Scan r;
        r.total = shfl_u64(inc, 31);
        r.before_me = shfl_u64(inc - x, rank);
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, lane < s && inc > t);
        r.first = bal ? __ffs(bal) - 1 : -1;
        r.before_first = bal ? shfl_u64(inc - x, r.first) : 0;
        return r;
    }

    // Total of this CTA's Wsum into S.slot[par][i].
    __device__ __forceinline__ void publish_wsum_total(int i) {
        __syncthreads();
        if (warp == 0) {
            uint64_t acc = 0;
            for (int e = lane; e < rounds * kWarps; e += 32) acc += Wsum[e];
            acc = warp_sum_u64(acc);
            if (lane == 0) S.slot[par][i] = acc;
        }
    }

    // First position of arr[0..n) whose inclusive prefix exceeds t (warp-wide).
    __device__ __forceinline__ static void warp_find(const uint64_t* arr, int n, uint64_t t, int& pos,
                                                     uint64_t& before, uint64_t& value) {
        const int ln = threadIdx.x & 31;
        uint64_t base = 0;
        pos = -1;
        before = 0;
        value = 0;
        for (int e0 = 0; e0 < n; e0 += 32) {
            const uint64_t x = (e0 + ln < n) ? arr[e0 + ln] : 0;
            const uint64_t inc = warp_inclusive_u64(x) + base;
            const unsigned bal = __ballot_sync(0xFFFFFFFFu, (e0 + ln < n) && inc > t);
            if (bal) {
                const int l = __ffs(bal) - 1;
                pos = e0 + l;
                before = shfl_u64(inc - x, l);
                value = shfl_u64(x, l);
                return;
            }
            base = shfl_u64(inc, 31);
        }
        before = base;  // the total when nothing crosses
    }

    // ---------------------------------------------------------------- histograms
    __device__ __forceinline__ static int bitlen(uint32_t x) { return x ? 32 - __clz(x) : 0; }
    __device__ __forceinline__ static Window make_window(uint32_t klo, uint32_t khi) {
        Window w;
        w.klo = klo;
        w.khi = khi;
        w.sh = max(0, bitlen(khi - klo) - kBinBits);
        return w;
    }
    __device__ __forceinline__ static float lo_float(uint32_t klo) {
        return klo <= 0x007FFFFFu ? -INFINITY : key_to_float(klo);
    }

    __device__ __forceinline__ void lhist_add(const Window& W, uint32_t k, uint64_t wt) {
        if (k < W.klo || k > W.khi) return;
        atomicAdd(reinterpret_cast<unsigned long long*>(&S.lhist[(W.khi - k) >> W.sh]),
                  static_cast<unsigned long long>(wt));
    }

    __device__ __forceinline__ void lhist_clear() {
        for (int b = tid; b < kBins; b += kThreads) S.lhist[b] = 0;
        __syncthreads();
    }

    // Clear the cluster histogram / candidate count after their last local
    // read.  A cluster barrier must separate a clear from the next remote
    // push into it; the push helpers add one when none has passed.
    __device__ __forceinline__ void ghist_clear() {
        __syncthreads();
        for (int b = tid; b < kBins; b += kThreads) S.ghist[b] = 0;
        ghist_zeroed = epoch;
    }
    __device__ __forceinline__ void cand_clear() {
        __syncthreads();
        if (tid == 0) S.ccount = 0;
        cand_zeroed = epoch;
    }

    // Add this CTA's non-zero bins into every CTA's cluster histogram.
    __device__ __forceinline__ void push_hist() {
        if (ghist_zeroed >= epoch) xsync();
        for (int b = tid; b < kBins; b += kThreads) {
            const uint64_t v = S.lhist[b];
            if (v)
                for (int q = 0; q < s; ++q)
                    atomicAdd(reinterpret_cast<unsigned long long*>(cl.map_shared_rank(S.ghist, q) + b),
                              static_cast<unsigned long long>(v));
        }
    }

    // Give a candidate (key, value) to every CTA of the cluster.  The count
    // keeps growing past kCand so that every CTA sees the true total.
    __device__ __forceinline__ void push_cand(uint32_t key, uint64_t val) {
        for (int q = 0; q < s; ++q) {
            const uint32_t slot_i = atomicAdd(cl.map_shared_rank(&S.ccount, q), 1u);
            if (slot_i < static_cast<uint32_t>(kCand)) {
                cl.map_shared_rank(S.ckey, q)[slot_i] = key;
                cl.map_shared_rank(S.cval, q)[slot_i] = val;
            }
        }
    }

    struct Sel {
        int bin;          // crossing bin (-1: the window does not reach the target)
        uint64_t before;  // weight in the bins above it
        uint64_t inbin;   // weight in it
    };

    // After the barrier that completes the cluster histogram: the first bin
    // whose inclusive prefix (from the top key down) is >= target.
    __device__ Sel ghist_find(uint64_t target) {
        if (warp == 0) {
            int pos;
            uint64_t bf, val;
            warp_find(S.ghist, kBins, target - 1, pos, bf, val);
            if (lane == 0) {
                S.bcast_i[0] = pos;
                S.bcast_u[0] = bf;
                S.bcast_u[1] = val;
            }
        }
        __syncthreads();
        Sel r;
        r.bin = S.bcast_i[0];
        r.before = S.bcast_u[0];
        r.inbin = S.bcast_u[1];
        return r;
    }

    // ---------------------------------------------------------------- index-order walk
    // In this CTA, the element whose running weight (in id order over the
    // Wsum chunks) first exceeds t.  Returns the row index or -1.
    template <class VecW, class VecWalk>
    __device__ int walk(uint64_t t, VecW vecw, VecWalk vecwalk) {
        if (warp == 0) {
            int pos;
            uint64_t bf, val;
            warp_find(Wsum, rounds * kWarps, t, pos, bf, val);
            int token = -1;
            if (pos >= 0) {
                const int j = pos / kWarps, w = pos % kWarps;
                const uint64_t t2 = t - bf;
                const int v = j * kThreads + w * 32 + lane;
                float z[VEC];
                uint64_t q = 0;
                if (v < nv) {
                    load(v, z);
                    q = vecw(z, a0 + v * VEC);
                }
                const uint64_t inc = warp_inclusive_u64(q);
                const unsigned bal = __ballot_sync(0xFFFFFFFFu, inc > t2);
                const int l = bal ? __ffs(bal) - 1 : -1;
                int e = -1;
                if (lane == l) e = vecwalk(z, a0 + v * VEC, t2 - (inc - q));
                if (l >= 0) {
                    e = __shfl_sync(0xFFFFFFFFu, e, l);
                    if (e >= 0) token = a0 + (j * kThreads + w * 32 + l) * VEC + e;
                }
            }
            if (lane == 0) S.bcast_i[1] = token;
        }
        __syncthreads();
        const int tok = S.bcast_i[1];
        __syncthreads();
        return tok;
    }
};

// Row parameters, read once with volatile loads so that no field is fetched
// after the first cluster barrier (rank 0 may rewrite `step` after it).
__device__ __forceinline__ arc_row_params load_params(const arc_row_params* p) {
    const volatile uint64_t* q = reinterpret_cast<const volatile uint64_t*>(p);
    uint64_t w[6];
#pragma unroll
    for (int i = 0; i < 6; ++i) w[i] = q[i];
    arc_row_params r;
    r.temperature = __uint_as_float(static_cast<uint32_t>(w[0]));
    r.top_k = static_cast<int32_t>(w[0] >> 32);
    r.top_p = __uint_as_float(static_cast<uint32_t>(w[1]));
    r.min_p = __uint_as_float(static_cast<uint32_t>(w[1] >> 32));
    r.repetition_penalty = __uint_as_float(static_cast<uint32_t>(w[2]));
    r.frequency_penalty = __uint_as_float(static_cast<uint32_t>(w[2] >> 32));
    r.presence_penalty = __uint_as_float(static_cast<uint32_t>(w[3]));
    r.flags = static_cast<uint32_t>(w[3] >> 32);
    r.seed = w[4];
    r.step = w[5];
    return r;
}

// Key range [lo, hi] of histogram bin `b` of window W.
__device__ __forceinline__ void bin_range(const Window& W, int b, uint32_t& lo, uint32_t& hi) {
    hi = W.khi - (static_cast<uint32_t>(b) << W.sh);
    int64_t lo64 = static_cast<int64_t>(hi) - ((int64_t{1} << W.sh) - 1);
    if (lo64 < static_cast<int64_t>(W.klo)) lo64 = static_cast<int64_t>(W.klo);
    lo = static_cast<uint32_t>(lo64);
}

// Local histogram of the ids of D whose keys lie in W: counts (MASS = false)
// or fixed-point masses.  Vectors whose max is below the window are skipped.
template <class Ctx, bool MASS>
__device__ void pass_hist(Ctx& X, const Window& W, const Surv& D) {
    constexpr int VEC = Ctx::VEC;
    X.lhist_clear();
    const float zlo = Ctx::lo_float(W.klo), zhi = key_to_float(W.khi);
    const float thr = fmaxf(zlo, D.zt);
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        if (v < X.nv && X.vmax[v] >= thr) {
            float z[VEC];
            X.load(v, z);
            const int g0 = X.a0 + v * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (z[e] >= zlo && z[e] <= zhi && D.test(z[e], g0 + e))
                    X.lhist_add(W, fkey(z[e]), MASS ? X.fix(X.weight(z[e])) : 1u);
        }
    }
    X.passes++;
    __syncthreads();
}

// Give every CTA the ids of D whose keys lie in [lo, hi] as candidates:
// (key, id) for counts, (key, mass) for masses.
template <class Ctx, bool MASS>
__device__ void pass_collect(Ctx& X, uint32_t lo, uint32_t hi, const Surv& D) {
    constexpr int VEC = Ctx::VEC;
    if (X.cand_zeroed >= X.epoch) X.xsync();
    const float zlo = Ctx::lo_float(lo), zhi = key_to_float(hi);
    const float thr = fmaxf(zlo, D.zt);
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        if (v < X.nv && X.vmax[v] >= thr) {
            float z[VEC];
            X.load(v, z);
            const int g0 = X.a0 + v * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if (z[e] >= zlo && z[e] <= zhi && D.test(z[e], g0 + e)) {
                    const uint32_t k = fkey(z[e]);
                    if (k >= lo && k <= hi)
                        X.push_cand(k, MASS ? X.fix(X.weight(z[e])) : static_cast<uint64_t>(g0 + e));
                }
            }
        }
    }
    X.passes++;
}

// Per-(round, warp) fixed-point masses of the survivors of D into Wsum; with
// HISTO also the local mass histogram of the survivors whose keys lie in W.
template <class Ctx, bool HISTO>
__device__ void pass_mass(Ctx& X, int mode, const Surv& D, const Window& W) {
    constexpr int VEC = Ctx::VEC;
    if (HISTO) X.lhist_clear();
    const float zlo = Ctx::lo_float(W.klo), zhi = key_to_float(W.khi);
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        uint64_t q = 0;
        if (v < X.nv && (mode == kAll || X.vmax[v] >= D.zt)) {
            float z[VEC];
            X.load(v, z);
            const int g0 = X.a0 + v * VEC;
            q = X.vec_mass(mode, z, g0, D);
            if (HISTO && X.vmax[v] >= zlo) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (z[e] >= zlo && z[e] <= zhi && Ctx::in_domain(mode, D, z[e], g0 + e))
                        X.lhist_add(W, fkey(z[e]), X.fix(X.weight(z[e])));
            }
        }
        q = warp_sum_u64(q);
        if (X.lane == 0) X.Wsum[j * kWarps + X.warp] = q;
    }
    X.passes++;
}

template <class Ctx>
__device__ __forceinline__ int mass_mode(const Ctx& X, const Surv& D) {
    if (!D.ge_form()) return kTie;
    return (D.zt == -INFINITY && !X.row_nan) ? kAll : kGe;
}

// The need-th id (1-based, id order) whose logit equals zt: the id bound of
// a top-k set whose ties at zt are too many to gather.
template <class Ctx>
__device__ int tie_walk(Ctx& X, float zt, uint64_t need) {
    constexpr int VEC = Ctx::VEC;
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        uint64_t q = 0;
        if (v < X.nv && X.vmax[v] >= zt) {
            float z[VEC];
            X.load(v, z);
#pragma unroll
            for (int e = 0; e < VEC; ++e) q += (z[e] == zt) ? 1u : 0u;
        }
        q = warp_sum_u64(q);
        if (X.lane == 0) X.Wsum[j * kWarps + X.warp] = q;
    }
    X.passes++;
    X.publish_wsum_total(0);
    X.xsync();
    const typename Ctx::Scan sc = X.xscan(0, need - 1);
    X.xnext();
    if (sc.first == X.rank) {
        const int pos = X.walk(
            need - 1 - sc.before_me,
            [&](const float(&z)[VEC], int) {
                uint64_t c = 0;
#pragma unroll
                for (int e = 0; e < VEC; ++e) c += (z[e] == zt) ? 1u : 0u;
                return c;
            },
            [&](const float(&z)[VEC], int, uint64_t t) {
                uint64_t c = 0;
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    c += (z[e] == zt) ? 1u : 0u;
                    if (c > t) return e;
                }
                return -1;
            });
        if (X.tid == 0) X.S.slot[X.par][0] = static_cast<uint64_t>(static_cast<uint32_t>(pos));
    }
    X.xsync();
    const int pos = (sc.first >= 0) ? static_cast<int>(static_cast<uint32_t>(X.xread(sc.first, 0))) : -1;
    X.xnext();
    return pos;
}

// Exact top-k survivor set: the first k ids by (z desc, id asc).
template <class Ctx>
__device__ Surv select_topk(Ctx& X, int k, uint32_t Km, uint32_t& err) {
    const Surv all{-INFINITY, INT_MAX};
    uint64_t tgt = static_cast<uint64_t>(k);
    // first window: 2^23 keys (one binade) below the max, widened 16x while it
    // holds fewer than k ids
    uint32_t width = 1u << 23;
    Window W = Ctx::make_window(Km > width - 1 ? Km - (width - 1) : 0u, Km);
    bool first = true;
    while (true) {
        pass_hist<Ctx, false>(X, W, all);
        X.push_hist();
        X.xsync();
        const typename Ctx::Sel r = X.ghist_find(tgt);
        X.ghist_clear();
        if (r.bin < 0) {
            if (first && W.klo > 0) {
                width = (width >= (1u << 27)) ? 0u : (width << 4);
                const uint32_t lo = (width == 0u || Km < width - 1) ? 0u : Km - (width - 1);
                W = Ctx::make_window(lo, Km);
                continue;
            }
            return all;  // fewer than k non-NaN ids: keep them all
        }
        first = false;
        uint32_t lo, hi;
        bin_range(W, r.bin, lo, hi);
        if (r.before + r.inbin == tgt) return Surv{Ctx::lo_float(lo), INT_MAX};
        tgt -= r.before;  // ids still needed from this bin
        if (r.inbin > static_cast<uint64_t>(kCand)) {
            if (W.sh > 0) {  // too many ids in the bin: bisect it further
                W.klo = lo;
                W.khi = hi;
                W.sh = max(0, W.sh - kBinBits);
                continue;
            }
            // one key with too many ties to gather: walk them in id order
            const float zt = key_to_float(hi);
            const int pos = tie_walk(X, zt, tgt);
            if (pos < 0) {
                err |= kErrInternal;
                return Surv{zt, INT_MAX};
            }
            return Surv{zt, pos + 1};
        }
        // gather the bin's ids into every CTA and rank them by (key desc, id asc)
        pass_collect<Ctx, false>(X, lo, hi, all);
        X.xsync();
        const int nc = static_cast<int>(min(X.S.ccount, static_cast<uint32_t>(kCand)));
        if (X.tid == 0) X.S.bcast_i[2] = -1;
        __syncthreads();
        if (X.tid < nc) {
            const uint32_t ki = X.S.ckey[X.tid];
            const int ii = static_cast<int>(X.S.cval[X.tid]);
            int rk = 0;
            for (int q = 0; q < nc; ++q) {
                const uint32_t kq = X.S.ckey[q];
                const int iq = static_cast<int>(X.S.cval[q]);
                rk += (kq > ki || (kq == ki && iq < ii)) ? 1 : 0;
            }
            if (rk == static_cast<int>(tgt) - 1) X.S.bcast_i[2] = X.tid;
        }
        __syncthreads();
        const int wi = X.S.bcast_i[2];
        Surv K = all;
        if (wi < 0) {
            err |= kErrInternal;
        } else {
            const uint32_t kw = X.S.ckey[wi];
            const int iw = static_cast<int>(X.S.cval[wi]);
            // more ids tied at kw beyond iw: the id bound matters
            int later = 0;
            for (int q = X.tid; q < nc; q += kThreads)
                later |= (X.S.ckey[q] == kw && static_cast<int>(X.S.cval[q]) > iw) ? 1 : 0;
            later = __syncthreads_or(later);
            K = Surv{key_to_float(kw), later ? iw + 1 : INT_MAX};
        }
        X.cand_clear();
        return K;
    }
}

// Top-p cutoff from the mass histogram of window W (already pushed, barrier
// passed): true and zp (z >= zp survives) when W holds the target mass.
template <class Ctx>
__device__ bool select_mass(Ctx& X, Window W, const Surv& K, uint64_t tgt, float& zp) {
    while (true) {
        const typename Ctx::Sel r = X.ghist_find(tgt);
        X.ghist_clear();
        if (r.bin < 0) return false;
        uint32_t lo, hi;
        bin_range(W, r.bin, lo, hi);
        if (W.sh == 0) {
            zp = key_to_float(hi);
            return true;
        }
        if (r.before + r.inbin == tgt) {
            zp = Ctx::lo_float(lo);
            return true;
        }
        tgt -= r.before;
        // gather the bin's ids (key, mass) into every CTA and find the largest
        // key whose mass at or above it reaches the target
        pass_collect<Ctx, true>(X, lo, hi, K);
        X.xsync();
        const uint32_t got = X.S.ccount;
        if (got <= static_cast<uint32_t>(kCand)) {
            const int nc = static_cast<int>(got);
            uint32_t best = 0;
            if (X.tid < nc) {
                const uint32_t ki = X.S.ckey[X.tid];
                uint64_t mge = 0;
                for (int q = 0; q < nc; ++q)
                    if (X.S.ckey[q] >= ki) mge += X.S.cval[q];
                if (mge >= tgt) best = ki;
            }
            best = __reduce_max_sync(0xFFFFFFFFu, best);
            if (X.lane == 0) X.S.wred32[X.warp] = best;
            __syncthreads();
            uint32_t kb = 0;
            for (int w = 0; w < kWarps; ++w) kb = max(kb, X.S.wred32[w]);
            X.cand_clear();  // (its barrier also orders the wred32 reads)
            zp = key_to_float(kb);
            return true;
        }
        // too many ids: bisect the bin with another histogram pass
        X.cand_clear();
        W.klo = lo;
        W.khi = hi;
        W.sh = max(0, W.sh - kBinBits);
        pass_hist<Ctx, true>(X, W, K);
        X.push_hist();
        X.xsync();
    }
}

template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads, 3) sample_kernel(const SampleArgs a) {
    using Ctx = RowCtx<DT, HIST>;
    using E = Elem<DT>;
    constexpr int VEC = E::kVec;
    extern __shared__ __align__(128) unsigned char dyn[];
    __shared__ SampleShared S;

    Ctx X(S, cg::this_cluster());
    X.s = static_cast<int>(X.cl.num_blocks());
    X.rank = static_cast<int>(X.cl.block_rank());
    X.row = blockIdx.x / X.s;
    X.tid = threadIdx.x;
    X.lane = X.tid & 31;
    X.warp = X.tid >> 5;
    X.a0 = X.rank * a.L;
    X.a1 = min(X.a0 + a.L, a.V);
    X.n = max(0, X.a1 - X.a0);
    X.nv = (X.n + VEC - 1) / VEC;
    X.nvf = X.n / VEC;
    X.rounds = (X.nv + kThreads - 1) / kThreads;
    X.data = dyn;
    X.vmax = reinterpret_cast<float*>(dyn + a.vmax_off);
    X.Wsum = reinterpret_cast<uint64_t*>(dyn + a.wsum_off);
    X.par = 0;
    X.passes = 0;
    X.epoch = 0;
    X.ghist_zeroed = -1;
    X.cand_zeroed = -1;
    X.has_patch = false;
    X.row_nan = false;
    X.bm = X.wp = nullptr;
    X.patch = nullptr;
    X.m = 0.0f;
    X.c = 0.0f;
    X.scale = 1.0f;
    X.infm = false;
    const int tid = X.tid, lane = X.lane, warp = X.warp, row = X.row;
    const int a0 = X.a0, a1 = X.a1, n = X.n;
    unsigned char* data = dyn;
    const char* rowp = static_cast<const char*>(a.logits) + static_cast<int64_t>(row) * a.ld * E::kBytes;

    // -------------------------------------------------------------- bulk copies of the slice
    const int rpp = max(1, (X.rounds + kPieces - 1) / kPieces);  // rounds per piece
    auto piece_v1 = [&](int p) { return min((p + 1) * rpp * kThreads, X.nvf); };
    if (tid == 0) {
        for (int p = 0; p < kPieces; ++p) mbar_init(&S.bar[p], 1);
        fence_mbar_init();
        S.flags = 0;
        S.ccount = 0;
    }
    // the cluster histogram must be zero before any CTA pushes into it (the
    // first cluster barrier orders this)
    for (int b = tid; b < kBins; b += kThreads) S.ghist[b] = 0;
    __syncthreads();
    if (a.aligned && tid == 0) {
        for (int p = 0; p < kPieces; ++p) {
            const int v0 = p * rpp * kThreads, v1 = piece_v1(p);
            if (v1 > v0) {
                const uint32_t bytes = static_cast<uint32_t>(v1 - v0) * 16u;
                mbar_arrive_expect_tx(&S.bar[p], bytes);
                bulk_load(data + static_cast<size_t>(v0) * 16,
                          rowp + static_cast<int64_t>(a0) * E::kBytes + static_cast<int64_t>(v0) * 16, bytes,
                          &S.bar[p]);
            }
        }
    }
    // -------------------------------------------------------------- parameters
    const arc_row_params P = load_params(a.params + row);
    uint32_t rerr = 0;
    {
        const float T = P.temperature;
        bool ok = isfinite(T) && T >= 0.0f;
        ok &= (P.top_p > 0.0f) && (P.top_p <= 1.0f);
        ok &= (P.min_p >= 0.0f) && (P.min_p <= 1.0f);
        ok &= isfinite(P.repetition_penalty) && P.repetition_penalty > 0.0f;
        ok &= isfinite(P.frequency_penalty) && isfinite(P.presence_penalty);
        ok &= P.flags == 0u;
        if (!ok) rerr |= ARC_ERR_PARAM;
    }
    // ids not covered by bulk copies: the ragged tail, or the whole slice when
    // rows are not 16-byte aligned.  The last vector is padded with -inf (zero
    // weight, never a maximum); its padded ids lie beyond V.
    {
        const int first = a.aligned ? X.nvf * VEC : 0;
        for (int i = first + tid; i < X.nv * VEC; i += kThreads) {
            if (i < n)
                E::store_smem_raw(data, i, rowp, a0 + i);
            else if (DT == ARC_BF16)
                reinterpret_cast<unsigned short*>(data)[i] = 0xFF80;
            else
                reinterpret_cast<uint32_t*>(data)[i] = 0xFF800000u;
        }
    }
    // -------------------------------------------------------------- history patches
    if (HIST && a.hist_off != nullptr) {
        const int hbeg = a.hist_off[row];
        const int hn = a.hist_off[row + 1] - hbeg;
        if (hn < 0) rerr |= ARC_ERR_HIST_ID;
        if (hn > a.hist_cap) rerr |= ARC_ERR_HIST_CAP;
        if (hn > 0 && rerr == 0) {
            const int nwords = (X.nv * VEC + 31) / 32;
            const int nwords_max = (a.rounds_max * kThreads * VEC + 31) / 32;
            uint32_t* bmw = reinterpret_cast<uint32_t*>(dyn + a.hist_off_b);
            uint32_t* wpw = bmw + nwords_max;
            uint32_t* cnt = wpw + nwords_max;
            float* pat = reinterpret_cast<float*>(cnt + a.hist_cap);
            for (int w = tid; w < nwords; w += kThreads) bmw[w] = 0;
            __syncthreads();
            for (int e = tid; e < hn; e += kThreads) {
                const int id = a.hist_ids[hbeg + e];
                if (id < 0 || id >= a.V)
                    atomicOr(&S.flags, ARC_ERR_HIST_ID);
                else if (id >= a0 && id < a1)
                    atomicOr(&bmw[(id - a0) >> 5], 1u << ((id - a0) & 31));
            }
            __syncthreads();
            rerr |= S.flags & ARC_ERR_HIST_ID;
            // rank of an id among the history ids of this slice: prefix popcount
            const int per = (nwords + kThreads - 1) / kThreads;
            const int w0 = min(nwords, tid * per), w1 = min(nwords, w0 + per);
            uint32_t mine = 0;
            for (int w = w0; w < w1; ++w) mine += __popc(bmw[w]);
            uint32_t inc = mine;
#pragma unroll
            for (int d = 1; d < 32; d <<= 1) {
                const uint32_t o = __shfl_up_sync(0xFFFFFFFFu, inc, d);
                if (lane >= d) inc += o;
            }
            if (lane == 31) S.wred32[warp] = inc;
            __syncthreads();
            uint32_t wbase = 0, distinct = 0;
            for (int w = 0; w < kWarps; ++w) {
                if (w < warp) wbase += S.wred32[w];
                distinct += S.wred32[w];
            }
            uint32_t run = wbase + inc - mine;
            for (int w = w0; w < w1; ++w) {
                wpw[w] = run;
                run += __popc(bmw[w]);
            }
            for (int q = tid; q < static_cast<int>(distinct); q += kThreads) cnt[q] = 0;
            __syncthreads();
            auto rank_of = [&](int li) {
                return static_cast<int>(wpw[li >> 5] + __popc(bmw[li >> 5] & ((1u << (li & 31)) - 1u)));
            };
            for (int e = tid; e < hn; e += kThreads) {
                const int id = a.hist_ids[hbeg + e];
                if (id >= a0 && id < a1) atomicAdd(&cnt[rank_of(id - a0)], 1u);
            }
            __syncthreads();
            const float rep = P.repetition_penalty, fr = P.frequency_penalty, pr = P.presence_penalty;
            for (int e = tid; e < hn; e += kThreads) {
                const int id = a.hist_ids[hbeg + e];
                if (id >= a0 && id < a1) {
                    const int q = rank_of(id - a0);
                    float z = E::load_scalar(rowp, id);
                    z = (z > 0.0f) ? __fdiv_rn(z, rep) : __fmul_rn(z, rep);
                    z = __fsub_rn(z, __fmul_rn(static_cast<float>(cnt[q]), fr));
                    z = __fsub_rn(z, pr);
                    pat[q] = z;  // duplicates of an id store the same value
                }
            }
            X.bm = bmw;
            X.wp = wpw;
            X.patch = pat;
            X.has_patch = distinct > 0;
        }
    }
    __syncthreads();

    // -------------------------------------------------------------- pass 1: max / argmax
    // Per vector a NaN-propagating max (packed bf16x2 for bf16); vectors with a
    // NaN take the element path.  The NaN-free vector max is cached in vmax[].
    float bv = -INFINITY;
    int bvi = -1;
    bool nanf = false, timeout = false;
    for (int j = 0; j < X.rounds; ++j) {
        if (a.aligned && (j % rpp) == 0) {
            const int p = j / rpp;
            if (piece_v1(p) > p * rpp * kThreads && !mbar_wait_bounded(&S.bar[p], 0)) timeout = true;
        }
        const int v = j * kThreads + tid;
        if (v < X.nv) {
            float vm;
            if (X.vec_patched(v)) {
                float z[VEC];
                X.load(v, z);
                vm = z[0];
#pragma unroll
                for (int e = 1; e < VEC; ++e) vm = fmax_nan(vm, z[e]);
            } else {
                vm = E::vmax_nan(reinterpret_cast<const uint4*>(data)[v]);
            }
            if (vm != vm) {
                nanf = true;
                float z[VEC];
                X.load(v, z);
                vm = -INFINITY;
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (z[e] > vm) vm = z[e];
            }
            X.vmax[v] = vm;
            if (vm > bv) {
                bv = vm;
                bvi = v;
            }
        }
    }
    int bi = -1;
    if (bvi >= 0) {
        float z[VEC];
        X.load(bvi, z);
#pragma unroll
        for (int e = VEC - 1; e >= 0; --e)
            if (z[e] == bv) bi = a0 + bvi * VEC + e;
    }
    X.passes = 1;
    warp_argmax(bv, bi);
    const bool wnan = __any_sync(0xFFFFFFFFu, nanf), wto = __any_sync(0xFFFFFFFFu, timeout);
    if (lane == 0) {
        S.wred[warp] = (static_cast<uint64_t>(static_cast<uint32_t>(bi)) << 32) | __float_as_uint(bv);
        if (wnan) atomicOr(&S.flags, ARC_ERR_NAN);
        if (wto) atomicOr(&S.flags, ARC_ERR_TIMEOUT);
    }
    __syncthreads();
    if (tid == 0) {
        float v = -INFINITY;
        int i = -1;
        for (int w = 0; w < kWarps; ++w)
            better(v, i, __uint_as_float(static_cast<uint32_t>(S.wred[w])), static_cast<int>(S.wred[w] >> 32));
        S.slot[X.par][0] = (static_cast<uint64_t>(static_cast<uint32_t>(i)) << 32) | __float_as_uint(v);
        S.slot[X.par][1] = S.flags & (ARC_ERR_NAN | ARC_ERR_TIMEOUT);
    }
    X.xsync();
    float m;
    int am;
    uint32_t dflags;
    {
        float v = -INFINITY;
        int i = -1;
        uint32_t f = 0;
        if (lane < X.s) {
            const uint64_t x = X.xread(lane, 0);
            v = __uint_as_float(static_cast<uint32_t>(x));
            i = static_cast<int>(x >> 32);
            f = static_cast<uint32_t>(X.xread(lane, 1));
        }
        warp_argmax(v, i);
        m = v;
        am = i;
        dflags = __reduce_or_sync(0xFFFFFFFFu, f);
    }
    X.xnext();
    X.row_nan = (dflags & ARC_ERR_NAN) != 0;
    if ((a.flags & ARC_OPT_STEP_AUTOINC) && X.rank == 0 && tid == 0) a.params[row].step = P.step + 1;

    // -------------------------------------------------------------- mode
    uint32_t err = rerr | dflags;
    const float T = P.temperature;
    const int k = P.top_k;
    const bool topk_on = k >= 1 && k < a.V;
    const bool topp_on = P.top_p < 1.0f;
    const bool minp_on = P.min_p > 0.0f;
    int mode;
    int token = -2;  // -2: decided by the draw
    if (rerr != 0 || (dflags & ARC_ERR_TIMEOUT)) {
        mode = -1;
        token = -1;
    } else {
        mode = (T == 0.0f || k == 1) ? 0 : ((!topk_on && !topp_on && !minp_on) ? 1 : 2);
        if (am < 0) {
            token = 0;
            err |= ARC_ERR_DEGENERATE;
        } else if (mode == 0) {
            token = am;
        }
    }

    uint32_t kap_k = 0, kap_r = 0;
    int iot_k = a.V, iot_r = a.V;
    uint64_t mass_k = 0, mass_r = 0, target = 0, rbits = 0;
    bool walk_fail = false;

    if (token != -2) {
        cluster_arrive();  // this CTA reads no other CTA's shared memory after this
    } else {
        // ---------------------------------------------------------- sampling rows
        X.m = m;
        X.infm = (m == INFINITY);
        X.c = __fdiv_rn(1.4426950408889634f, T);  // w = 2^((z - m) * log2(e) / T)
        X.scale = __uint_as_float(static_cast<uint32_t>(127 + a.F) << 23);
        const uint32_t Km = fkey(m);
        // per-row fp64 thresholds, one lane per warp:
        //   zm: min-p, w >= min_p  <=>  z >= m + T ln(min_p), rounded up to fp32
        //   zb: top-p window floor; ids below it carry < half of (1 - top_p) of the mass
        float zm = -INFINITY, zb = -INFINITY;
        if (lane == 0) {
            if (minp_on)
                zm = __double2float_ru(static_cast<double>(m) +
                                       static_cast<double>(T) * log(static_cast<double>(P.min_p)));
            if (topp_on)
                zb = __double2float_rd(static_cast<double>(m) +
                                       static_cast<double>(T) * log((1.0 - static_cast<double>(P.top_p)) /
                                                                    (2.0 * static_cast<double>(a.V))));
        }
        zm = __shfl_sync(0xFFFFFFFFu, zm, 0);
        zb = __shfl_sync(0xFFFFFFFFu, zb, 0);

        Surv K{-INFINITY, INT_MAX};  // every non-NaN id
        if (topk_on) {
            K = select_topk(X, k, Km, err);
            kap_k = (K.zt == -INFINITY && K.ge_form()) ? 0u : fkey(K.zt);
            iot_k = K.ge_form() ? a.V : K.iota;
        }
        Surv R = K;
        bool wsum_is_R = false;
        if (topp_on) {
            // masses over K, plus the mass histogram of a key window that holds
            // the top-p cutoff
            const float zfloor = fmaxf(zm, K.zt);
            float zlo = fmaxf(zb, zfloor);
            Window W = Ctx::make_window(fkey(zlo), Km);
            const int mk = mass_mode(X, K);
            pass_mass<Ctx, true>(X, mk, K, W);
            X.publish_wsum_total(0);
            X.push_hist();
            X.xsync();
            mass_k = X.xscan(0, ~0ull).total;
            X.xnext();
            uint64_t tgt = 1;
            if (lane == 0)
                tgt = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(mass_k)));
            tgt = shfl_u64(tgt, 0);
            if (tgt == 0) tgt = 1;
            float zp = -INFINITY;
            bool found = select_mass(X, W, K, tgt, zp);
            if (!found && zlo > zfloor) {
                // rounding left the first window just short: retry down to the hard bound
                zlo = zfloor;
                W = Ctx::make_window(fkey(zlo), Km);
                pass_hist<Ctx, true>(X, W, K);
                X.push_hist();
                X.xsync();
                found = select_mass(X, W, K, tgt, zp);
            }
            // short of the target even then: min-p (or top-k) bounds the window,
            // so the top-p cutoff lies below every id those filters keep
            const float zx = found ? fmaxf(zp, zm) : zm;
            if (zx > K.zt)
                R = Surv{zx, INT_MAX};
            else
                wsum_is_R = true;
        } else if (minp_on && zm > K.zt) {
            R = Surv{zm, INT_MAX};
        }
        kap_r = (R.zt == -INFINITY && R.ge_form()) ? 0u : fkey(R.zt);
        iot_r = R.ge_form() ? a.V : R.iota;

        // ---------------------------------------------------------- inverse-CDF draw
        const int mr = mass_mode(X, R);
        if (!wsum_is_R) pass_mass<Ctx, false>(X, mr, R, Window{0u, 0u, 0});
        X.publish_wsum_total(0);
        rbits = splitmix64(P.seed ^ (static_cast<uint64_t>(row) << 32) ^ P.step) >> 11;
        X.xsync();
        mass_r = X.xscan(0, ~0ull).total;
        target = scale_by_u(rbits, mass_r);
        const typename Ctx::Scan sc = X.xscan(0, target);
        X.xnext();
        cluster_arrive();  // this CTA reads no other CTA's shared memory after this
        if (sc.first < 0) {
            err |= kErrInternal;
            token = am;
        } else if (sc.first == X.rank) {
            const uint64_t t = target - sc.before_me;
            int tok = X.walk(
                t, [&](const float(&z)[VEC], int g0) { return X.vec_mass(mr, z, g0, R); },
                [&](const float(&z)[VEC], int g0, uint64_t tt) { return X.vec_mass_walk(mr, z, g0, R, tt); });
            if (tok < 0) {
                tok = am;
                walk_fail = true;
            }
            if (tid == 0) {
                a.out[row] = tok;
                if (a.debug) a.debug[row].token = tok;
            }
        }
    }

    // -------------------------------------------------------------- results
    if (X.rank == 0 && tid == 0) {
        if (token != -2) a.out[row] = token;
        if (err != 0 && a.err_word) atomicOr(a.err_word, err);
        if (a.debug) {
            arc_row_debug& d = a.debug[row];
            d.mode = mode;
            d.err = err;
            if (token != -2) d.token = token;
            d.passes = X.passes;
            d.kappa_k = kap_k;
            d.iota_k = iot_k;
            d.kappa_r = kap_r;
            d.iota_r = iot_r;
            d.max_z = m;
            d.frac_bits = a.F;
            d.rbits = rbits;
            d.mass_k = mass_k;
            d.mass_r = mass_r;
            d.target = target;
        }
    }
    // no CTA may leave while another can still read its shared memory
    cluster_wait();
    if (walk_fail && tid == 0) {
        if (a.err_word) atomicOr(a.err_word, kErrInternal);
        if (a.debug) atomicOr(&a.debug[row].err, kErrInternal);
    }
    if (timeout && a.aligned) {
        // give bulk copies still in flight a bounded chance to land before exit
        for (int p = 0; p < kPieces; ++p)
            if (piece_v1(p) > p * rpp * kThreads) (void)mbar_wait_bounded(&S.bar[p], 0);
    }
}

}  // namespace arc
