// Exact selection over a row by multi-way threshold bisection: the path the
// finish kernel falls back to when the floor from the chunk maxima admits too
// many ids (flat or heavily tied rows, top-p alone on diffuse rows).
//
// The row is read from global memory (or shared memory, for a slice staged
// there); a per-chunk (or per-vector) max table lets every pass skip the
// chunks that cannot hold an id at or above the pass's threshold.
//
// Thresholds are found on the order-preserving u32 key of the logit: a
// 512-bin histogram of the keys in a window below the row max locates the bin
// that crosses the target count (top-k) or mass (top-p); the few ids in that
// bin are gathered and ranked exactly.  Bins that hold too many ids are
// bisected further, 9 bits per pass; ties at a top-k boundary too many to
// gather are resolved by an id-order count walk.
//
// The helpers are written for a thread-block cluster of s CTAs sharing one
// row, each with a contiguous part of it (partials exchanged through
// distributed shared memory, decisions taken identically by every CTA): the
// finish kernel uses them with its cluster of CTAs per row (s = 1 for large
// batches, up to 8 when the batch leaves SMs idle).
//
// Masses are fixed-point integers (units of 2^-F of the max weight), so sums
// are exact, associative and identical in every pass.
#pragma once

#include <climits>

#include "arc_device.cuh"

namespace arc {

// The local histogram keeps each bin's 64-bit sum as two 32-bit words updated
// with native 32-bit shared atomics (a 64-bit shared atomic add is a
// compare-and-swap loop, which heavy ties turn into long retry chains): the
// low word adds the low half, and the high word the high half plus one for
// every add that wrapped the low word, so the sum is exact in any order.

struct __align__(16) SampleShared {
    uint32_t lhist[kBins * 2];  // this CTA's histogram: bin b's sum is lhist[2b] + 2^32 lhist[2b + 1]
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
constexpr int kBatch = 8;  // rounds whose loads a pass issues together

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
    int v0;                     // the row's vector index of this CTA's first vector (a0 / VEC)
    const unsigned char* data;  // the slice: shared memory, or global memory when src_global
    bool src_global;
    bool src_aligned;
    float* vmax;                // max per vector (vps == 0) or per 32-vector chunk, or nullptr
    int vps;                    // vectors per slice of the chunk table (0: vmax is per vector)
    int cps;                    // chunk slots per slice
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
        const int l0 = (v0 + v) * VEC;
        return ((bm[l0 >> 5] >> (l0 & 31)) & ((1u << VEC) - 1u)) != 0;
    }

    __device__ __forceinline__ uint4 raw_vec(int v) const {
        return src_global ? E::global_vec(data, v, n, src_aligned) : reinterpret_cast<const uint4*>(data)[v];
    }
    // false only when vector v cannot hold an id >= thr
    __device__ __forceinline__ bool may_hold(int v, float thr) const {
        if (vmax == nullptr) return true;
        if (vps == 0) return vmax[v] >= thr;
        const int gv = v0 + v;  // the table is the whole row's
        const int c = gv / vps;
        return vmax[c * cps + ((gv - c * vps) >> 5)] >= thr;
    }

    __device__ __forceinline__ void load(int v, float (&z)[VEC]) const { unpack_patched(v, raw_vec(v), z); }

    // vector v's logits from its raw 16 bytes, history penalties applied
    __device__ __forceinline__ void unpack_patched(int v, const uint4& raw, float (&z)[VEC]) const {
        E::unpack(raw, z);
        if (HIST && has_patch) {
            const int l0 = (v0 + v) * VEC;  // the patch tables are the whole row's
            const uint32_t word = bm[l0 >> 5];
            const uint32_t bits = (word >> (l0 & 31)) & ((1u << VEC) - 1u);
            if (bits) {
                const int base = patch_word_base(bm, wp, l0 >> 5);
#pragma unroll
                for (int e = 0; e < VEC; ++e) {
                    const int li = l0 + e;
                    if ((bits >> e) & 1u) z[e] = patch[base + __popc(word & ((1u << (li & 31)) - 1u))];
                }
            }
        }
    }

    // One pass over this thread's vectors v = j * kThreads + tid, j < rounds:
    // the loads of kBatch rounds go out together (a pass over a row in global
    // memory costs rounds / kBatch round trips, not rounds).  body(j, v, z)
    // runs for the vectors with want(v); end(j) runs after round j in every
    // thread (uniform, so it may hold warp collectives).
    template <class Want, class Body, class End>
    __device__ __forceinline__ void batched_pass(Want want, Body body, End end) const {
        for (int j0 = 0; j0 < rounds; j0 += kBatch) {
            uint4 raw[kBatch];
            bool ok[kBatch];
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                const int v = (j0 + u) * kThreads + tid;
                ok[u] = (j0 + u) < rounds && v < nv && want(v);
                if (ok[u]) raw[u] = raw_vec(v);
            }
#pragma unroll
            for (int u = 0; u < kBatch; ++u) {
                if (j0 + u < rounds) {
                    const int v = (j0 + u) * kThreads + tid;
                    if (ok[u]) {
                        float z[VEC];
                        unpack_patched(v, raw[u], z);
                        body(j0 + u, v, z);
                    }
                    end(j0 + u);
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
        if (s == 1)
            __syncthreads();  // one CTA: every exchange stays in its own shared memory
        else
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
        uint32_t* h = &S.lhist[((W.khi - k) >> W.sh) * 2];
        const uint32_t lo = static_cast<uint32_t>(wt), hi = static_cast<uint32_t>(wt >> 32);
        const uint32_t old = atomicAdd(h, lo);
        const uint32_t carry = (old + lo < old) ? 1u : 0u;
        if (hi + carry) atomicAdd(h + 1, hi + carry);
    }
    __device__ __forceinline__ uint64_t lhist_bin(int b) const {
        return (static_cast<uint64_t>(S.lhist[2 * b + 1]) << 32) | S.lhist[2 * b];
    }

    __device__ __forceinline__ void lhist_clear() {
        for (int b = tid; b < kBins * 2; b += kThreads) S.lhist[b] = 0;
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
            const uint64_t v = lhist_bin(b);
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

// The parameter record from its six 64-bit words.
__device__ __forceinline__ arc_row_params params_from_words(const uint64_t (&w)[6]) {
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
    X.batched_pass([&](int v) { return X.may_hold(v, thr); },
                   [&](int, int v, const float(&z)[VEC]) {
                       const int g0 = X.a0 + v * VEC;
#pragma unroll
                       for (int e = 0; e < VEC; ++e)
                           if (z[e] >= zlo && z[e] <= zhi && D.test(z[e], g0 + e))
                               X.lhist_add(W, fkey(z[e]), MASS ? X.fix(X.weight(z[e])) : 1u);
                   },
                   [](int) {});
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
    X.batched_pass([&](int v) { return X.may_hold(v, thr); },
                   [&](int, int v, const float(&z)[VEC]) {
                       const int g0 = X.a0 + v * VEC;
#pragma unroll
                       for (int e = 0; e < VEC; ++e) {
                           if (z[e] >= zlo && z[e] <= zhi && D.test(z[e], g0 + e)) {
                               const uint32_t k = fkey(z[e]);
                               if (k >= lo && k <= hi)
                                   X.push_cand(k, MASS ? X.fix(X.weight(z[e])) : static_cast<uint64_t>(g0 + e));
                           }
                       }
                   },
                   [](int) {});
    X.passes++;
}

// Per-(round, warp) fixed-point masses of the survivors of D into Wsum; with
// HISTO also the local mass histogram of the survivors whose keys lie in W.
template <class Ctx, bool HISTO>
__device__ void pass_mass(Ctx& X, int mode, const Surv& D, const Window& W) {
    constexpr int VEC = Ctx::VEC;
    if (HISTO) X.lhist_clear();
    const float zlo = Ctx::lo_float(W.klo), zhi = key_to_float(W.khi);
    uint64_t q = 0;
    X.batched_pass([&](int v) { return mode == kAll || X.may_hold(v, D.zt); },
                   [&](int, int v, const float(&z)[VEC]) {
                       const int g0 = X.a0 + v * VEC;
                       q = X.vec_mass(mode, z, g0, D);
                       if (HISTO && X.may_hold(v, zlo)) {
#pragma unroll
                           for (int e = 0; e < VEC; ++e)
                               if (z[e] >= zlo && z[e] <= zhi && Ctx::in_domain(mode, D, z[e], g0 + e))
                                   X.lhist_add(W, fkey(z[e]), X.fix(X.weight(z[e])));
                       }
                   },
                   [&](int j) {
                       const uint64_t t = warp_sum_u64(q);
                       if (X.lane == 0) X.Wsum[j * kWarps + X.warp] = t;
                       q = 0;
                   });
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
    uint64_t q = 0;
    X.batched_pass([&](int v) { return X.may_hold(v, zt); },
                   [&](int, int, const float(&z)[VEC]) {
#pragma unroll
                       for (int e = 0; e < VEC; ++e) q += (z[e] == zt) ? 1u : 0u;
                   },
                   [&](int j) {
                       const uint64_t t = warp_sum_u64(q);
                       if (X.lane == 0) X.Wsum[j * kWarps + X.warp] = t;
                       q = 0;
                   });
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

// Exact top-k survivor set: the first k ids by (z desc, id asc).  zhint, when
// finite, is a known lower bound of the k-th largest logit: the first window
// starts there.
template <class Ctx>
__device__ Surv select_topk(Ctx& X, int k, uint32_t Km, uint32_t& err, float zhint = -INFINITY) {
    const Surv all{-INFINITY, INT_MAX};
    uint64_t tgt = static_cast<uint64_t>(k);
    // first window: from the hint, else 2^23 keys (one binade) below the max,
    // widened 16x while it holds fewer than k ids
    uint32_t width = 1u << 23;
    const bool hinted = zhint > -INFINITY && zhint <= key_to_float(Km);
    Window W = hinted ? Ctx::make_window(fkey(zhint), Km)
                      : Ctx::make_window(Km > width - 1 ? Km - (width - 1) : 0u, Km);
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
        // no id in the bin weighs more than its top key: a bin whose mass is
        // above kCand such weights holds more ids than a gather keeps (a run
        // of ties, typically), so it is bisected without gathering
        const uint64_t wtop = X.fix(X.weight(key_to_float(hi)));
        const bool too_many = wtop == 0 || r.inbin / wtop > static_cast<uint64_t>(kCand);
        // gather the bin's ids (key, mass) into every CTA and find the largest
        // key whose mass at or above it reaches the target
        uint32_t got = UINT32_MAX;
        if (!too_many) {
            pass_collect<Ctx, true>(X, lo, hi, K);
            X.xsync();
            got = X.S.ccount;
        }
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
        if (!too_many) X.cand_clear();
        W.klo = lo;
        W.khi = hi;
        W.sh = max(0, W.sh - kBinBits);
        pass_hist<Ctx, true>(X, W, K);
        X.push_hist();
        X.xsync();
    }
}

}  // namespace arc
