// Fused per-row sampling kernel: one thread-block cluster of s CTAs per row.
//
// Each CTA bulk-copies (TMA, cp.async.bulk) its contiguous slice of the row
// into shared memory once; every later look at the row -- max, top-k select,
// top-p select, masses, the inverse-CDF walk -- runs out of shared memory.
// CTAs of a row combine partial results through distributed shared memory
// (DSMEM) and cluster barriers; every decision is computed redundantly and
// identically by all CTAs, so control flow stays uniform across the cluster.
//
// Thresholds are found by multi-way threshold bisection on the order-
// preserving u32 key of the logit: a 1024-bin histogram over a key window
// below the row max narrows the window by 10 bits per pass until the bin that
// crosses the target count (top-k) or target mass (top-p) holds one key.
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
    int data_bytes;  // bytes reserved for the slice in dynamic shared memory
    int rounds_max;  // rounds of the largest slice
    int hist_cap;    // history entries per row (patch table capacity)
    int F;           // fixed-point fraction bits
    uint32_t flags;  // ARC_OPT_*
    int aligned;     // rows start on 16-byte boundaries: bulk copies allowed
};

struct __align__(16) SampleShared {
    uint64_t bar[kPieces];
    uint64_t hist[kBins];
    uint64_t seg[kBins / 2];
    uint64_t slot[2][8];
    uint64_t wred[kWarps];
    uint64_t bcast_u[4];
    int bcast_i[4];
    uint32_t wred32[kWarps];
    uint32_t mm[2];
    uint32_t flags;
};

// internal error bit: a search that exact integer arithmetic guarantees failed
constexpr uint32_t kErrInternal = 0x40u;

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

template <int DT, bool HIST>
struct RowCtx {
    using E = Elem<DT>;
    static constexpr int VEC = E::kVec;

    SampleShared& S;
    cg::cluster_group cl;
    int s, rank, row, tid, lane, warp;
    int a0, a1, n, nv, nvf, rounds;
    const unsigned char* data;
    uint64_t* Wsum;
    // history patches
    const uint32_t* bm;
    const uint32_t* wp;
    const float* patch;
    bool has_patch;
    // weights: w = ex2((z - m) * c), or [z == m] when m = +inf
    float m, c, scale;
    bool infm;
    int par;      // exchange ring parity
    int passes;

    __device__ RowCtx(SampleShared& S_, cg::cluster_group cl_) : S(S_), cl(cl_) {}

    // ---------------------------------------------------------------- loads
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

    // fixed-point mass of the survivors of one vector (fp32 sum in id order, then rounded)
    template <bool TIE>
    __device__ __forceinline__ uint64_t vec_mass(const float (&z)[VEC], int g0, const Surv& d) const {
        bool in[VEC];
        bool any = false;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            in[e] = TIE ? d.test(z[e], g0 + e) : (z[e] >= d.zt);
            any |= in[e];
        }
        if (!any) return 0;
        float sum = 0.0f;
#pragma unroll
        for (int e = 0; e < VEC; ++e)
            if (in[e]) sum = __fadd_rn(sum, weight(z[e]));
        return fix(sum);
    }

    // first element of the vector whose running fixed-point mass exceeds t
    template <bool TIE>
    __device__ __forceinline__ int vec_mass_walk(const float (&z)[VEC], int g0, const Surv& d,
                                                 uint64_t t) const {
        float sum = 0.0f;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            const bool in = TIE ? d.test(z[e], g0 + e) : (z[e] >= d.zt);
            if (in) sum = __fadd_rn(sum, weight(z[e]));
            if (fix(sum) > t) return e;
        }
        return -1;
    }

    __device__ __forceinline__ static uint64_t vec_count_eq(const float (&z)[VEC], float zt) {
        uint64_t c = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) c += (z[e] == zt) ? 1u : 0u;
        return c;
    }

    __device__ __forceinline__ static int vec_count_walk(const float (&z)[VEC], float zt, uint64_t t) {
        uint64_t c = 0;
#pragma unroll
        for (int e = 0; e < VEC; ++e) {
            c += (z[e] == zt) ? 1u : 0u;
            if (c > t) return e;
        }
        return -1;
    }

    // ---------------------------------------------------------------- cluster exchange
    // Thread 0 wrote S.slot[par][*]; after sync every CTA reads every rank's slot.
    __device__ __forceinline__ void xsync() { cl.sync(); }
    __device__ __forceinline__ uint64_t xread(int r, int i) const {
        return cl.map_shared_rank(&S.slot[par][0], r)[i];
    }
    __device__ __forceinline__ void xnext() { par ^= 1; }

    // Sum of a per-CTA value over the cluster plus the exclusive prefix of
    // this CTA and the first rank whose inclusive prefix exceeds t (or -1).
    struct Scan {
        uint64_t total, before_me;
        int first;
        uint64_t before_first;
    };
    __device__ __forceinline__ Scan xscan(int i, uint64_t t) const {
        uint64_t x = (lane < s) ? xread(lane, i) : 0;
        const uint64_t inc = warp_inclusive_u64(x);
        Scan r;
        r.total = shfl_u64(inc, 31);
        r.before_me = shfl_u64(inc - x, rank);
        const unsigned bal = __ballot_sync(0xFFFFFFFFu, lane < s && inc > t);
        r.first = bal ? __ffs(bal) - 1 : -1;
        r.before_first = bal ? shfl_u64(inc - x, r.first) : 0;
        return r;
    }

    // Total of Wsum[0 .. rounds*kWarps) of this CTA into slot i (thread 0 of warp 0).
    __device__ __forceinline__ void publish_wsum_total(int i) {
        __syncthreads();
        if (warp == 0) {
            uint64_t acc = 0;
            for (int e = lane; e < rounds * kWarps; e += 32) acc += Wsum[e];
            acc = warp_sum_u64(acc);
            if (lane == 0) S.slot[par][i] = acc;
        }
    }

    // warp-level search of arr[0..n) (generic pointer, may be remote) for the
    // first position whose inclusive prefix exceeds t.  All lanes get the result.
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
    }

    // ---------------------------------------------------------------- histogram select
    struct Window {
        uint32_t klo, khi;
        int sh;
    };
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

    // Adds `wt` to the bin of key `k` if it lies in the window.
    __device__ __forceinline__ void hist_add(const Window& W, uint32_t k, uint64_t wt, bool track) {
        if (k < W.klo || k > W.khi) return;
        atomicAdd(reinterpret_cast<unsigned long long*>(&S.hist[(W.khi - k) >> W.sh]),
                  static_cast<unsigned long long>(wt));
        if (track) {
            atomicMin(&S.mm[0], k);
            atomicMax(&S.mm[1], k);
        }
    }

    __device__ __forceinline__ void hist_clear() {
        for (int b = tid; b < kBins; b += kThreads) S.hist[b] = 0;
        if (tid == 0) {
            S.mm[0] = 0xFFFFFFFFu;
            S.mm[1] = 0u;
        }
        __syncthreads();
    }

    struct Sel {
        int bin;          // crossing bin (-1: window total does not reach the target)
        uint64_t before;  // weight in bins above it
        uint64_t inbin;   // weight in it
        uint64_t total;   // weight in the window
        uint32_t mmin, mmax;
    };

    // Combine the CTAs' histograms and find the first bin whose inclusive
    // prefix (from the top key down) reaches target (>= target).
    __device__ Sel hist_exchange(uint64_t target) {
        Sel r;
        const int segsz = kBins / s;
        uint64_t* segp = (s == 1) ? S.hist : S.seg;
        xsync();  // A: histograms complete in every CTA
        uint64_t part = 0;
        if (s > 1) {
            const int b0 = rank * segsz;
            for (int b = tid; b < segsz; b += kThreads) {
                uint64_t acc = 0;
                for (int q = 0; q < s; ++q) acc += cl.map_shared_rank(S.hist, q)[b0 + b];
                S.seg[b] = acc;
                part += acc;
            }
        } else {
            for (int b = tid; b < segsz; b += kThreads) part += S.hist[b];
        }
        part = warp_sum_u64(part);
        if (lane == 0) S.wred[warp] = part;
        __syncthreads();
        if (tid == 0) {
            uint64_t tot = 0;
            for (int w = 0; w < kWarps; ++w) tot += S.wred[w];
            S.slot[par][0] = tot;
            S.slot[par][1] = S.mm[0];
            S.slot[par][2] = S.mm[1];
        }
        xsync();  // B: segments combined
        const Scan sc = xscan(0, target - 1);
        uint32_t mn = (lane < s) ? static_cast<uint32_t>(xread(lane, 1)) : 0xFFFFFFFFu;
        uint32_t mx = (lane < s) ? static_cast<uint32_t>(xread(lane, 2)) : 0u;
        mn = __reduce_min_sync(0xFFFFFFFFu, mn);
        mx = __reduce_max_sync(0xFFFFFFFFu, mx);
        r.total = sc.total;
        r.mmin = mn;
        r.mmax = mx;
        r.bin = -1;
        r.before = r.inbin = 0;
        if (sc.first >= 0) {
            if (warp == 0) {
                const uint64_t* remote = cl.map_shared_rank(segp, sc.first);
                int pos;
                uint64_t bf, val;
                warp_find(remote, segsz, target - 1 - sc.before_first, pos, bf, val);
                if (lane == 0) {
                    S.bcast_i[0] = pos < 0 ? -1 : sc.first * segsz + pos;
                    S.bcast_u[0] = sc.before_first + bf;
                    S.bcast_u[1] = val;
                }
            }
            __syncthreads();
            r.bin = S.bcast_i[0];
            r.before = S.bcast_u[0];
            r.inbin = S.bcast_u[1];
            __syncthreads();
        }
        xnext();
        return r;
    }

    // ---------------------------------------------------------------- index-order walk
    // In CTA `owner`, find the element whose running weight (in id order over
    // this CTA's Wsum chunks) first exceeds t.  Returns the row index or -1.
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

// Key range [bin_lo, bin_hi] of histogram bin `b` of window W.
template <class Ctx>
__device__ __forceinline__ void bin_range(const typename Ctx::Window& W, int b, uint32_t& lo, uint32_t& hi) {
    hi = W.khi - (static_cast<uint32_t>(b) << W.sh);
    int64_t lo64 = static_cast<int64_t>(hi) - ((int64_t{1} << W.sh) - 1);
    if (lo64 < static_cast<int64_t>(W.klo)) lo64 = static_cast<int64_t>(W.klo);
    lo = static_cast<uint32_t>(lo64);
}

// Count histogram of the keys in window W (every non-NaN id).
template <class Ctx>
__device__ void pass_count_hist(Ctx& X, const typename Ctx::Window& W, bool track) {
    constexpr int VEC = Ctx::VEC;
    X.hist_clear();
    const float zlo = Ctx::lo_float(W.klo), zhi = key_to_float(W.khi);
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        if (v < X.nv) {
            float z[VEC];
            X.load(v, z);
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (z[e] >= zlo && z[e] <= zhi) X.hist_add(W, fkey(z[e]), 1, track);
        }
    }
    X.passes++;
    __syncthreads();
}

// Mass histogram of the ids of K whose keys lie in window W.
template <class Ctx>
__device__ void pass_mass_hist(Ctx& X, const typename Ctx::Window& W, const Surv& K, bool track) {
    constexpr int VEC = Ctx::VEC;
    X.hist_clear();
    const float zlo = Ctx::lo_float(W.klo), zhi = key_to_float(W.khi);
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        if (v < X.nv) {
            float z[VEC];
            X.load(v, z);
            const int g0 = X.a0 + v * VEC;
#pragma unroll
            for (int e = 0; e < VEC; ++e)
                if (z[e] >= zlo && z[e] <= zhi && (K.ge_form() || K.test(z[e], g0 + e)))
                    X.hist_add(W, fkey(z[e]), X.fix(X.weight(z[e])), track);
        }
    }
    X.passes++;
    __syncthreads();
}

// Per-(round, warp) fixed-point masses of the survivors of D into Wsum; when
// W is given, also the mass histogram of the survivors in that key window.
template <class Ctx, bool TIE, bool WITH_HIST>
__device__ void pass_mass(Ctx& X, const Surv& D, const typename Ctx::Window& W) {
    constexpr int VEC = Ctx::VEC;
    if (WITH_HIST) X.hist_clear();
    const float zlo = Ctx::lo_float(W.klo), zhi = key_to_float(W.khi);
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        uint64_t q = 0;
        if (v < X.nv) {
            float z[VEC];
            X.load(v, z);
            const int g0 = X.a0 + v * VEC;
            q = X.template vec_mass<TIE>(z, g0, D);
            if (WITH_HIST) {
#pragma unroll
                for (int e = 0; e < VEC; ++e)
                    if (z[e] >= zlo && z[e] <= zhi && (!TIE || D.test(z[e], g0 + e)))
                        X.hist_add(W, fkey(z[e]), X.fix(X.weight(z[e])), false);
            }
        }
        q = warp_sum_u64(q);
        if (X.lane == 0) X.Wsum[j * kWarps + X.warp] = q;
    }
    X.passes++;
}

template <class Ctx>
__device__ __forceinline__ void pass_mass_any(Ctx& X, const Surv& D) {
    typename Ctx::Window W{0u, 0u, 0};
    if (D.ge_form())
        pass_mass<Ctx, false, false>(X, D, W);
    else
        pass_mass<Ctx, true, false>(X, D, W);
}

// top-k survivor set: the first k ids by (z desc, id asc).  Exact.
template <class Ctx>
__device__ Surv select_topk(Ctx& X, int k, uint32_t Km, uint32_t& err) {
    constexpr int VEC = Ctx::VEC;
    using Window = typename Ctx::Window;
    uint64_t tgt = static_cast<uint64_t>(k);
    // first window: 2^23 keys (one binade) below the max, widened 16x while it
    // holds fewer than k ids
    uint32_t width = 1u << 23;
    Window W = Ctx::make_window(Km > width - 1 ? Km - (width - 1) : 0u, Km);
    int level = 0;
    float zt = -INFINITY;
    bool tie = false;
    while (true) {
        pass_count_hist(X, W, level > 0);
        const typename Ctx::Sel r = X.hist_exchange(tgt);
        if (r.bin < 0) {
            if (level == 0 && W.klo > 0) {
                width = (width >= (1u << 27)) ? 0u : (width << 4);
                const uint32_t lo = (width == 0u || Km < width - 1) ? 0u : Km - (width - 1);
                W = Ctx::make_window(lo, Km);
                continue;
            }
            return Surv{-INFINITY, INT_MAX};  // fewer than k non-NaN ids: keep all
        }
        if (level > 0 && r.mmin == r.mmax) {
            // the window (the previous crossing bin) holds one key
            zt = key_to_float(r.mmin);
            if (tgt == r.total) return Surv{zt, INT_MAX};
            tie = true;
            break;
        }
        uint32_t lo, hi;
        bin_range<Ctx>(W, r.bin, lo, hi);
        if (r.before + r.inbin == tgt) return Surv{Ctx::lo_float(lo), INT_MAX};
        tgt -= r.before;
        if (W.sh == 0) {
            zt = key_to_float(hi);
            tie = true;
            break;
        }
        W.klo = lo;
        W.khi = hi;
        W.sh = max(0, W.sh - kBinBits);
        level++;
    }
    (void)tie;
    // keep the first `tgt` ids (in id order) tied at zt: find the tgt-th one
    for (int j = 0; j < X.rounds; ++j) {
        const int v = j * kThreads + X.tid;
        uint64_t q = 0;
        if (v < X.nv) {
            float z[VEC];
            X.load(v, z);
            q = Ctx::vec_count_eq(z, zt);
        }
        q = warp_sum_u64(q);
        if (X.lane == 0) X.Wsum[j * kWarps + X.warp] = q;
    }
    X.passes++;
    X.publish_wsum_total(0);
    X.xsync();
    const typename Ctx::Scan sc = X.xscan(0, tgt - 1);
    X.xnext();
    if (sc.first == X.rank) {
        const int pos = X.walk(
            tgt - 1 - sc.before_me, [&](const float(&z)[VEC], int) { return Ctx::vec_count_eq(z, zt); },
            [&](const float(&z)[VEC], int, uint64_t t) { return Ctx::vec_count_walk(z, zt, t); });
        if (X.tid == 0) X.S.slot[X.par][0] = static_cast<uint64_t>(static_cast<uint32_t>(pos));
    }
    X.xsync();
    const int pos = (sc.first >= 0) ? static_cast<int>(static_cast<uint32_t>(X.xread(sc.first, 0))) : -1;
    X.xnext();
    if (pos < 0) {
        err |= kErrInternal;
        return Surv{zt, INT_MAX};
    }
    return Surv{zt, pos + 1};
}

// Continue a mass select from a window whose histogram is built: returns
// true and the cutoff zp (z >= zp survives) when the window reaches `tgt`.
template <class Ctx>
__device__ bool select_mass(Ctx& X, typename Ctx::Window W, const Surv& K, uint64_t tgt, float& zp) {
    int level = 0;
    while (true) {
        const typename Ctx::Sel r = X.hist_exchange(tgt);
        if (r.bin < 0) return false;
        if (level > 0 && r.mmin == r.mmax) {
            zp = key_to_float(r.mmin);
            return true;
        }
        uint32_t lo, hi;
        bin_range<Ctx>(W, r.bin, lo, hi);
        if (W.sh == 0) {
            zp = key_to_float(hi);
            return true;
        }
        if (r.before + r.inbin == tgt) {
            zp = Ctx::lo_float(lo);
            return true;
        }
        tgt -= r.before;
        W.klo = lo;
        W.khi = hi;
        W.sh = max(0, W.sh - kBinBits);
        level++;
        pass_mass_hist(X, W, K, true);
    }
}

template <int DT, bool HIST>
__global__ void __launch_bounds__(kThreads) sample_kernel(const SampleArgs a) {
    using Ctx = RowCtx<DT, HIST>;
    using E = Elem<DT>;
    using Window = typename Ctx::Window;
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
    X.Wsum = reinterpret_cast<uint64_t*>(dyn + a.data_bytes);
    X.par = 0;
    X.passes = 0;
    X.has_patch = false;
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
    }
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
    // rows are not 16-byte aligned.  The last vector is padded with NaN, which
    // no predicate, maximum or weight ever selects.
    {
        const int first = a.aligned ? X.nvf * VEC : 0;
        for (int i = first + tid; i < X.nv * VEC; i += kThreads) {
            if (i < n)
                E::store_smem_raw(data, i, rowp, a0 + i);
            else if (DT == ARC_BF16)
                reinterpret_cast<unsigned short*>(data)[i] = 0x7FC0;
            else
                reinterpret_cast<uint32_t*>(data)[i] = 0x7FC00000u;
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
            uint32_t* bmw = reinterpret_cast<uint32_t*>(dyn + a.data_bytes + a.rounds_max * kWarps * 8);
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
    float bv = -INFINITY;
    int bi = -1;
    bool nanf = false, timeout = false;
    for (int j = 0; j < X.rounds; ++j) {
        if (a.aligned && (j % rpp) == 0) {
            const int p = j / rpp;
            if (piece_v1(p) > p * rpp * kThreads && !mbar_wait_bounded(&S.bar[p], 0)) timeout = true;
        }
        const int v = j * kThreads + tid;
        if (v < X.nv) {
            float z[VEC];
            X.load(v, z);
#pragma unroll
            for (int e = 0; e < VEC; ++e) {
                if (v * VEC + e < n) nanf |= (z[e] != z[e]);
                if (z[e] > bv) {
                    bv = z[e];
                    bi = a0 + v * VEC + e;
                }
            }
        }
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

    if (token == -2) {
        // ---------------------------------------------------------- sampling rows
        X.m = m;
        X.infm = (m == INFINITY);
        X.c = __fdiv_rn(1.4426950408889634f, T);  // w = 2^((z - m) * log2(e) / T)
        X.scale = __uint_as_float(static_cast<uint32_t>(127 + a.F) << 23);
        const uint32_t Km = fkey(m);
        Surv K{-INFINITY, INT_MAX};  // every non-NaN id
        if (topk_on) {
            K = select_topk(X, k, Km, err);
            kap_k = (K.zt == -INFINITY && K.ge_form()) ? 0u : fkey(K.zt);
            iot_k = K.ge_form() ? a.V : K.iota;
        }
        // min-p: w >= min_p  <=>  z >= m + T ln(min_p), rounded up to fp32
        float zm = -INFINITY;
        if (minp_on)
            zm = __double2float_ru(static_cast<double>(m) +
                                   static_cast<double>(T) * log(static_cast<double>(P.min_p)));
        Surv R = K;
        bool wsum_is_R = false;
        if (topp_on) {
            // masses over K, plus a mass histogram over the keys whose weight is
            // at least (1 - top_p) / (2V): the ids below carry less than half of
            // the (1 - top_p) share of K's mass, so the cutoff lies inside
            const float zfloor = fmaxf(zm, K.zt);
            const double zb = static_cast<double>(m) +
                              static_cast<double>(T) *
                                  log((1.0 - static_cast<double>(P.top_p)) / (2.0 * static_cast<double>(a.V)));
            float zlo = fmaxf(__double2float_rd(zb), zfloor);
            Window W = Ctx::make_window(fkey(zlo), Km);
            if (K.ge_form())
                pass_mass<Ctx, false, true>(X, K, W);
            else
                pass_mass<Ctx, true, true>(X, K, W);
            X.publish_wsum_total(0);
            X.xsync();
            mass_k = X.xscan(0, ~0ull).total;
            X.xnext();
            uint64_t tgt = static_cast<uint64_t>(ceil(static_cast<double>(P.top_p) * static_cast<double>(mass_k)));
            if (tgt == 0) tgt = 1;
            float zp = -INFINITY;
            bool found = select_mass(X, W, K, tgt, zp);
            if (!found && zlo > zfloor) {
                // rounding left the first window just short: retry down to the hard bound
                zlo = zfloor;
                W = Ctx::make_window(fkey(zlo), Km);
                pass_mass_hist(X, W, K, false);
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
        if (!wsum_is_R) pass_mass_any(X, R);
        X.publish_wsum_total(0);
        rbits = splitmix64(P.seed ^ (static_cast<uint64_t>(row) << 32) ^ P.step) >> 11;
        X.xsync();
        mass_r = X.xscan(0, ~0ull).total;
        target = scale_by_u(rbits, mass_r);
        const typename Ctx::Scan sc = X.xscan(0, target);
        X.xnext();
        if (sc.first < 0) {
            err |= kErrInternal;
            token = am;
        } else if (sc.first == X.rank) {
            const uint64_t t = target - sc.before_me;
            int tok;
            if (R.ge_form())
                tok = X.walk(
                    t, [&](const float(&z)[VEC], int g0) { return X.template vec_mass<false>(z, g0, R); },
                    [&](const float(&z)[VEC], int g0, uint64_t tt) {
                        return X.template vec_mass_walk<false>(z, g0, R, tt);
                    });
            else
                tok = X.walk(
                    t, [&](const float(&z)[VEC], int g0) { return X.template vec_mass<true>(z, g0, R); },
                    [&](const float(&z)[VEC], int g0, uint64_t tt) {
                        return X.template vec_mass_walk<true>(z, g0, R, tt);
                    });
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
    X.cl.sync();
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
