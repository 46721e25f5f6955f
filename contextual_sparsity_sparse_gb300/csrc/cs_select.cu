// Selection: top-k, threshold and positive-pre-activation compaction.
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (the top-k scores are the
// predicted active set); "Activation sparsity", section "Implementation
// sketch" (predict_active: scores >= threshold); "Contextual Sparsity and
// Activation Predictors", first section (a neuron is active when its gate
// pre-activation passes the ReLU).
//
// Ranking: larger score first, equal scores by lower id, -0 == +0, NaN below
// -inf (as order-preserving 32-bit keys).  Top-k needs the k-th key K and the
// number of ties at K to take:
//   1. bounds of the finite scores: their min / max (one CTA), or on a
//      cluster the range of a fixed sample of the row, widened (scores past
//      it share the end buckets);
//   2. a 4096-bucket histogram of a monotone linear map of the score (NaN,
//      -inf and +inf get their own end buckets), so buckets hold a handful of
//      scores for any smooth distribution;
//   3. a suffix scan finds the bucket B holding the k-th score;
//   4. B's members are ranked exactly against each other (key, then id); the
//      member of rank k-1 gives K and the number of ties to take.  A bucket
//      with more than 64 members (a mass of near-equal scores) is resolved
//      instead by a radix select on the exact keys of its members.
// Compaction is in ascending id order: every thread owns a contiguous run of
// ids, so one exclusive scan of the packed (greater, tie) counts gives each
// thread its output position and the ties before it (the lowest ids win).
//
// Rows of f >= 2048 scores run on a cluster of 8 CTAs (the per-element passes
// split 8 ways, the CTAs exchanging through distributed shared memory);
// shorter rows on one CTA, and rows of at most 64 scores on one warp (exact
// ranks by pairwise comparison).  None takes a global atomic or a grid-wide
// barrier.
#include <cooperative_groups.h>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kBuckets = 4096;

// Order-preserving key: larger score -> larger key.  -0 is folded onto +0;
// NaN maps to 0, below the key of -inf (0x007fffff).
__device__ __forceinline__ uint32_t score_key(float s) {
    if (s != s) return 0u;
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// ---------------------------------------------------------------------------
// Row kernel: one CTA of 1024 threads per token row; thread t owns the
// contiguous ids [t*E, t*E + E), E = ceil(f / 1024) <= ET, held in registers.
// Every per-element pass is a short register loop and every block-wide step
// a warp-shuffle reduction or one prefix scan.
// ---------------------------------------------------------------------------
constexpr int kRowThreads = 1024;
constexpr int kCandSmall = 64;

__device__ __forceinline__ float warp_min(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}
__device__ __forceinline__ int warp_isum(int v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Exclusive prefix sum of one unsigned value per thread (wraps modulo 2^32,
// so two 16-bit counts packed in one word scan independently).
__device__ __forceinline__ uint32_t block_excl_scan_u32(uint32_t v, uint32_t *wsum, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    constexpr int nw = kRowThreads / 32;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = wsum[lane];
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += n;
        }
        wsum[lane] = w;
    }
    __syncthreads();
    const uint32_t base = warp > 0 ? wsum[warp - 1] : 0u;
    *total = wsum[nw - 1];
    __syncthreads();
    return base + inc - v;
}

// Bucket of a score for the row kernel: NaN 0, -inf 1, +inf kBuckets-1, a
// finite s 2 + round(clamp(s * scale + off, 0, kBuckets - 4)).  Monotone in s:
// a correctly rounded fma of a linear map with scale >= 0, a clamp and a
// round-to-nearest are each non-decreasing.  The rounding adds 1.5 * 2^23,
// which leaves round(t) in the low mantissa bits (0 <= t < 2^22).
__device__ __forceinline__ int bucket_fast(float s, float scale, float off) {
    float t = fmaf(s, scale, off);
    t = fminf(fmaxf(t, 0.f), (float)(kBuckets - 4));
    int b = __float_as_int(t + 12582912.f) - 0x4B400000 + 2;
    b = fabsf(s) == INFINITY ? (s > 0.f ? kBuckets - 1 : 1) : b;
    return s != s ? 0 : b;
}

// The ranking of score keys as float comparisons against the pivot's value pv
// (key(s) > key(p) iff s > p for non-NaN s, p; -0 == +0 either way).  A NaN
// pivot (key 0) makes every NaN a tie and every other score greater.
__device__ __forceinline__ void rank_flags(float s, float pv, bool pnan, bool &gt, bool &eq) {
    const bool snan = s != s;
    gt = pnan ? !snan : s > pv;
    eq = pnan ? snan : s == pv;
}

template <int ET, int KIND>
__global__ void __launch_bounds__(kRowThreads, 1)
select_row_kernel(const float *scores, int f, int k, float tau,
                  int32_t *__restrict__ idx, int ld_idx, int32_t *__restrict__ count,
                  uint32_t *__restrict__ mask, int hot) {
    __shared__ __align__(16) uint32_t hist[kBuckets];
    __shared__ uint32_t ckey[kCandSmall], cid[kCandSmall];
    __shared__ float wlo[32], whi[32];
    __shared__ uint32_t usum[32];
    __shared__ uint32_t s_bucket, s_rem, s_ncand, s_fill, s_pivot, s_need;
    __shared__ uint32_t bits[kSelectMaxF / 32];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int b = blockIdx.x;
    const float *s = scores + (size_t)b * f;
    // a hot prefix of `hot` neurons (a multiple of 32) comes first: ids
    // 0 .. hot-1, then hot + the tail's selection; the scores are the tail's
    int32_t *const row = idx + (size_t)b * ld_idx;
    int32_t *out = row + hot;
    const int words = (f + 31) >> 5;                 // the tail's mask words
    const int mwords = (hot + f + 31) >> 5;          // a mask row
    const int E = (f + kRowThreads - 1) / kRowThreads;
    const int j0 = tid * E;
    const int ne = max(0, min(E, f - j0));

    if (tid == 0) s_fill = 0u;
    if (mask)
        for (int w = tid; w < words; w += kRowThreads) bits[w] = 0u;

    pdl_launch_dependents();  // single CTA: let the consumer kernel get resident
    pdl_wait();               // scores come from the previous kernel

    float v[ET];
    const bool vec = (E & 3) == 0 && (reinterpret_cast<uintptr_t>(s) & 15) == 0;
#pragma unroll
    for (int q = 0; q < ET; q += 4) {
        if (vec && q + 4 <= ne) {
            const float4 t = ld_dep(reinterpret_cast<const float4 *>(s + j0 + q));
            v[q] = t.x; v[q + 1] = t.y; v[q + 2] = t.z; v[q + 3] = t.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[q + e] = q + e < ne ? ld_dep(s + j0 + q + e) : 0.f;
        }
    }

    const int kk = k < 0 ? 0 : (k > f ? f : k);
    float pv = 0.f;      // pivot value (top-k)
    bool pnan = false;   // pivot is NaN
    int need = 0;        // ties at the pivot to take, lowest ids first
    if (KIND == SEL_TOPK && kk > 0 && kk < f) {
        float lo = INFINITY, hi = -INFINITY;
#pragma unroll
        for (int e = 0; e < ET; ++e)
            if (e < ne && fabsf(v[e]) < INFINITY) { lo = fminf(lo, v[e]); hi = fmaxf(hi, v[e]); }
        lo = warp_min(lo);
        hi = warp_max(hi);
        if (lane == 0) { wlo[warp] = lo; whi[warp] = hi; }
        reinterpret_cast<uint4 *>(hist)[tid] = make_uint4(0u, 0u, 0u, 0u);
        __syncthreads();
        const float smin = warp_min(wlo[lane]), smax = warp_max(whi[lane]);
        const float scale = smax > smin ? (float)(kBuckets - 4) / (smax - smin) : 0.f;
        const float off = -smin * scale;
#pragma unroll
        for (int e = 0; e < ET; ++e)
            if (e < ne) atomicAdd(&hist[bucket_fast(v[e], scale, off)], 1u);
        __syncthreads();
        // thread t owns bins [4t, 4t + 4); members above them = total - prefix - own
        static_assert(kBuckets == 4 * kRowThreads, "four bins per thread");
        const uint4 hb = reinterpret_cast<const uint4 *>(hist)[tid];
        const uint32_t cb[4] = {hb.x, hb.y, hb.z, hb.w};
        const uint32_t own = hb.x + hb.y + hb.z + hb.w;
        uint32_t total;
        const uint32_t pre = block_excl_scan_u32(own, usum, &total);
        uint32_t run = total - pre - own;
#pragma unroll
        for (int q = 3; q >= 0; --q) {
            if (run < (uint32_t)kk && run + cb[q] >= (uint32_t)kk) {
                s_bucket = (uint32_t)(4 * tid + q);
                s_rem = (uint32_t)kk - run;
                s_ncand = cb[q];
            }
            run += cb[q];
        }
        __syncthreads();
        const int B_ = (int)s_bucket;
        const uint32_t rem = s_rem, ncand = s_ncand;
        uint32_t pkey;
        if (ncand <= (uint32_t)kCandSmall) {
            // the bucket's members, ranked exactly (key descending, id ascending)
#pragma unroll
            for (int e = 0; e < ET; ++e) {
                if (e < ne && bucket_fast(v[e], scale, off) == B_) {
                    const uint32_t p = atomicAdd(&s_fill, 1u);
                    ckey[p] = score_key(v[e]);
                    cid[p] = (uint32_t)(j0 + e);
                }
            }
            __syncthreads();
            // warp w ranks members w, w + 32, ...: lanes split the comparisons
            for (int c = warp; c < (int)ncand; c += kRowThreads / 32) {
                const uint32_t kc = ckey[c], ic = cid[c];
                int rk = 0, gt = 0;
                for (int o = lane; o < (int)ncand; o += 32) {
                    const uint32_t ko = ckey[o];
                    rk += (ko > kc) || (ko == kc && cid[o] < ic);
                    gt += ko > kc;
                }
                rk = warp_isum(rk);
                gt = warp_isum(gt);
                if (lane == 0 && rk == (int)rem - 1) {
                    s_pivot = kc;
                    s_need = rem - (uint32_t)gt;
                }
            }
            __syncthreads();
            pkey = s_pivot;
            need = (int)s_need;
        } else {
            // a crowded bucket (near-equal scores): radix select over its
            // members' exact keys, eight bits at a time
            uint32_t prefix = 0u, pmask = 0u, r_ = rem;
            for (int pass = 0; pass < 4; ++pass) {
                const int shift = 24 - 8 * pass;
                if (tid < 256) hist[tid] = 0u;
                __syncthreads();
#pragma unroll
                for (int e = 0; e < ET; ++e) {
                    if (e < ne && bucket_fast(v[e], scale, off) == B_) {
                        const uint32_t key = score_key(v[e]);
                        if ((key & pmask) == prefix) atomicAdd(&hist[(key >> shift) & 255u], 1u);
                    }
                }
                __syncthreads();
                if (warp == 0) {
                    // lane l holds digits 255 - 8l - i, i = 0..7 (descending)
                    uint32_t c8[8], sum = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) { c8[i] = hist[255 - 8 * lane - i]; sum += c8[i]; }
                    uint32_t inc = sum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t nn = __shfl_up_sync(kFull, inc, o);
                        if (lane >= o) inc += nn;
                    }
                    uint32_t run8 = inc - sum;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (run8 < r_ && run8 + c8[i] >= r_) {
                            s_pivot = (uint32_t)(255 - 8 * lane - i);
                            s_need = r_ - run8;
                        }
                        run8 += c8[i];
                    }
                }
                __syncthreads();
                prefix |= s_pivot << shift;
                pmask |= 255u << shift;
                r_ = s_need;
                __syncthreads();
            }
            pkey = prefix;
            need = (int)r_;
        }
        // back from the key to the value (keys of -0 and NaN never arise here
        // except key 0, a NaN pivot)
        pnan = pkey == 0u;
        pv = __uint_as_float((pkey & 0x80000000u) ? (pkey & 0x7fffffffu) : ~pkey);
    }

    // compaction: packed (greater, tie) counts of this thread's chunk -> one scan
    auto flags = [&](float x, bool &gt, bool &eq) {
        if (KIND == SEL_TOPK) {
            if (kk == f) { gt = true; eq = false; }
            else if (kk == 0) { gt = false; eq = false; }
            else rank_flags(x, pv, pnan, gt, eq);
        } else if (KIND == SEL_THRESHOLD) {
            gt = x >= tau;
            eq = false;
        } else if (KIND == SEL_SILU_MAG) {
            gt = fabsf(gate_act(CS_ACT_SILU, x)) > tau;
            eq = false;
        } else {   // SEL_POSITIVE: relu(x) > tau, tau >= 0
            gt = x > tau;
            eq = false;
        }
    };
    uint32_t cg = 0, ce = 0;
#pragma unroll
    for (int e = 0; e < ET; ++e) {
        if (e < ne) {
            bool gt, eq;
            flags(v[e], gt, eq);
            cg += gt;
            ce += eq;
        }
    }
    // f <= kSelectMaxF < 2^16: both block totals fit their 16-bit halves
    static_assert(kSelectMaxF < 65536, "packed counts");
    uint32_t tot;
    const uint32_t ex = block_excl_scan_u32((cg << 16) | ce, usum, &tot);
    int eq_run = (int)(ex & 0xffffu);
    int pos = (int)(ex >> 16) + min(eq_run, need);
#pragma unroll
    for (int e = 0; e < ET; ++e) {
        if (e < ne) {
            bool gt, eq;
            flags(v[e], gt, eq);
            const bool take = gt || (eq && eq_run < need);
            eq_run += eq;
            if (take) {
                const int j = j0 + e;
                out[pos++] = hot + j;
                if (mask) atomicOr(&bits[j >> 5], 1u << (j & 31));
            }
        }
    }
    if (tid == kRowThreads - 1) count[b] = hot + (int)(tot >> 16) + min((int)(tot & 0xffffu), need);
    for (int i = tid; i < hot; i += kRowThreads) row[i] = i;
    if (mask) {
        uint32_t *mrow = mask + (size_t)b * mwords;
        for (int w = tid; w < (hot >> 5); w += kRowThreads) mrow[w] = 0xffffffffu;
        __syncthreads();
        for (int w = tid; w < words; w += kRowThreads) mrow[(hot >> 5) + w] = bits[w];
    }
}

// ---------------------------------------------------------------------------
// Cluster row kernel: one cluster of kCl CTAs x 512 threads per token row.
// CTA r owns the 32-aligned id slice [r*SL, r*SL + SL); thread t of it the
// contiguous ids [t*E, t*E + E) of that slice, in registers.  The four steps
// of the row kernel run with the per-element passes split kCl ways.  The
// bucket map's bounds come from a fixed sample of the row that every CTA
// reads alike, so they need no exchange.  Small data is pushed into every
// CTA's shared memory before a cluster barrier, so that after it each CTA
// finds it locally: per-slice histogram totals, the pivot bucket's members,
// and the (greater, tie) totals behind the output offsets.  The one pull is
// the pivot slice's 512 bins from every CTA (all loads in flight together).
// Two cluster barriers when the sample has spread and the pivot bucket is
// small (every CTA then derives all CTAs' totals from the exchanged members
// and the pushed above-bucket counts); one more for a sample without spread
// (the exact min / max exchanged) and one more for a crowded pivot bucket.
// No shared memory is touched remotely after the last one, so CTAs may leave
// at once.  Half an SM's threads per CTA: the per-element loops are short
// and the block-wide steps still cheap (measured against 256 and 1024).
// ---------------------------------------------------------------------------
constexpr int kCl = 8;
constexpr int kClBins = kBuckets / kCl;     // bins per CTA slice
constexpr int kClMaxSlice = kSelectMaxF / kCl;
constexpr int kClT = 512;
constexpr int kClW = kClT / 32;
static_assert(kClW % kCl == 0, "whole warps per histogram slice");
static_assert((((kSelectMaxF / kCl) + 31) / 32 * 32 + kClT - 1) / kClT <= 12, "ET covers the largest row");

struct ClSmem {
    uint32_t hist[kBuckets];                  // local histogram
    uint32_t ptot[kCl][kCl];                // [source CTA][slice] partial slice totals
    float plo[kCl], phi[kCl];               // min / max from each CTA
    // [source CTA] pivot-bucket members; rows padded by one word so that lanes
    // walking different CTAs' rows at one position hit different banks
    uint32_t ckey[kCl][kCandSmall + 1];
    uint32_t cid[kCl][kCandSmall + 1];
    uint32_t ccnt[kCl];
    uint32_t pgt[kCl], peq[kCl];            // (greater, tie) totals from each CTA
    uint32_t pabove[kCl];                   // scores above the pivot bucket in each CTA
    uint32_t wab[kClW];
    uint32_t wsl[kClW];                     // per-warp histogram sums
    uint32_t lkey[kCandSmall], lid[kCandSmall];
    uint32_t rhist[256];                      // radix digits (crowded bucket)
    uint32_t akey[kCandSmall], aid[kCandSmall];
    uint32_t bits[kClMaxSlice / 32];
    uint32_t usum[32];
    float wlo[kClW], whi[kClW];
    uint32_t nfill;
    uint32_t bucket, rem, ncand, pivot, need;
};

// Exclusive scan over one CTA of the cluster kernel (unsigned, wraps modulo 2^32).
__device__ __forceinline__ uint32_t cta_excl_scan(uint32_t v, uint32_t *wsum, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    const uint32_t wv = lane < kClW ? wsum[lane] : 0u;
    uint32_t w = wv;
#pragma unroll
    for (int o = 1; o < kClW; o <<= 1) {
        const uint32_t n = __shfl_up_sync(kFull, w, o);
        if (lane >= o) w += n;
    }
    const uint32_t wex = __shfl_sync(kFull, w - wv, warp);
    *total = __shfl_sync(kFull, w, kClW - 1);
    __syncthreads();
    return wex + inc - v;
}

template <int ET, int KIND>
__global__ void __launch_bounds__(kClT, 1)
select_cl_kernel(const float *scores, int f, int k, float tau,
                 int32_t *__restrict__ idx, int ld_idx, int32_t *__restrict__ count,
                 uint32_t *__restrict__ mask, int hot) {
    namespace cg = cooperative_groups;
    cg::cluster_group cl = cg::this_cluster();
    __shared__ __align__(16) ClSmem S;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int rank = (int)cl.block_rank();
    const int b = blockIdx.x / kCl;
    const float *s = scores + (size_t)b * f;
    // hot prefix as in the row kernel: ids 0 .. hot-1 first (hot a multiple of 32)
    int32_t *const row = idx + (size_t)b * ld_idx;
    int32_t *out = row + hot;
    const int mwords = (hot + f + 31) >> 5;
    const int SL = (((f + kCl - 1) / kCl) + 31) & ~31;
    const int beg = min(rank * SL, f), n_my = min(SL, f - beg);
    const int E = (SL + kClT - 1) / kClT;
    const int j0 = tid * E;                      // within the slice
    const int ne = max(0, min(E, n_my - j0));

    // Zero what peers add into before the first barrier; nothing here reads
    // the scores, so it runs ahead of the wait.
#pragma unroll
    for (int i = tid; i < kBuckets / 4; i += kClT) reinterpret_cast<uint4 *>(S.hist)[i] = make_uint4(0u, 0u, 0u, 0u);
    if (mask)
        for (int w = tid; w < SL / 32; w += kClT) S.bits[w] = 0u;
    if (tid == 0) S.nfill = 0u;

    pdl_launch_dependents();
    pdl_wait();  // scores come from the previous kernel

    float v[ET];
    const bool vec = (E & 3) == 0 && ((reinterpret_cast<uintptr_t>(s) + 4u * (uint32_t)beg) & 15) == 0;
#pragma unroll
    for (int q = 0; q < ET; q += 4) {
        if (vec && q + 4 <= ne) {
            const float4 t = ld_dep(reinterpret_cast<const float4 *>(s + beg + j0 + q));
            v[q] = t.x; v[q + 1] = t.y; v[q + 2] = t.z; v[q + 3] = t.w;
        } else {
#pragma unroll
            for (int e = 0; e < 4; ++e) v[q + e] = q + e < ne ? ld_dep(s + beg + j0 + q + e) : 0.f;
        }
    }

    // one score of a fixed sample of the whole row per thread: the same ids
    // in every CTA (f >= 2048 > kClT, so the ids are distinct and in range)
    const float smp = KIND == SEL_TOPK ? ld_dep(s + (int)(((long long)tid * f) / kClT)) : 0.f;

    const int kk = k < 0 ? 0 : (k > f ? f : k);
    float pv = 0.f;
    bool pnan = false;
    int need = 0;
    bool fast = false;   // the per-CTA totals come from the exchanged candidates (no 4th barrier)
    if (KIND == SEL_TOPK && kk > 0 && kk < f) {
        // 1. bounds of the bucket map: the finite range of the sample widened
        //    by half its width on either side, identical in every CTA (same
        //    ids, exact min / max), so no exchange.  Scores beyond the bounds
        //    fall into the end buckets; the map stays monotone, so the result
        //    is exact whatever the bounds, which only set how many scores
        //    share the pivot bucket.  A sample without spread (or a range
        //    near overflow) takes the exact min / max of the row instead,
        //    pushed to every CTA.
        const bool sf = fabsf(smp) < INFINITY;
        float lo = warp_min(sf ? smp : INFINITY), hi = warp_max(sf ? smp : -INFINITY);
        if (lane == 0) { S.wlo[warp] = lo; S.whi[warp] = hi; }
        __syncthreads();
        float smin = warp_min(lane < kClW ? S.wlo[lane] : INFINITY);
        float smax = warp_max(lane < kClW ? S.whi[lane] : -INFINITY);
        const float half = 0.5f * (smax - smin);
        const float wlo_ = smin - half, whi_ = smax + half;
        if (smax > smin && fabsf(wlo_) < INFINITY && fabsf(whi_) < INFINITY &&
            (float)(kBuckets - 4) / (whi_ - wlo_) < INFINITY) {
            smin = wlo_;
            smax = whi_;
        } else {
            lo = INFINITY;
            hi = -INFINITY;
#pragma unroll
            for (int e = 0; e < ET; ++e)
                if (e < ne && fabsf(v[e]) < INFINITY) { lo = fminf(lo, v[e]); hi = fmaxf(hi, v[e]); }
            lo = warp_min(lo);
            hi = warp_max(hi);
            __syncthreads();   // every warp has read the sample's partials
            if (lane == 0) { S.wlo[warp] = lo; S.whi[warp] = hi; }
            __syncthreads();
            if (warp == 0) {
                lo = warp_min(lane < kClW ? S.wlo[lane] : INFINITY);
                hi = warp_max(lane < kClW ? S.whi[lane] : -INFINITY);
                if (lane < kCl) {
                    *cl.map_shared_rank(&S.plo[rank], lane) = lo;
                    *cl.map_shared_rank(&S.phi[rank], lane) = hi;
                }
            }
            cl.sync();                                                    // (1)
            smin = warp_min(lane < kCl ? S.plo[lane] : INFINITY);
            smax = warp_max(lane < kCl ? S.phi[lane] : -INFINITY);
        }
        const float scale = smax > smin ? (float)(kBuckets - 4) / (smax - smin) : 0.f;
        const float off = -smin * scale;
        // 2. local histogram; this CTA's total of each slice w (bins
        //    [w*512, w*512 + 512), summed by kClW / kCl warps) pushed to
        //    every CTA
        int bk[ET];  // each score's bucket, kept for the candidate pass
#pragma unroll
        for (int e = 0; e < ET; ++e) {
            bk[e] = e < ne ? bucket_fast(v[e], scale, off) : -1;
            if (e < ne) atomicAdd(&S.hist[bk[e]], 1u);
        }
        __syncthreads();
        {
            constexpr int WPS = kClW / kCl;                 // warps per slice
            constexpr int BPL = kClBins / (32 * WPS);       // bins per lane
            const int bin0 = warp * (kClBins / WPS) + lane * BPL;
            uint32_t sum = 0;
#pragma unroll
            for (int q = 0; q < BPL; q += 4) {
                const uint4 h4 = *reinterpret_cast<const uint4 *>(&S.hist[bin0 + q]);
                sum += h4.x + h4.y + h4.z + h4.w;
            }
            sum = (uint32_t)warp_isum((int)sum);
            if (WPS == 1) {
                if (lane < kCl) *cl.map_shared_rank(&S.ptot[rank][warp], lane) = sum;
            } else {
                if (lane == 0) S.wsl[warp] = sum;
                __syncthreads();
                if (warp < kCl && lane < kCl) {
                    uint32_t t = 0;
#pragma unroll
                    for (int q = 0; q < WPS; ++q) t += S.wsl[warp * WPS + q];
                    *cl.map_shared_rank(&S.ptot[rank][warp], lane) = t;
                }
            }
        }
        cl.sync();                                                        // (2)
        // 3. the slice holding the kk-th largest (slice w holds higher scores
        //    than slice w - 1), then its bins summed over the CTAs (all remote
        //    loads in flight together), then the bucket
        uint32_t tw = 0;
        if (lane < kCl) {
#pragma unroll
            for (int r = 0; r < kCl; ++r) tw += S.ptot[r][lane];
        }
        uint32_t above = 0, above_owner = 0;
        int owner = 0;
#pragma unroll
        for (int r = kCl - 1; r >= 0; --r) {
            const uint32_t t = __shfl_sync(kFull, tw, r);
            if (above < (uint32_t)kk && above + t >= (uint32_t)kk) { owner = r; above_owner = above; }
            above += t;
        }
        {
            // BPT of the slice's bins per thread (threads past the slice idle)
            constexpr int BPT = kClBins >= kClT ? kClBins / kClT : 1;
            const int bin = owner * kClBins + BPT * tid;
            const bool has = BPT * tid < kClBins;
            uint32_t got[kCl][BPT];
#pragma unroll
            for (int r = 0; r < kCl; ++r)
#pragma unroll
                for (int q = 0; q < BPT; ++q) got[r][q] = has ? *cl.map_shared_rank(&S.hist[bin + q], r) : 0u;
            uint32_t cb[BPT], own = 0;
#pragma unroll
            for (int q = 0; q < BPT; ++q) {
                cb[q] = 0u;
#pragma unroll
                for (int r = 0; r < kCl; ++r) cb[q] += got[r][q];
                own += cb[q];
            }
            uint32_t tot_o;
            const uint32_t pre = cta_excl_scan(own, S.usum, &tot_o);
            uint32_t run = above_owner + (tot_o - pre - own);
#pragma unroll
            for (int q = BPT - 1; q >= 0; --q) {
                if (run < (uint32_t)kk && run + cb[q] >= (uint32_t)kk) {
                    S.bucket = (uint32_t)(bin + q);
                    S.rem = (uint32_t)kk - run;
                    S.ncand = cb[q];
                }
                run += cb[q];
            }
        }
        __syncthreads();
        const int B_ = (int)S.bucket;
        const uint32_t rem = S.rem, ncand = S.ncand;
        uint32_t pkey;
        if (ncand <= (uint32_t)kCandSmall) {
            // 4. the bucket's members, pushed to every CTA, ranked exactly
#pragma unroll
            for (int e = 0; e < ET; ++e) {
                if (bk[e] == B_) {
                    const uint32_t p = atomicAdd(&S.nfill, 1u);
                    S.lkey[p] = score_key(v[e]);
                    S.lid[p] = (uint32_t)(beg + j0 + e);
                }
            }
            // and this CTA's count of scores above the pivot bucket
            {
                uint32_t ab = 0;
#pragma unroll
                for (int e = 0; e < ET; ++e) ab += bk[e] > B_;
                ab = (uint32_t)warp_isum((int)ab);
                if (lane == 0) S.wab[warp] = ab;
            }
            __syncthreads();
            const uint32_t nmine = S.nfill;
            for (uint32_t i = tid; i < nmine * kCl; i += kClT) {
                const uint32_t p = i / kCl, r = i % kCl;
                *cl.map_shared_rank(&S.ckey[rank][p], r) = S.lkey[p];
                *cl.map_shared_rank(&S.cid[rank][p], r) = S.lid[p];
            }
            if (tid < kCl) {
                uint32_t ab = 0;
#pragma unroll
                for (int w = 0; w < kClW; ++w) ab += S.wab[w];
                *cl.map_shared_rank(&S.ccnt[rank], tid) = nmine;
                *cl.map_shared_rank(&S.pabove[rank], tid) = ab;
            }
            cl.sync();                                                    // (3)
            if (warp == 0) {
                const uint32_t nr = lane < kCl ? S.ccnt[lane] : 0u;
                uint32_t inc = nr;
#pragma unroll
                for (int o = 1; o < kCl; o <<= 1) {
                    const uint32_t n = __shfl_up_sync(kFull, inc, o);
                    if (lane >= o) inc += n;
                }
                // lane r copies CTA r's members to positions [inc - nr, inc)
                if (lane < kCl)
                    for (uint32_t p = 0; p < nr; ++p) {
                        S.akey[inc - nr + p] = S.ckey[lane][p];
                        S.aid[inc - nr + p] = S.cid[lane][p];
                    }
            }
            __syncthreads();
            for (int c = warp; c < (int)ncand; c += kClW) {
                const uint32_t kc = S.akey[c], ic = S.aid[c];
                int rk = 0, gt = 0;
                for (int o = lane; o < (int)ncand; o += 32) {
                    const uint32_t ko = S.akey[o];
                    rk += (ko > kc) || (ko == kc && S.aid[o] < ic);
                    gt += ko > kc;
                }
                rk = warp_isum(rk);
                gt = warp_isum(gt);
                if (lane == 0 && rk == (int)rem - 1) {
                    S.pivot = kc;
                    S.need = rem - (uint32_t)gt;
                }
            }
            __syncthreads();
            pkey = S.pivot;
            need = (int)S.need;
            // every CTA's (greater, tie) totals: above the bucket, plus its
            // members above / equal to the pivot (a higher bucket means a
            // strictly larger score; equal scores share a bucket)
            if (warp == 0 && lane < kCl) {
                uint32_t gt = S.pabove[lane], eq = 0;
                for (uint32_t p = 0; p < S.ccnt[lane]; ++p) {
                    const uint32_t kv = S.ckey[lane][p];
                    gt += kv > pkey;
                    eq += kv == pkey;
                }
                S.pgt[lane] = gt;
                S.peq[lane] = eq;
            }
            fast = true;   // (the next barrier publishes pgt / peq within the CTA)
        } else {
            // a crowded bucket: each CTA resolves it alone with a radix select
            // over the whole row's members of the bucket (read from global)
            uint32_t prefix = 0u, pmask = 0u, r_ = rem;
            for (int pass = 0; pass < 4; ++pass) {
                const int shift = 24 - 8 * pass;
                if (tid < 256) S.rhist[tid] = 0u;
                __syncthreads();
                for (int j = tid; j < f; j += kClT) {
                    const float x = ld_dep(s + j);
                    if (bucket_fast(x, scale, off) == B_) {
                        const uint32_t key = score_key(x);
                        if ((key & pmask) == prefix) atomicAdd(&S.rhist[(key >> shift) & 255u], 1u);
                    }
                }
                __syncthreads();
                if (warp == 0) {
                    uint32_t c8[8], sum = 0;
#pragma unroll
                    for (int i = 0; i < 8; ++i) { c8[i] = S.rhist[255 - 8 * lane - i]; sum += c8[i]; }
                    uint32_t inc = sum;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t nn = __shfl_up_sync(kFull, inc, o);
                        if (lane >= o) inc += nn;
                    }
                    uint32_t run8 = inc - sum;
#pragma unroll
                    for (int i = 0; i < 8; ++i) {
                        if (run8 < r_ && run8 + c8[i] >= r_) {
                            S.pivot = (uint32_t)(255 - 8 * lane - i);
                            S.need = r_ - run8;
                        }
                        run8 += c8[i];
                    }
                }
                __syncthreads();
                prefix |= S.pivot << shift;
                pmask |= 255u << shift;
                r_ = S.need;
                __syncthreads();
            }
            pkey = prefix;
            need = (int)r_;
        }
        pnan = pkey == 0u;
        pv = __uint_as_float((pkey & 0x80000000u) ? (pkey & 0x7fffffffu) : ~pkey);
    }

    // 5. compaction: packed (greater, tie) counts -> CTA scan -> totals pushed
    //    to every CTA -> this CTA's output offsets
    auto flags = [&](float x, bool &gt, bool &eq) {
        if (KIND == SEL_TOPK) {
            if (kk == f) { gt = true; eq = false; }
            else if (kk == 0) { gt = false; eq = false; }
            else rank_flags(x, pv, pnan, gt, eq);
        } else if (KIND == SEL_THRESHOLD) {
            gt = x >= tau;
            eq = false;
        } else if (KIND == SEL_SILU_MAG) {
            gt = fabsf(gate_act(CS_ACT_SILU, x)) > tau;
            eq = false;
        } else {   // SEL_POSITIVE: relu(x) > tau, tau >= 0
            gt = x > tau;
            eq = false;
        }
    };
    // the (greater, tie) flags of this thread's scores as bit masks (ET <= 32)
    static_assert(ET <= 32, "flag masks");
    uint32_t gmask = 0, emask = 0;
#pragma unroll
    for (int e = 0; e < ET; ++e) {
        if (e < ne) {
            bool gt, eq;
            flags(v[e], gt, eq);
            gmask |= (uint32_t)gt << e;
            emask |= (uint32_t)eq << e;
        }
    }
    const uint32_t cgt = __popc(gmask), ceq = __popc(emask);
    uint32_t tot;
    const uint32_t ex = cta_excl_scan((cgt << 16) | ceq, S.usum, &tot);  // also orders pgt / peq
    if (!fast) {
        if (tid < kCl) {
            *cl.map_shared_rank(&S.pgt[rank], tid) = tot >> 16;
            *cl.map_shared_rank(&S.peq[rank], tid) = tot & 0xffffu;
        }
        cl.sync();                                                        // (4)
    }
    // offsets of this CTA: lanes r < kCl hold CTA r's totals (every warp alike)
    const uint32_t g_ = lane < kCl ? S.pgt[lane] : 0u, e_ = lane < kCl ? S.peq[lane] : 0u;
    uint32_t gi = g_, ei = e_;
#pragma unroll
    for (int o = 1; o < kCl; o <<= 1) {
        const uint32_t a1 = __shfl_up_sync(kFull, gi, o), a2 = __shfl_up_sync(kFull, ei, o);
        if (lane >= o) { gi += a1; ei += a2; }
    }
    const int gb = (int)__shfl_sync(kFull, gi - g_, rank), eb = (int)__shfl_sync(kFull, ei - e_, rank);
    int eq_run = eb + (int)(ex & 0xffffu);
    int pos = gb + (int)(ex >> 16) + min(eq_run, need);
    // ascending ids: greater scores always, ties while the quota lasts
    for (uint32_t m = gmask | emask; m; m &= m - 1) {
        const int e = __ffs(m) - 1;
        const bool eq = (emask >> e) & 1u;
        const bool take = ((gmask >> e) & 1u) || (eq && eq_run < need);
        eq_run += eq;
        if (take) {
            const int jl = j0 + e;
            out[pos++] = hot + beg + jl;
            if (mask) atomicOr(&S.bits[jl >> 5], 1u << (jl & 31));
        }
    }
    if (rank == 0 && warp == 0) {
        const uint32_t gt_all = __shfl_sync(kFull, gi, kCl - 1), eq_all = __shfl_sync(kFull, ei, kCl - 1);
        if (lane == 0) count[b] = hot + (int)gt_all + min((int)eq_all, need);
    }
    for (int i = rank * kClT + tid; i < hot; i += kCl * kClT) row[i] = i;
    if (mask) {
        uint32_t *mrow = mask + (size_t)b * mwords;
        for (int w = rank * kClT + tid; w < (hot >> 5); w += kCl * kClT) mrow[w] = 0xffffffffu;
        __syncthreads();
        const int nw = (n_my + 31) >> 5;
        for (int w = tid; w < nw; w += kClT) mrow[(hot >> 5) + (beg >> 5) + w] = S.bits[w];
    }
}

template <int ET, int KIND>
cudaError_t run_select_cl(const SelectArgs &a, cudaStream_t s) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCl * a.B);
    cfg.blockDim = dim3(kClT);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kCl;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    int n = 1;
    if (pdl_enabled()) {
        attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[1].val.programmaticStreamSerializationAllowed = 1;
        n = 2;
    }
    cfg.attrs = attr;
    cfg.numAttrs = n;
    return cudaLaunchKernelEx(&cfg, select_cl_kernel<ET, KIND>, a.scores, a.f, a.k, a.tau, a.idx, a.ld_idx,
                              a.count, a.mask, a.hot);
}

template <int ET>
cudaError_t run_select_cl_kind(const SelectArgs &a, cudaStream_t s) {
    if (a.kind == SEL_TOPK) return run_select_cl<ET, SEL_TOPK>(a, s);
    if (a.kind == SEL_THRESHOLD) return run_select_cl<ET, SEL_THRESHOLD>(a, s);
    if (a.kind == SEL_SILU_MAG) return run_select_cl<ET, SEL_SILU_MAG>(a, s);
    return run_select_cl<ET, SEL_POSITIVE>(a, s);
}

cudaError_t launch_select_cl(const SelectArgs &a, cudaStream_t s) {
    const int SL = (((a.f + kCl - 1) / kCl) + 31) & ~31;
    const int E = (SL + kClT - 1) / kClT;     // <= 12 for f <= kSelectMaxF
    if (E <= 4) return run_select_cl_kind<4>(a, s);
    if (E <= 8) return run_select_cl_kind<8>(a, s);
    return run_select_cl_kind<12>(a, s);
}

template <int ET, int KIND>
cudaError_t run_select_row(const SelectArgs &a, cudaStream_t s) {
    return launch(select_row_kernel<ET, KIND>, dim3(a.B), dim3(kRowThreads), 0, s, pdl_enabled(), a.scores,
                  a.f, a.k, a.tau, a.idx, a.ld_idx, a.count, a.mask, a.hot);
}

template <int ET>
cudaError_t run_select_kind(const SelectArgs &a, cudaStream_t s) {
    if (a.kind == SEL_TOPK) return run_select_row<ET, SEL_TOPK>(a, s);
    if (a.kind == SEL_THRESHOLD) return run_select_row<ET, SEL_THRESHOLD>(a, s);
    if (a.kind == SEL_SILU_MAG) return run_select_row<ET, SEL_SILU_MAG>(a, s);
    return run_select_row<ET, SEL_POSITIVE>(a, s);
}

cudaError_t launch_select_row(const SelectArgs &a, cudaStream_t s) {
    const int E = (a.f + kRowThreads - 1) / kRowThreads;
    // rows of f < 2048 only (longer rows run on a cluster): E <= 2
    if (E <= 4) return run_select_kind<4>(a, s);
    return cudaErrorInvalidValue;
}

// ---------------------------------------------------------------------------
// Warp row kernel: rows of f <= 64 scores (one score per attention head, say)
// on one warp each; lane l holds ids l and l + 32.  Top-k ranks every score
// exactly: its rank is the number of scores ahead of it (a larger key, or an
// equal key at a lower id), found by broadcasting each key in turn; the
// scores of rank < k are taken.  Ballots compact the taken ids in ascending
// order.  No shared memory and no barrier.
// ---------------------------------------------------------------------------
constexpr int kWarpRowMaxF = 64;

template <int KIND>
__global__ void __launch_bounds__(32) select_warp_kernel(const float *scores, int f, int k, float tau,
                                                         int32_t *__restrict__ idx, int ld_idx,
                                                         int32_t *__restrict__ count, uint32_t *__restrict__ mask,
                                                         int hot) {
    const int lane = threadIdx.x, b = blockIdx.x;
    const float *s = scores + (size_t)b * f;
    int32_t *const row = idx + (size_t)b * ld_idx;
    int32_t *out = row + hot;
    pdl_launch_dependents();
    pdl_wait();  // scores come from the previous kernel
    const bool in0 = lane < f, in1 = lane + 32 < f;
    const float v0 = in0 ? ld_dep(s + lane) : 0.f, v1 = in1 ? ld_dep(s + lane + 32) : 0.f;
    bool t0, t1;
    if (KIND == SEL_TOPK) {
        const int kk = k < 0 ? 0 : (k > f ? f : k);
        const uint32_t k0 = score_key(v0), k1 = score_key(v1);
        int r0 = 0, r1 = 0;
        for (int j = 0; j < f; ++j) {
            const uint32_t kj = __shfl_sync(kFull, j < 32 ? k0 : k1, j & 31);
            r0 += (kj > k0) || (kj == k0 && j < lane);
            r1 += (kj > k1) || (kj == k1 && j < lane + 32);
        }
        t0 = in0 && r0 < kk;
        t1 = in1 && r1 < kk;
    } else if (KIND == SEL_THRESHOLD) {
        t0 = in0 && v0 >= tau;
        t1 = in1 && v1 >= tau;
    } else if (KIND == SEL_SILU_MAG) {
        t0 = in0 && fabsf(gate_act(CS_ACT_SILU, v0)) > tau;
        t1 = in1 && fabsf(gate_act(CS_ACT_SILU, v1)) > tau;
    } else {   // SEL_POSITIVE
        t0 = in0 && v0 > tau;
        t1 = in1 && v1 > tau;
    }
    const uint32_t m0 = __ballot_sync(kFull, t0), m1 = __ballot_sync(kFull, t1);
    const uint32_t below = (1u << lane) - 1u;
    const int n0 = __popc(m0);
    if (t0) out[__popc(m0 & below)] = hot + lane;
    if (t1) out[n0 + __popc(m1 & below)] = hot + lane + 32;
    if (lane == 0) count[b] = hot + n0 + __popc(m1);
    for (int i = lane; i < hot; i += 32) row[i] = i;
    if (mask) {
        uint32_t *mrow = mask + (size_t)b * ((hot + f + 31) >> 5);
        for (int w = lane; w < (hot >> 5); w += 32) mrow[w] = 0xffffffffu;
        if (lane == 0 && f > 0) mrow[hot >> 5] = m0;
        if (lane == 1 && f > 32) mrow[(hot >> 5) + 1] = m1;
    }
}

cudaError_t launch_select_warp(const SelectArgs &a, cudaStream_t s) {
    auto go = [&](auto kern) {
        return launch(kern, dim3(a.B), dim3(32), 0, s, pdl_enabled(), a.scores, a.f, a.k, a.tau, a.idx, a.ld_idx,
                      a.count, a.mask, a.hot);
    };
    if (a.kind == SEL_TOPK) return go(select_warp_kernel<SEL_TOPK>);
    if (a.kind == SEL_THRESHOLD) return go(select_warp_kernel<SEL_THRESHOLD>);
    if (a.kind == SEL_SILU_MAG) return go(select_warp_kernel<SEL_SILU_MAG>);
    return go(select_warp_kernel<SEL_POSITIVE>);
}

}  // namespace

cudaError_t launch_select(const SelectArgs &a, cudaStream_t s) {
    if (a.f >= 2048) return launch_select_cl(a, s);
    if (a.f <= kWarpRowMaxF) return launch_select_warp(a, s);
    return launch_select_row(a, s);
}

}  // namespace cs
