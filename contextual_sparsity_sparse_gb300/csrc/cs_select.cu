// Selection: top-k, threshold and positive-pre-activation compaction.
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (the top-k scores are the
// predicted active set); "Activation sparsity", section "Implementation
// sketch" (predict_active: scores >= threshold); "Contextual Sparsity and
// Activation Predictors", first section (a neuron is active when its gate
// pre-activation passes the ReLU).
//
// One CTA of 1024 threads per token row; the row's scores sit in shared
// memory.  Ranking: larger score first, equal scores by lower id, -0 == +0,
// NaN below -inf (as order-preserving 32-bit keys).  Top-k needs the k-th key
// K and the number of ties at K to take:
//   1. min / max of the finite scores (block reduction);
//   2. a 4096-bucket histogram of a monotone linear map of the score (NaN,
//      -inf and +inf get their own end buckets), so buckets hold a handful of
//      scores for any smooth distribution;
//   3. a suffix scan finds the bucket B holding the k-th score;
//   4. B's members are ranked exactly against each other (key, then id);
//      the member of rank k-1 gives K and the number of ties to take.  A
//      bucket with more than 2048 members (a mass of equal scores) is
//      resolved instead by a radix select on the exact keys of its members.
// Compaction is in ascending id order: each warp owns a contiguous range taken
// 32 ids at a time; warp ballots give in-warp ranks (and the mask words), one
// scan over the 32 warps gives (a) the K-ties before each warp, so the lowest
// ids win, and (b) each warp's output position.  No global atomics and no
// grid-wide synchronisation: a grid barrier costs microseconds here.
#include <cstdlib>
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kSelThreads = 1024;
constexpr int kBuckets = 4096;
constexpr int kCandMax = 2048;

// Order-preserving key: larger score -> larger key.  -0 is folded onto +0;
// NaN maps to 0, below the key of -inf (0x007fffff).
__device__ __forceinline__ uint32_t score_key(float s) {
    if (s != s) return 0u;
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__device__ __forceinline__ int bucket_of(float s, float smin, float scale) {
    if (s != s) return 0;
    if (s == -INFINITY) return 1;
    if (s == INFINITY) return kBuckets - 1;
    const float t = (s - smin) * scale;  // monotone in s
    int b = (int)t;
    b = b < 0 ? 0 : (b > kBuckets - 4 ? kBuckets - 4 : b);
    return 2 + b;
}

__device__ __forceinline__ int warp_id() { return threadIdx.x >> 5; }

__device__ __forceinline__ float block_min(float v, float *wred) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fminf(v, __shfl_xor_sync(kFull, v, o));
    if ((threadIdx.x & 31) == 0) wred[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = wred[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fminf(r, wred[w]);
    __syncthreads();
    return r;
}

__device__ __forceinline__ float block_max(float v, float *wred) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    if ((threadIdx.x & 31) == 0) wred[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = wred[0];
    for (int w = 1; w < (int)(blockDim.x >> 5); ++w) r = fmaxf(r, wred[w]);
    __syncthreads();
    return r;
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ scores, int f, int kind, int k, float tau,
              int32_t *__restrict__ idx, int ld_idx, int32_t *__restrict__ count,
              uint32_t *__restrict__ mask) {
    extern __shared__ uint32_t sm[];
    float *vals = reinterpret_cast<float *>(sm);      // [f] scores
    uint32_t *hist = sm + f;                           // [kBuckets]; later candidates
    __shared__ int wsum[32];
    __shared__ float wred[32];
    __shared__ uint32_t tots[kSelThreads];
    __shared__ uint32_t above[kSelThreads];
    __shared__ uint32_t s_bucket, s_rem, s_pivot, s_need, s_ncand, s_fill;

    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31;
    const int words = (f + 31) >> 5;
    const float *s = scores + (size_t)b * f;
    int32_t *out = idx + (size_t)b * ld_idx;

    pdl_launch_dependents();  // single CTA: let the consumer kernel get resident
    pdl_wait();  // scores come from the previous kernel

    float lo = INFINITY, hi = -INFINITY;
    if ((f & 3) == 0 && (reinterpret_cast<uintptr_t>(s) & 15) == 0) {
        // all of a thread's 16-byte loads are in flight together
        const float4 *s4 = reinterpret_cast<const float4 *>(s);
        float4 *v4 = reinterpret_cast<float4 *>(vals);
        const int f4 = f >> 2;
#pragma unroll 8
        for (int j = tid; j < f4; j += kSelThreads) {
            const float4 v = __ldg(s4 + j);
            v4[j] = v;
            const float e[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int q = 0; q < 4; ++q)
                if (e[q] - e[q] == 0.f) { lo = fminf(lo, e[q]); hi = fmaxf(hi, e[q]); }
        }
    } else {
#pragma unroll 8
        for (int j = tid; j < f; j += kSelThreads) {
            const float v = __ldg(s + j);
            vals[j] = v;
            if (v - v == 0.f) {  // finite
                lo = fminf(lo, v);
                hi = fmaxf(hi, v);
            }
        }
    }
    __syncthreads();

    uint32_t pivot = 0u;
    int need = 0;
    const int kk = k < 0 ? 0 : (k > f ? f : k);
    if (kind == SEL_TOPK && kk > 0 && kk < f) {
        const float smin = block_min(lo, wred);
        const float smax = block_max(hi, wred);
        const float scale = smax > smin ? (float)(kBuckets - 4) / (smax - smin) : 0.f;
        for (int i = tid; i < kBuckets; i += kSelThreads) hist[i] = 0u;
        __syncthreads();
        for (int j = tid; j < f; j += kSelThreads) atomicAdd(&hist[bucket_of(vals[j], smin, scale)], 1u);
        __syncthreads();
        // bucket of the kk-th largest: thread t owns buckets [4t, 4t+4)
        {
            constexpr int BPT = kBuckets / kSelThreads;
            uint32_t cb[BPT], tot = 0;
#pragma unroll
            for (int q = 0; q < BPT; ++q) { cb[q] = hist[tid * BPT + q]; tot += cb[q]; }
            // count of members in buckets above this thread's: a scan in
            // reversed thread order, handed back to the owning thread
            tots[tid] = tot;
            __syncthreads();
            int total_unused;
            const int excl = block_excl_scan((int)tots[kSelThreads - 1 - tid], wsum, &total_unused);
            above[kSelThreads - 1 - tid] = (uint32_t)excl;
            __syncthreads();
            uint32_t run = above[tid];
            const uint32_t rem = (uint32_t)kk;
#pragma unroll
            for (int q = BPT - 1; q >= 0; --q) {
                if (run < rem && run + cb[q] >= rem) {
                    s_bucket = (uint32_t)(tid * BPT + q);
                    s_rem = rem - run;
                    s_ncand = cb[q];
                }
                run += cb[q];
            }
            __syncthreads();
        }
        const int B_ = (int)s_bucket;
        const uint32_t rem = s_rem;       // how many of bucket B_ are taken (>= 1)
        const uint32_t ncand = s_ncand;
        if (ncand <= (uint32_t)kCandMax) {
            // gather bucket B_'s members as (key, id), rank them exactly
            uint32_t *ckey = hist;                 // [kCandMax]
            uint32_t *cid = hist + kCandMax;       // [kCandMax]
            if (tid == 0) s_fill = 0u;
            __syncthreads();
            for (int j = tid; j < f; j += kSelThreads) {
                const float v = vals[j];
                if (bucket_of(v, smin, scale) == B_) {
                    const uint32_t p = atomicAdd(&s_fill, 1u);
                    ckey[p] = score_key(v);
                    cid[p] = (uint32_t)j;
                }
            }
            __syncthreads();
            for (int c = tid; c < (int)ncand; c += kSelThreads) {
                const uint32_t kc = ckey[c], ic = cid[c];
                uint32_t rank = 0;
                for (int o = 0; o < (int)ncand; ++o) {
                    const uint32_t ko = ckey[o];
                    rank += (ko > kc) || (ko == kc && cid[o] < ic);
                }
                if (rank == rem - 1u) s_pivot = kc;
            }
            __syncthreads();
            // ties at the pivot that rank inside the top kk
            int gtc = 0;
            for (int c = tid; c < (int)ncand; c += kSelThreads) gtc += ckey[c] > s_pivot;
            int tot_gt;
            block_excl_scan(gtc, wsum, &tot_gt);
            pivot = s_pivot;
            need = (int)rem - tot_gt;
        } else {
            // a mass of near-equal scores: radix select on the members' keys
            uint32_t prefix = 0u, pmask = 0u, r_ = rem;
            uint32_t *h = hist;  // 256 bins
            for (int pass = 0; pass < 4; ++pass) {
                const int shift = 24 - 8 * pass;
                if (tid < 256) h[tid] = 0u;
                __syncthreads();
                for (int j = tid; j < f; j += kSelThreads) {
                    const float v = vals[j];
                    const uint32_t key = score_key(v);
                    if (bucket_of(v, smin, scale) == B_ && (key & pmask) == prefix)
                        atomicAdd(&h[(key >> shift) & 255u], 1u);
                }
                __syncthreads();
                if (tid < 256) {
                    // bins from the top: thread t looks at digit 255 - t
                    const uint32_t c = h[255 - tid];
                    uint32_t inc = c;
#pragma unroll
                    for (int o = 1; o < 32; o <<= 1) {
                        const uint32_t nn = __shfl_up_sync(kFull, inc, o);
                        if (lane >= o) inc += nn;
                    }
                    if (lane == 31) wsum[tid >> 5] = (int)inc;
                    named_sync(1, 256);
                    uint32_t base_ = 0;
                    for (int w = 0; w < (tid >> 5); ++w) base_ += (uint32_t)wsum[w];
                    const uint32_t ge = base_ + inc, gt = ge - c;
                    if (ge >= r_ && gt < r_) {
                        s_pivot = 255u - (uint32_t)tid;
                        s_need = r_ - gt;
                    }
                }
                __syncthreads();
                prefix |= s_pivot << shift;
                pmask |= 255u << shift;
                r_ = s_need;
                __syncthreads();
            }
            pivot = prefix;
            need = (int)r_;
        }
    }

    // compaction: warp w owns ids [w*S, (w+1)*S), S a multiple of 32, taken
    // 32 at a time; ballots give in-warp ranks and, directly, the mask words
    const int nw = kSelThreads / 32;
    const int S = (((f + nw - 1) / nw) + 31) & ~31;
    const int wbeg = min(warp_id() * S, f), wend = min(wbeg + S, f);
    const unsigned lt = (1u << lane) - 1u;
    auto flags = [&](int j, bool &gt, bool &eq) {
        gt = false;
        eq = false;
        if (j >= wend) return;
        const float v = vals[j];
        if (kind == SEL_TOPK) {
            if (kk == f) gt = true;
            else if (kk > 0) { const uint32_t key = score_key(v); gt = key > pivot; eq = key == pivot; }
        } else if (kind == SEL_THRESHOLD) {
            gt = v >= tau;
        } else {
            gt = v > 0.f;
        }
    };
    int w_gt = 0, w_eq = 0;
    for (int base = wbeg; base < wend; base += 32) {
        bool gt, eq;
        flags(base + lane, gt, eq);
        w_gt += __popc(__ballot_sync(kFull, gt));
        w_eq += __popc(__ballot_sync(kFull, eq));
    }
    // per-warp totals -> exclusive prefixes (ties first: the lowest ids win)
    __shared__ int s_eqb[32], s_selb[32], s_total;
    if (lane == 0) { tots[warp_id()] = (uint32_t)w_gt; above[warp_id()] = (uint32_t)w_eq; }
    __syncthreads();
    if (warp_id() == 0) {
        const int g_ = (int)tots[lane], e_ = (int)above[lane];
        int eb = e_;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) { const int nn = __shfl_up_sync(kFull, eb, o); if (lane >= o) eb += nn; }
        eb -= e_;                                   // ties in earlier warps
        const int take = max(0, min(e_, need - eb));
        const int sel = g_ + take;
        int sb = sel;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) { const int nn = __shfl_up_sync(kFull, sb, o); if (lane >= o) sb += nn; }
        s_eqb[lane] = eb;
        s_selb[lane] = sb - sel;
        if (lane == 31) s_total = sb;
    }
    __syncthreads();
    int eq_run = s_eqb[warp_id()], pos = s_selb[warp_id()];
    for (int base = wbeg; base < wend; base += 32) {
        bool gt, eq;
        const int j = base + lane;
        flags(j, gt, eq);
        const unsigned be = __ballot_sync(kFull, eq);
        const bool take = gt || (eq && eq_run + __popc(be & lt) < need);
        const unsigned bs = __ballot_sync(kFull, take);
        if (take) out[pos + __popc(bs & lt)] = j;
        if (mask && lane == 0) mask[(size_t)b * words + (base >> 5)] = bs;
        eq_run += __popc(be);
        pos += __popc(bs);
    }
    if (tid == 0) count[b] = s_total;
}

// ---------------------------------------------------------------------------
// Cluster variant: one thread-block cluster of kCl CTAs per token row.  CTA r
// owns the 32-aligned id slice [r*S, (r+1)*S).  The same four steps run with
// the element work split kCl ways; the CTAs exchange min/max, histogram
// slices, the pivot bucket's members and their per-CTA counts through
// distributed shared memory, separated by hardware cluster barriers (no global
// atomics, no grid-wide barrier).
// ---------------------------------------------------------------------------
constexpr int kCl = 8;
constexpr int kClThreads = 1024;
constexpr int kClSliceMax = 6144;            // f <= kCl * kClSliceMax
constexpr int kClBinsPerCta = kBuckets / kCl;

struct ClSmem {
    float vals[kClSliceMax];
    uint32_t hist[kBuckets];
    uint32_t red[kClBinsPerCta];
    uint32_t ckey[kCandMax];
    uint32_t cid[kCandMax];
    uint32_t wtot[32][2];
    uint32_t loc[kClBinsPerCta];             // a remote bin slice, copied locally
    float rlo[kCl], rhi[kCl];
    uint32_t rtot[kCl];
    int rgt[kCl], req[kCl];
    float lo, hi;
    uint32_t slice_total;
    uint32_t ncand_fill;
    int cta_gt, cta_eq;
    uint32_t s_bucket, s_rem, s_ncand, s_pivot;
    int s_need, s_base, s_eqb, s_total, s_slow;
};

__device__ __forceinline__ uint32_t cl_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cl_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// address of the same shared variable in CTA `rank` of the cluster
__device__ __forceinline__ uint32_t cl_map(const void *p, uint32_t rank) {
    uint32_t out;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(out) : "r"(smem_addr(p)), "r"(rank));
    return out;
}
__device__ __forceinline__ uint32_t cl_ld_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ float cl_ld_f32(uint32_t addr) { return __uint_as_float(cl_ld_u32(addr)); }
__device__ __forceinline__ void cl_st_u32(uint32_t addr, uint32_t v) {
    asm volatile("st.shared::cluster.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t cl_atom_add(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}

__global__ void __launch_bounds__(kClThreads)
select_cluster_kernel(const float *__restrict__ scores, int f, int kind, int k, float tau,
                      int32_t *__restrict__ idx, int ld_idx, int32_t *__restrict__ count,
                      uint32_t *__restrict__ mask) {
    extern __shared__ __align__(16) uint8_t dyn[];
    ClSmem &S = *reinterpret_cast<ClSmem *>(dyn);
    __shared__ int wsum[32];
    __shared__ float wred[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cl_rank();
    const int b = blockIdx.x / kCl;
    const int words = (f + 31) >> 5;
    const int SL = (((f + kCl - 1) / kCl) + 31) & ~31;
    const int beg = min((int)rank * SL, f), end = min(beg + SL, f);
    const int n_my = end - beg;
    const float *s = scores + (size_t)b * f;
    int32_t *out = idx + (size_t)b * ld_idx;

    pdl_launch_dependents();
    pdl_wait();  // scores come from the previous kernel

    float lo = INFINITY, hi = -INFINITY;
    for (int j = tid; j < n_my; j += kClThreads) {
        const float v = __ldg(s + beg + j);
        S.vals[j] = v;
        if (v - v == 0.f) { lo = fminf(lo, v); hi = fmaxf(hi, v); }
    }
    __syncthreads();  // vals[] is read across threads from here on
    const int kk = k < 0 ? 0 : (k > f ? f : k);
    const bool radix = kind == SEL_TOPK && kk > 0 && kk < f;
    uint32_t pivot = 0u;
    int need = 0;
    if (radix) {
        lo = block_min(lo, wred);
        hi = block_max(hi, wred);
        if (tid == 0) { S.lo = lo; S.hi = hi; S.ncand_fill = 0u; }
        for (int i = tid; i < kBuckets; i += kClThreads) S.hist[i] = 0u;
        cl_sync();
        // cluster-wide min / max (every CTA the same): one remote load per CTA
        if (tid < kCl) {
            S.rlo[tid] = cl_ld_f32(cl_map(&S.lo, (uint32_t)tid));
            S.rhi[tid] = cl_ld_f32(cl_map(&S.hi, (uint32_t)tid));
        }
        __syncthreads();
        float smin = INFINITY, smax = -INFINITY;
#pragma unroll
        for (int r = 0; r < kCl; ++r) { smin = fminf(smin, S.rlo[r]); smax = fmaxf(smax, S.rhi[r]); }
        const float scale = smax > smin ? (float)(kBuckets - 4) / (smax - smin) : 0.f;
        for (int j = tid; j < n_my; j += kClThreads) atomicAdd(&S.hist[bucket_of(S.vals[j], smin, scale)], 1u);
        cl_sync();
        // reduce-scatter: this CTA sums bins [rank*512, rank*512 + 512) over the cluster
        uint32_t part = 0;
        if (tid < kClBinsPerCta) {
            const int bin = (int)rank * kClBinsPerCta + tid;
            uint32_t sum = 0;
            for (uint32_t r = 0; r < kCl; ++r) sum += cl_ld_u32(cl_map(&S.hist[bin], r));
            S.red[tid] = sum;
            part = sum;
        }
        int tot;
        block_excl_scan((int)part, wsum, &tot);
        if (tid == 0) S.slice_total = (uint32_t)tot;
        cl_sync();
        // which CTA's bin slice holds the kk-th largest (slices are ordered by
        // score: the last CTA has the top bins), then which bin
        if (tid < kCl) S.rtot[tid] = cl_ld_u32(cl_map(&S.slice_total, (uint32_t)tid));
        __syncthreads();
        int owner = 0;
        uint32_t above_owner = 0;
        {
            uint32_t run = 0;
            for (int r = kCl - 1; r >= 0; --r) {
                if (run + S.rtot[r] >= (uint32_t)kk) { owner = r; break; }
                run += S.rtot[r];
            }
            above_owner = run;
        }
        if (tid < kClBinsPerCta) S.loc[tid] = cl_ld_u32(cl_map(&S.red[tid], (uint32_t)owner));
        __syncthreads();
        {
            // suffix counts over the owner's bins: thread t (< 512) holds bin t
            const uint32_t cb = tid < kClBinsPerCta ? S.loc[tid] : 0u;
            int tot_unused;
            // reversed scan: thread t feeds bin (511 - t)
            const uint32_t rb = tid < kClBinsPerCta ? S.loc[kClBinsPerCta - 1 - tid] : 0u;
            const int excl = block_excl_scan((int)rb, wsum, &tot_unused);
            __syncthreads();
            if (tid < kClBinsPerCta) S.hist[kClBinsPerCta - 1 - tid] = (uint32_t)excl;  // count above bin
            __syncthreads();
            if (tid < kClBinsPerCta) {
                const uint32_t run = above_owner + S.hist[tid];
                if (run < (uint32_t)kk && run + cb >= (uint32_t)kk) {
                    S.s_bucket = (uint32_t)(owner * kClBinsPerCta + tid);
                    S.s_rem = (uint32_t)kk - run;
                    S.s_ncand = cb;
                }
            }
        }
        __syncthreads();
        const int B_ = (int)S.s_bucket;
        const uint32_t rem = S.s_rem, ncand = S.s_ncand;
        if (ncand <= (uint32_t)kCandMax) {
            // every CTA sends its members of bucket B_ to CTA 0
            const uint32_t fill0 = cl_map(&S.ncand_fill, 0);
            for (int j = tid; j < n_my; j += kClThreads) {
                const float v = S.vals[j];
                if (bucket_of(v, smin, scale) == B_) {
                    const uint32_t p = cl_atom_add(fill0, 1u);
                    cl_st_u32(cl_map(&S.ckey[p], 0), score_key(v));
                    cl_st_u32(cl_map(&S.cid[p], 0), (uint32_t)(beg + j));
                }
            }
            cl_sync();
            // every CTA copies the members from CTA 0 once, then ranks them
            // locally: the member of rank rem-1 is the pivot
            if (rank != 0) {
                const uint32_t ck0 = cl_map(&S.ckey[0], 0), ci0 = cl_map(&S.cid[0], 0);
                for (int c = tid; c < (int)ncand; c += kClThreads) {
                    S.ckey[c] = cl_ld_u32(ck0 + 4u * c);
                    S.cid[c] = cl_ld_u32(ci0 + 4u * c);
                }
            }
            __syncthreads();
            for (int c = tid; c < (int)ncand; c += kClThreads) {
                const uint32_t kc = S.ckey[c], ic = S.cid[c];
                uint32_t rk = 0;
                for (int o = 0; o < (int)ncand; ++o) {
                    const uint32_t ko = S.ckey[o];
                    rk += (ko > kc) || (ko == kc && S.cid[o] < ic);
                }
                if (rk == rem - 1u) S.s_pivot = kc;
            }
            __syncthreads();
            int gtc = 0;
            for (int c = tid; c < (int)ncand; c += kClThreads) gtc += S.ckey[c] > S.s_pivot;
            int tot_gt;
            block_excl_scan(gtc, wsum, &tot_gt);
            pivot = S.s_pivot;
            need = (int)rem - tot_gt;
        } else {
            // a mass of equal scores: every CTA resolves it alone from the full row
            // (radix select over the members' exact keys, read from global memory)
            uint32_t prefix = 0u, pmask = 0u, r_ = rem;
            uint32_t *h = S.hist;
            for (int pass = 0; pass < 4; ++pass) {
                const int shift = 24 - 8 * pass;
                __syncthreads();
                if (tid < 256) h[tid] = 0u;
                __syncthreads();
                for (int j = tid; j < f; j += kClThreads) {
                    const float v = __ldg(s + j);
                    const uint32_t key = score_key(v);
                    if (bucket_of(v, smin, scale) == B_ && (key & pmask) == prefix)
                        atomicAdd(&h[(key >> shift) & 255u], 1u);
                }
                __syncthreads();
                if (tid == 0) {
                    uint32_t run = 0;
                    for (int dgt = 255; dgt >= 0; --dgt) {
                        const uint32_t c = h[dgt];
                        if (run < r_ && run + c >= r_) { S.s_pivot = (uint32_t)dgt; S.s_rem = r_ - run; break; }
                        run += c;
                    }
                }
                __syncthreads();
                prefix |= S.s_pivot << shift;
                pmask |= 255u << shift;
                r_ = S.s_rem;
            }
            pivot = prefix;
            need = (int)r_;
        }
    }

    // compaction of this CTA's slice: warp w owns [w*W, (w+1)*W) within it
    const int nw = kClThreads / 32;
    const int WL = (((n_my + nw - 1) / nw) + 31) & ~31;
    const int wbeg = min(warp * WL, n_my), wend = min(wbeg + WL, n_my);
    const unsigned lt = (1u << lane) - 1u;
    auto flags = [&](int jl, bool &gt, bool &eq) {
        gt = false;
        eq = false;
        if (jl >= wend) return;
        const float v = S.vals[jl];
        if (kind == SEL_TOPK) {
            if (kk == f) gt = true;
            else if (kk > 0) { const uint32_t key = score_key(v); gt = key > pivot; eq = key == pivot; }
        } else if (kind == SEL_THRESHOLD) {
            gt = v >= tau;
        } else {
            gt = v > 0.f;
        }
    };
    int w_gt = 0, w_eq = 0;
    for (int base = wbeg; base < wend; base += 32) {
        bool gt, eq;
        flags(base + lane, gt, eq);
        w_gt += __popc(__ballot_sync(kFull, gt));
        w_eq += __popc(__ballot_sync(kFull, eq));
    }
    if (lane == 0) { S.wtot[warp][0] = (uint32_t)w_gt; S.wtot[warp][1] = (uint32_t)w_eq; }
    __syncthreads();
    if (tid == 0) {
        int g_ = 0, e_ = 0;
        for (int w = 0; w < nw; ++w) { g_ += (int)S.wtot[w][0]; e_ += (int)S.wtot[w][1]; }
        S.cta_gt = g_;
        S.cta_eq = e_;
    }
    cl_sync();
    // this CTA's place: ties and selections of the CTAs before it
    if (tid < kCl) {
        S.rgt[tid] = (int)cl_ld_u32(cl_map(&S.cta_gt, (uint32_t)tid));
        S.req[tid] = (int)cl_ld_u32(cl_map(&S.cta_eq, (uint32_t)tid));
    }
    __syncthreads();
    if (tid == 0) {
        int eqb = 0, selb = 0;
        for (int r = 0; r < kCl; ++r) {
            const int take = max(0, min(S.req[r], need - eqb));
            if (r == (int)rank) { S.s_base = selb; S.s_eqb = eqb; }
            eqb += S.req[r];
            selb += S.rgt[r] + take;
        }
        S.s_total = selb;
    }
    __syncthreads();
    if (warp == 0) {
        // warp offsets inside the CTA (ties first, so the lowest ids win)
        const int g_ = (int)S.wtot[lane][0], e_ = (int)S.wtot[lane][1];
        int eb = e_;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) { const int nn = __shfl_up_sync(kFull, eb, o); if (lane >= o) eb += nn; }
        eb = eb - e_ + S.s_eqb;
        const int take = max(0, min(e_, need - eb));
        const int sel = g_ + take;
        int sb = sel;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) { const int nn = __shfl_up_sync(kFull, sb, o); if (lane >= o) sb += nn; }
        S.wtot[lane][0] = (uint32_t)(sb - sel + S.s_base);
        S.wtot[lane][1] = (uint32_t)eb;
    }
    __syncthreads();
    int pos = (int)S.wtot[warp][0], eq_run = (int)S.wtot[warp][1];
    for (int base = wbeg; base < wend; base += 32) {
        bool gt, eq;
        const int jl = base + lane;
        flags(jl, gt, eq);
        const unsigned be = __ballot_sync(kFull, eq);
        const bool take = gt || (eq && eq_run + __popc(be & lt) < need);
        const unsigned bs = __ballot_sync(kFull, take);
        if (take) out[pos + __popc(bs & lt)] = beg + jl;
        if (mask && lane == 0) mask[(size_t)b * words + ((beg + base) >> 5)] = bs;
        eq_run += __popc(be);
        pos += __popc(bs);
    }
    if (rank == 0 && tid == 0) count[b] = S.s_total;
    cl_sync();  // no CTA leaves while another may still read its shared memory
}

size_t select_smem(int f) { return sizeof(uint32_t) * ((size_t)f + kBuckets); }

bool cluster_select_enabled() {
    static const bool on = [] {
        const char *v = getenv("CS_SELECT_CLUSTER");
        return !(v && v[0] == '0');
    }();
    return on;
}

}  // namespace

cudaError_t launch_select_cluster(const SelectArgs &a, cudaStream_t s) {
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    const size_t smem = sizeof(ClSmem);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(select_cluster_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kCl * a.B);
    cfg.blockDim = dim3(kClThreads);
    cfg.dynamicSmemBytes = smem;
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
    return cudaLaunchKernelEx(&cfg, select_cluster_kernel, a.scores, a.f, (int)a.kind, a.k, a.tau, a.idx,
                              a.ld_idx, a.count, a.mask);
}

cudaError_t launch_select(const SelectArgs &a, cudaStream_t s) {
    if (a.f >= 2048 && a.f <= kCl * kClSliceMax && cluster_select_enabled()) return launch_select_cluster(a, s);
    static int configured_dev = -1;
    int dev = 0;
    cudaGetDevice(&dev);
    if (configured_dev != dev) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)select_smem(kSelectMaxF));
        if (e != cudaSuccess) return e;
        configured_dev = dev;
    }
    return launch(select_kernel, dim3(a.B), dim3(kSelThreads), select_smem(a.f), s, pdl_enabled(), a.scores,
                  a.f, (int)a.kind, a.k, a.tau, a.idx, a.ld_idx, a.count, a.mask);
}

}  // namespace cs
