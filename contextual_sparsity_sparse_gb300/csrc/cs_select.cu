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

size_t select_smem(int f) { return sizeof(uint32_t) * ((size_t)f + kBuckets); }

}  // namespace

cudaError_t launch_select(const SelectArgs &a, cudaStream_t s) {
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
