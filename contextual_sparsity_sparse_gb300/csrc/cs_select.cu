// Selection: top-k, threshold and positive-pre-activation compaction.
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (the top-k scores are the
// predicted active set); "Activation sparsity", section "Implementation
// sketch" (predict_active: scores >= threshold); "Contextual Sparsity and
// Activation Predictors", first section (a neuron is active when its gate
// pre-activation passes the ReLU).
//
// One CTA of 1024 threads per token row.  Top-k is an exact radix select on
// order-preserving 32-bit keys (four 8-bit digit passes over a shared-memory
// histogram, warp-aggregated with match.any), which yields the k-th key K and
// the number of ties at K to take.  Compaction is in ascending neuron order:
// each thread owns a contiguous segment, two block scans give (a) the ties
// that precede the segment, so the lowest-id ties are taken, and (b) the
// output position of the segment.
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kSelThreads = 1024;

// Order-preserving key: larger score -> larger key.  -0 is folded onto +0;
// NaN maps to 0, below the key of -inf (0x007fffff).
__device__ __forceinline__ uint32_t score_key(float s) {
    if (s != s) return 0u;
    uint32_t u = __float_as_uint(s);
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kSelThreads)
select_kernel(const float *__restrict__ scores, int f, int kind, int k, float tau,
              int32_t *__restrict__ idx, int ld_idx, int32_t *__restrict__ count,
              uint32_t *__restrict__ mask) {
    extern __shared__ uint32_t sm[];
    uint32_t *keys = sm;                 // [f]
    uint32_t *smask = sm + f;            // [words]
    __shared__ uint32_t hist[256];
    __shared__ int wsum[32];
    __shared__ uint32_t s_digit, s_rem;

    const int b = blockIdx.x;
    const int tid = threadIdx.x, lane = tid & 31;
    const int words = (f + 31) >> 5;
    const float *s = scores + (size_t)b * f;
    int32_t *out = idx + (size_t)b * ld_idx;

    pdl_wait();  // scores come from the previous kernel

    for (int w = tid; w < words; w += kSelThreads) smask[w] = 0u;

    // keys: top-k ranks keys; threshold/positive keep the raw float bits
    for (int j = tid; j < f; j += kSelThreads) {
        const float v = s[j];
        keys[j] = kind == SEL_TOPK ? score_key(v) : __float_as_uint(v);
    }
    __syncthreads();

    uint32_t pivot = 0u;
    int need = 0;  // ties at the pivot to take (top-k)
    int kk = k < 0 ? 0 : (k > f ? f : k);
    if (kind == SEL_TOPK && kk > 0 && kk < f) {
        uint32_t prefix = 0u, pmask = 0u;
        uint32_t rem = (uint32_t)kk;
#pragma unroll 1
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            if (tid < 256) hist[tid] = 0u;
            __syncthreads();
#pragma unroll 1
            for (int base = 0; base < f; base += kSelThreads) {
                const int j = base + tid;
                uint32_t key = j < f ? keys[j] : 0u;
                const bool valid = j < f && (key & pmask) == prefix;
                const unsigned act = __ballot_sync(kFull, valid);
                if (valid) {
                    const uint32_t dig = (key >> shift) & 255u;
                    const unsigned peers = __match_any_sync(act, dig);
                    if (lane == __ffs(peers) - 1) atomicAdd(&hist[dig], (uint32_t)__popc(peers));
                }
            }
            __syncthreads();
            // thread t < 256 looks at digit 255 - t; inclusive scan over t gives
            // the number of candidates with digit >= 255 - t
            if (tid < 256) {
                const uint32_t c = hist[255 - tid];
                uint32_t inc = c;
#pragma unroll
                for (int o = 1; o < 32; o <<= 1) {
                    uint32_t n = __shfl_up_sync(kFull, inc, o);
                    if (lane >= o) inc += n;
                }
                if (lane == 31) wsum[tid >> 5] = (int)inc;
                __syncwarp();
                // wait for the 8 warp totals (only warps 0..7 take part)
                asm volatile("bar.sync 1, 256;" ::: "memory");
                uint32_t base_ = 0;
                for (int w = 0; w < (tid >> 5); ++w) base_ += (uint32_t)wsum[w];
                const uint32_t ge = base_ + inc;        // candidates with digit >= dig
                const uint32_t gt = ge - c;              // candidates with digit > dig
                if (ge >= rem && gt < rem) {
                    s_digit = 255u - (uint32_t)tid;
                    s_rem = rem - gt;
                }
            }
            __syncthreads();
            prefix |= s_digit << shift;
            pmask |= 255u << shift;
            rem = s_rem;
            __syncthreads();
        }
        pivot = prefix;
        need = (int)rem;
    }

    // segment of this thread
    const int E = (f + kSelThreads - 1) / kSelThreads;
    const int beg = min(tid * E, f), end = min(beg + E, f);
    int n_gt = 0, n_eq = 0;
    for (int j = beg; j < end; ++j) {
        const uint32_t key = keys[j];
        bool gt, eq = false;
        if (kind == SEL_TOPK) {
            if (kk == 0) gt = false;
            else if (kk == f) gt = true;
            else { gt = key > pivot; eq = key == pivot; }
        } else if (kind == SEL_THRESHOLD) {
            gt = __uint_as_float(key) >= tau;
        } else {
            gt = __uint_as_float(key) > 0.f;
        }
        n_gt += gt;
        n_eq += eq;
    }
    int total_eq;
    const int eq_before = block_excl_scan(n_eq, wsum, &total_eq);
    const int take_eq = max(0, min(n_eq, need - eq_before));
    int total;
    int pos = block_excl_scan(n_gt + take_eq, wsum, &total);
    int eq_seen = eq_before;
    for (int j = beg; j < end; ++j) {
        const uint32_t key = keys[j];
        bool sel;
        if (kind == SEL_TOPK) {
            if (kk == 0) sel = false;
            else if (kk == f) sel = true;
            else if (key > pivot) sel = true;
            else if (key == pivot) sel = eq_seen++ < need;
            else sel = false;
        } else if (kind == SEL_THRESHOLD) {
            sel = __uint_as_float(key) >= tau;
        } else {
            sel = __uint_as_float(key) > 0.f;
        }
        if (sel) {
            out[pos++] = j;
            if (mask) atomicOr(&smask[j >> 5], 1u << (j & 31));
        }
    }
    if (tid == 0) count[b] = total;
    if (mask) {
        __syncthreads();
        for (int w = tid; w < words; w += kSelThreads) mask[(size_t)b * words + w] = smask[w];
    }
}

}  // namespace

cudaError_t launch_select(const SelectArgs &a, cudaStream_t s) {
    const int words = (a.f + 31) / 32;
    const size_t smem = sizeof(uint32_t) * ((size_t)a.f + words);
    static bool configured = false;
    if (!configured) {
        cudaError_t e = cudaFuncSetAttribute(select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                             (int)(sizeof(uint32_t) * (kSelectMaxF + kSelectMaxF / 32)));
        if (e != cudaSuccess) return e;
        configured = true;
    }
    return launch(select_kernel, dim3(a.B), dim3(kSelThreads), smem, s, pdl_enabled(), a.scores,
                  a.f, (int)a.kind, a.k, a.tau, a.idx, a.ld_idx, a.count, a.mask);
}

}  // namespace cs
