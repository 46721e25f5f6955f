// Internal device and host helpers shared by the library's translation units.
// Nothing here is part of the public C ABI (include/cs.h).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <utility>

#include "cs.h"

namespace cs {

constexpr unsigned kFull = 0xffffffffu;

// ----------------------------------------------------------------------------
// Workspace layout.  The first 256 bytes are control words; the error word is
// at offset 0.  Every region starts on a 256-byte boundary.
// ----------------------------------------------------------------------------
constexpr size_t kControlBytes = 256;

struct WsLayout {
    size_t err = 0;         // uint32 error bits
    size_t part = 0;        // [G, B, dp] fp32 per-CTA partial sums of y
    size_t h = 0;           // [B, r] fp32 predictor bottleneck
    size_t st_x = 0;        // [dp] fp32 stack ping-pong buffer
    size_t st_scores = 0;   // [f] fp32 stack scores
    size_t st_pre = 0;      // [f] fp32 stack pre-activations (exact mode)
    size_t st_idx = 0;      // [2, f] int32 stack selection slots
    size_t st_count = 0;    // [2] int32 stack counts
    size_t st_h = 0;        // [r] fp32 stack predictor bottleneck
    size_t io_y = 0;        // [dp] fp32 single-layer step: y staged for a host copy
    size_t io_x = 0;        // [dp] fp32 stack: x staged for host copies
    size_t bt_a = 0;        // [Bmax, fu] fp32 batched activations
    size_t tc = 0;          // tensor-core path buffers (tc_workspace_bytes), 0 bytes when B < 2
    size_t total = 0;
    int G = 0;              // partial-sum slots (CTAs of the gather kernel)
    int dp = 0;             // padded row length of partial sums
};

inline size_t align256(size_t v) { return (v + 255) & ~size_t(255); }

WsLayout ws_layout(int d, int f, int r, int B, int num_sms);
int device_sm_count();

// ----------------------------------------------------------------------------
// dtype traits: 16 bytes hold N elements
// ----------------------------------------------------------------------------
template <typename T> struct Vec;
template <> struct Vec<float> { static constexpr int N = 4; };
template <> struct Vec<__half> { static constexpr int N = 8; };
template <> struct Vec<__nv_bfloat16> { static constexpr int N = 8; };

__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[4], const float *) {
    o[0] = __uint_as_float(v.x); o[1] = __uint_as_float(v.y);
    o[2] = __uint_as_float(v.z); o[3] = __uint_as_float(v.w);
}

__device__ __forceinline__ void half2x(uint32_t w, float &lo, float &hi) {
    __half2 h = *reinterpret_cast<const __half2 *>(&w);
    float2 f = __half22float2(h);
    lo = f.x; hi = f.y;
}

__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[8], const __half *) {
    half2x(v.x, o[0], o[1]); half2x(v.y, o[2], o[3]);
    half2x(v.z, o[4], o[5]); half2x(v.w, o[6], o[7]);
}

// bf16 -> fp32 is exact: the bf16 bits are the top half of the fp32 bits.
__device__ __forceinline__ void bf2x(uint32_t w, float &lo, float &hi) {
    lo = __uint_as_float(w << 16);
    hi = __uint_as_float(w & 0xffff0000u);
}

__device__ __forceinline__ void unpack16(const uint4 &v, float (&o)[8], const __nv_bfloat16 *) {
    bf2x(v.x, o[0], o[1]); bf2x(v.y, o[2], o[3]);
    bf2x(v.z, o[4], o[5]); bf2x(v.w, o[6], o[7]);
}

template <typename T>
__device__ __forceinline__ void unpack(const uint4 &v, float (&o)[Vec<T>::N]) {
    unpack16(v, o, static_cast<const T *>(nullptr));
}

// Streaming 16-byte load that does not allocate in L1 (weights are read once).
__device__ __forceinline__ uint4 ld_stream(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

// ----------------------------------------------------------------------------
// Programmatic dependent launch.  wait: block until the grids this one
// depends on have completed and their writes are visible (a no-op when the
// launch carried no programmatic dependency).  launch_dependents: allow the
// next grid in the stream to start its prologue.
// ----------------------------------------------------------------------------
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ----------------------------------------------------------------------------
// Loads of data that an earlier kernel of the stream wrote (scores, index
// lists, counts, activations, partial sums).  With programmatic dependent
// launch this kernel may start before that kernel ends, so such loads must
// stay after pdl_wait().  __ldg is a non-coherent load that the compiler may
// treat as invariant and hoist above the wait (it did, once its loads were
// fully unrolled); these are plain loads, which the wait's memory clobber
// keeps after it (the pointers they read through are not __restrict__, which
// would let the compiler treat them as read-only in the same way).  Weights
// and other data that no kernel writes keep __ldg.
// ----------------------------------------------------------------------------
template <typename T>
__device__ __forceinline__ T ld_dep(const T *p) { return *p; }

// ----------------------------------------------------------------------------
// mbarrier + bulk async copy (TMA engine, non-tensor form)
// ----------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_addr(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_addr(bar)), "r"(count)
                 : "memory");
}

__device__ __forceinline__ void mbar_fence_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_addr(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15):
// sync waits for `count` arrivals (its own included); arrive does not wait.
__device__ __forceinline__ void named_sync(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(int id, int count) {
    asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_addr(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Wait for phase `parity` of an mbarrier, giving up after `limit_ns`.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity,
                                          uint64_t limit_ns = 2000000000ull) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 32; ++i)
            if (mbar_try_wait(bar, parity)) return true;
        if (global_ns() - t0 > limit_ns) return false;
    }
}

// Global -> shared bulk copy; completion is counted in bytes on `bar`.
// dst, src and bytes must be multiples of 16.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes,
                                         uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::
            "r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar))
        : "memory");
}

// Per-thread asynchronous global -> shared copies (16 bytes, or 4), grouped
// with commit/wait.  Only the issuing thread's own copies are waited for.
__device__ __forceinline__ void cp_async16(void *dst, const void *src) {
    asm volatile("cp.async.cg.shared.global.L2::128B [%0], [%1], 16;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async4(void *dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_addr(dst)), "l"(src) : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Same, with an L2 eviction-priority policy (evict_first for data read once).
__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t p;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
    return p;
}

__device__ __forceinline__ void bulk_g2s_hint(void *dst, const void *src, uint32_t bytes,
                                              uint64_t *bar, uint64_t policy) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint "
        "[%0], [%1], %2, [%3], %4;" ::"r"(smem_addr(dst)),
        "l"(src), "r"(bytes), "r"(smem_addr(bar)), "l"(policy)
        : "memory");
}

// The gate's activation: relu(g), or silu(g) = g / (1 + e^-g) with CUDA's
// expf and an IEEE division (silu(-inf) = -inf / inf is NaN, never taken by
// a magnitude cut; +inf stays +inf).
__device__ __forceinline__ float gate_act(int act, float g) {
    return act == CS_ACT_SILU ? g / (1.f + expf(-g)) : fmaxf(g, 0.f);
}

// ----------------------------------------------------------------------------
// Reductions (fixed order, so results are bit-reproducible)
// ----------------------------------------------------------------------------
__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// Exclusive prefix sum over the block of one int per thread.  `wsum` is
// shared scratch of 32 ints.  Returns the exclusive prefix; *total gets the
// block sum.  Every thread of the block must call it.
__device__ __forceinline__ int block_excl_scan(int v, int *wsum, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int nw = (blockDim.x + 31) >> 5;
    int inc = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(kFull, inc, o);
        if (lane >= o) inc += n;
    }
    if (lane == 31) wsum[warp] = inc;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nw ? wsum[lane] : 0;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(kFull, w, o);
            if (lane >= o) w += n;
        }
        if (lane < nw) wsum[lane] = w;
    }
    __syncthreads();
    const int base = warp > 0 ? wsum[warp - 1] : 0;
    *total = wsum[nw - 1];
    __syncthreads();
    return base + inc - v;
}

// ----------------------------------------------------------------------------
// Host side
// ----------------------------------------------------------------------------
void set_error(const char *fmt, ...);
cs_status cuda_fail(cudaError_t e, const char *what);

// Launch with optional programmatic-dependent-launch attribute.
template <typename... KArgs, typename... Args>
cudaError_t launch(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                   bool pdl, Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    cfg.numAttrs = 0;
    if (pdl) {
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
    }
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Whether launches use programmatic dependent launch (on by default; the
// environment variable CS_PDL=0 turns it off).
bool pdl_enabled();

// ---- internal launchers (stream-ordered, already validated) ----------------
struct PredictArgs {
    int d, r, f, B;
    cs_dtype dtype;
    int ld_down, ld_up;
    const void *p_down, *p_up;
    const float *x;
    float *h;      // [B, r]
    float *scores; // [B, f]
    uint32_t *err = nullptr;
};
cudaError_t launch_predict(const PredictArgs &a, cudaStream_t s);
// out[b, row] = epi(sum_c W[row, c] v[b, c]) for rows < nrows and B tokens of
// v [B, ncols]: epi 0 none, 1 relu, 2 + bias[row] (the predictor's streaming
// GEMV, for calibration batches)
cudaError_t launch_gemv_batch(cs_dtype dt, const void *W, int ldb_bytes, int ncols, int nrows, const float *v,
                              int B, float *out, const float *bias, int epi, uint32_t *err, cudaStream_t s);

// SEL_POSITIVE: relu(s) > tau, i.e. s > tau (tau >= 0); SEL_SILU_MAG:
// |silu(s)| > tau.  Both never take NaN.
enum SelKind { SEL_TOPK = 0, SEL_THRESHOLD = 1, SEL_POSITIVE = 2, SEL_SILU_MAG = 3 };
struct SelectArgs {
    const float *scores;
    int B, f;
    SelKind kind;
    int k;
    float tau;
    int32_t *idx;   // [B, ld_idx], ld_idx >= hot + f
    int ld_idx;
    int32_t *count; // [B]
    uint32_t *mask; // [B, ceil((hot + f) / 32)] or null
    int hot = 0;    // ids 0 .. hot-1 always taken (a multiple of 32); the f scores are neurons hot ..
};
cudaError_t launch_select(const SelectArgs &a, cudaStream_t s);
constexpr int kSelectMaxF = 49152;

struct FfnArgs {
    int d, f, ld, B;
    cs_dtype dtype;
    const void *w_gate, *w_up, *w_down_t;
    const float *bias;
    const float *x;         // [B, d]
    const int32_t *idx;
    const int32_t *count;
    const float *preact;    // exact mode: [f] gate pre-activations (bias included), else null
    float *y;               // [B, d]
    const float *resid;     // null, or [B, d]: y = resid + scale * FFN
    float scale;
    uint32_t *err;
    float *part;            // workspace partials
    int G, dp;
    int act = CS_ACT_RELU;  // the gate's activation
    void *tc_x = nullptr;   // tensor-core path: [NP, d] split activations (or null)
    void *tc_a = nullptr;   // tensor-core path: [NP, roundup(f, 128)] split activations (or null)
};
cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s);

// Head-sparse attention (cs_attn.cu) over one layer's KV cache, with the
// workspace whose partial rows it uses.
struct AttnCall {
    cs_attn_layer layer;
    const void *k_cache, *v_cache;
    int seq_len;
    void *ws;
    size_t ws_bytes;
};
// Checks the layer, the caches and the length (host only), then the
// workspace (its size depends on the device's SM count); both set the error.
cs_status attn_check(const AttnCall &c, const char *who);
cs_status attn_check_ws(const AttnCall &c, const char *who);
// Enqueues y = the listed heads' attention (x 16-byte aligned, y not x).
cudaError_t attn_launch(const AttnCall &c, const float *x, const int32_t *heads, const int32_t *count, float *y,
                        cudaStream_t s);

// Arguments of the gather kernels (one CTA per SM over a chunk of the list).
struct FfnK {
    const uint8_t *w_gate, *w_up, *w_down_t;
    const float *bias, *x, *preact;
    const int32_t *idx, *count;
    float *part;
    uint32_t *err;
    int d, f, B, dp;
    int ldb;        // row pitch in bytes
    int nvec;       // 16-byte vectors per row
    int ng;         // neurons per group
    int sg;         // groups in the ring (2 or 3)
    int act;        // the gate's activation (CS_ACT_*)
};
// The one-token gather with a compile-time group size (cs_ffn1.cu).
bool gather1_applies(const FfnK &k, int B);
cudaError_t launch_gather1(cs_dtype dt, const FfnK &k, size_t smem, int G, bool glu, bool pre, cudaStream_t s);

// y[b, :] = (resid[b, :] + scale *) sum_{c < G'} part[c, b, :], fixed order;
// G' = G, or min(G, *gcount) when gcount (device) is given
cudaError_t launch_ffn_reduce(const float *part, int G, int B, int d, int dp, const float *resid, float scale,
                              float *y, cudaStream_t s, const int32_t *gcount = nullptr);

// Tensor-core (tcgen05) batched path for dense unions: fp16 / bf16 weights,
// d a multiple of 64, 2 <= B <= kTcMaxB.
constexpr int kTcMaxB = 32;
constexpr int kTcDefaultMinB = 4;   // batch from which the tensor-core path is taken
int tc_min_batch();                 // kTcDefaultMinB, or CS_TC_MIN_B from the environment
int tc_act_pitch(int f);
size_t tc_workspace_bytes(int d, int f, int B);
size_t tc_x_bytes(int d, int B);   // the first buffer: split activations X
size_t tc_a_bytes(int f, int B);   // the second: split activations A
size_t tc_pieces_bytes(int B, int P);  // the third: partial tile sums of the gate GEMM
bool tc_path_applies(const FfnArgs &a);
cudaError_t launch_ffn_tc(const FfnArgs &a, cudaStream_t s);

struct PreactArgs {
    int d, f, ld;
    cs_dtype dtype;
    const void *w_gate;
    const float *bias;
    const float *x;
    float *pre;
    uint32_t *err = nullptr;
};
cudaError_t launch_preact(const PreactArgs &a, cudaStream_t s);

struct UnionArgs {
    const uint32_t *masks;
    int B, f;
    uint32_t *umask;
    int32_t *uidx;
    int32_t *ucount;
};
cudaError_t launch_union(const UnionArgs &a, cudaStream_t s);

size_t dtype_size(cs_dtype t);

// Host-side checks of a layer descriptor (sets the error text); *ld_out gets
// the effective row stride.
cs_status validate_layer(const cs_ffn_layer *layer, int *ld_out);

}  // namespace cs
