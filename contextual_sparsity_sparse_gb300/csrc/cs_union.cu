// Batch union of active-neuron masks, and the neuron-major layout packer.
//
// Union source: "Contextual Sparsity and Activation Predictors", section "When
// it breaks": the tokens of a batch have different active sets and the layer
// must read their union.  umask = OR over tokens; uidx = set bits ascending.
// Two kernels over 128-word blocks: the OR (one word per thread), then the
// ids, each block placing its own after the set bits of the words before it.
//
// Packer source: "Contextual Sparsity: Activation-Aware LLM Inference and the
// Deja Vu Paradigm", section "Kernel-Level Implementation" (indexing into the
// row-major down projection breaks coalescing): W_down [d, f] is transposed
// to neuron-major rows, 32x32 tiles through shared memory.
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kUnionThreads = 128;   // words (one per thread) per CTA

// OR of word w over the B masks, 32 (then 8) loads in flight at a time.
__device__ __forceinline__ uint32_t or_word(const uint32_t *masks, int B, int words, int w) {
    uint32_t acc = 0;
    int b = 0;
    for (; b + 32 <= B; b += 32) {
        uint32_t t[32];
#pragma unroll
        for (int i = 0; i < 32; ++i) t[i] = ld_dep(masks + (size_t)(b + i) * words + w);
#pragma unroll
        for (int i = 0; i < 32; ++i) acc |= t[i];
    }
    for (; b + 8 <= B; b += 8) {
        uint32_t t[8];
#pragma unroll
        for (int i = 0; i < 8; ++i) t[i] = ld_dep(masks + (size_t)(b + i) * words + w);
#pragma unroll
        for (int i = 0; i < 8; ++i) acc |= t[i];
    }
    for (; b < B; ++b) acc |= ld_dep(masks + (size_t)b * words + w);
    return acc;
}

// 1. umask: one word per thread (bits past f cleared).
__global__ void __launch_bounds__(kUnionThreads) union_or_kernel(const uint32_t *masks, int B, int f,
                                                                  uint32_t *umask) {
    pdl_launch_dependents();
    pdl_wait();  // the masks may come from an earlier kernel
    const int words = (f + 31) >> 5;
    const int w = blockIdx.x * kUnionThreads + threadIdx.x;
    if (w < words) {
        uint32_t u = or_word(masks, B, words, w);
        if (w == words - 1 && (f & 31)) u &= (1u << (f & 31)) - 1u;
        umask[w] = u;
    }
}

// 2. uidx: a CTA's ids start after the set bits of all earlier words (summed
//    here from umask); a block scan places each word's ids, each warp stages
//    its run in shared memory and stores it with coalesced writes.  The last
//    CTA writes the count.
__global__ void __launch_bounds__(kUnionThreads) union_ids_kernel(const uint32_t *umask, int f, int32_t *uidx,
                                                                  int32_t *ucount) {
    __shared__ int32_t stage[kUnionThreads / 32][32 * 32];   // a warp's ids: at most 32 per lane
    __shared__ int wsum[32];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int words = (f + 31) >> 5;
    const int w0 = blockIdx.x * kUnionThreads;
    pdl_launch_dependents();
    pdl_wait();  // umask comes from the OR kernel
    int part = 0;
    for (int w = tid; w < w0; w += kUnionThreads) part += __popc(ld_dep(umask + w));
    int before;
    (void)block_excl_scan(part, wsum, &before);
    const int w = w0 + tid;
    const uint32_t u = w < words ? ld_dep(umask + w) : 0u;
    const int n = __popc(u);
    int total;
    const int pos = block_excl_scan(n, wsum, &total);
    const int wbase = __shfl_sync(kFull, pos, 0);
    int *st = stage[warp];
    int o = pos - wbase;
    for (uint32_t x = u; x; x &= x - 1) st[o++] = w * 32 + __ffs(x) - 1;
    __syncwarp();
    const int run = __shfl_sync(kFull, pos - wbase + n, 31);
    for (int q = lane; q < run; q += 32) uidx[before + wbase + q] = st[q];
    if (blockIdx.x == gridDim.x - 1 && tid == 0) *ucount = before + total;
}

template <typename S> __device__ __forceinline__ float load_as_float(const void *p, size_t i);
template <> __device__ __forceinline__ float load_as_float<float>(const void *p, size_t i) {
    return static_cast<const float *>(p)[i];
}
template <> __device__ __forceinline__ float load_as_float<__half>(const void *p, size_t i) {
    return __half2float(static_cast<const __half *>(p)[i]);
}
template <> __device__ __forceinline__ float load_as_float<__nv_bfloat16>(const void *p, size_t i) {
    return __bfloat162float(static_cast<const __nv_bfloat16 *>(p)[i]);
}

template <typename D> __device__ __forceinline__ void store_from_float(void *p, size_t i, float v);
template <> __device__ __forceinline__ void store_from_float<float>(void *p, size_t i, float v) {
    static_cast<float *>(p)[i] = v;
}
template <> __device__ __forceinline__ void store_from_float<__half>(void *p, size_t i, float v) {
    static_cast<__half *>(p)[i] = __float2half_rn(v);
}
template <> __device__ __forceinline__ void store_from_float<__nv_bfloat16>(void *p, size_t i, float v) {
    static_cast<__nv_bfloat16 *>(p)[i] = __float2bfloat16_rn(v);
}

template <typename S, typename D>
__global__ void __launch_bounds__(256)
transpose_kernel(const void *__restrict__ src, int rows, int cols, int ld_src, void *__restrict__ dst,
                 int ld_dst) {
    __shared__ float tile[32][33];
    const int c0 = blockIdx.x * 32, r0 = blockIdx.y * 32;
    const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
    pdl_wait();
    for (int yy = ty; yy < 32; yy += 8) {
        const int r = r0 + yy, c = c0 + tx;
        tile[yy][tx] = (r < rows && c < cols) ? load_as_float<S>(src, (size_t)r * ld_src + c) : 0.f;
    }
    __syncthreads();
    for (int yy = ty; yy < 32; yy += 8) {
        const int c = c0 + yy, r = r0 + tx;  // dst row = source column
        if (c < cols && r < rows) store_from_float<D>(dst, (size_t)c * ld_dst + r, tile[tx][yy]);
    }
}

template <typename S>
cudaError_t pick_dst(const void *src, int rows, int cols, int ld_src, void *dst, cs_dtype dt, int ld_dst,
                     cudaStream_t s) {
    dim3 g((cols + 31) / 32, (rows + 31) / 32);
    const bool pdl = pdl_enabled();
    switch (dt) {
    case CS_F32: return launch(transpose_kernel<S, float>, g, dim3(256), 0, s, pdl, src, rows, cols, ld_src, dst, ld_dst);
    case CS_F16: return launch(transpose_kernel<S, __half>, g, dim3(256), 0, s, pdl, src, rows, cols, ld_src, dst, ld_dst);
    default: return launch(transpose_kernel<S, __nv_bfloat16>, g, dim3(256), 0, s, pdl, src, rows, cols, ld_src, dst, ld_dst);
    }
}

}  // namespace

cudaError_t launch_union(const UnionArgs &a, cudaStream_t s) {
    const int words = (a.f + 31) >> 5;
    const dim3 g((words + kUnionThreads - 1) / kUnionThreads);
    cudaError_t e = launch(union_or_kernel, g, dim3(kUnionThreads), 0, s, pdl_enabled(), a.masks, a.B, a.f, a.umask);
    if (e != cudaSuccess) return e;
    return launch(union_ids_kernel, g, dim3(kUnionThreads), 0, s, pdl_enabled(),
                  static_cast<const uint32_t *>(a.umask), a.f, a.uidx, a.ucount);
}

cudaError_t launch_transpose(const void *src, cs_dtype st, int rows, int cols, int ld_src, void *dst,
                             cs_dtype dt, int ld_dst, cudaStream_t s) {
    switch (st) {
    case CS_F32: return pick_dst<float>(src, rows, cols, ld_src, dst, dt, ld_dst, s);
    case CS_F16: return pick_dst<__half>(src, rows, cols, ld_src, dst, dt, ld_dst, s);
    default: return pick_dst<__nv_bfloat16>(src, rows, cols, ld_src, dst, dt, ld_dst, s);
    }
}

}  // namespace cs
