// Predictor GEMVs.
//
// Source: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja Vu
// Paradigm", section "The Prediction Problem" (SparsityPredictor): a
// bias-free down projection to a small bottleneck, ReLU, and a bias-free up
// projection to one score per neuron.  The page's closing sigmoid is monotone
// and is not applied; scores are logits.  "Contextual Sparsity and Activation
// Predictors", section "The predictor and its budget", bounds what the
// predictor may read; both GEMVs here are pure weight streams.
//
//   P1: h[b, i] = relu(sum_t P_down[i, t] x[b, t])     r rows of d
//   P2: s[b, j] = sum_i P_up[j, i] h[b, i]              f rows of r
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kThreads = 256;

// P1: a CTA owns RPC consecutive rows and TB tokens; its threads stride over
// the rows' 16-byte vectors, so each row is streamed once, coalesced.
template <typename T, int RPC, int TB>
__global__ void __launch_bounds__(kThreads)
pred_down_kernel(const T *__restrict__ W, int ld, int d, int r, const float *__restrict__ x, int B,
                 float *__restrict__ h) {
    constexpr int V = Vec<T>::N;
    __shared__ float red[kThreads / 32][RPC * TB];
    const int row0 = blockIdx.x * RPC;
    const int b0 = blockIdx.y * TB;
    const int nvec = (d + V - 1) / V;
    float acc[RPC][TB];
#pragma unroll
    for (int q = 0; q < RPC; ++q)
#pragma unroll
        for (int t = 0; t < TB; ++t) acc[q][t] = 0.f;

    pdl_wait();  // x may come from the previous kernel in the stream

    for (int v = threadIdx.x; v < nvec; v += kThreads) {
        const int c0 = v * V;
        const int ne = min(V, d - c0);
        uint4 raw[RPC];
#pragma unroll
        for (int q = 0; q < RPC; ++q) {
            const int row = min(row0 + q, r - 1);
            raw[q] = ld_stream(W + (size_t)row * ld + c0);
        }
        float xv[TB][V];
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const int b = min(b0 + t, B - 1);
#pragma unroll
            for (int e = 0; e < V; ++e) xv[t][e] = e < ne ? __ldg(x + (size_t)b * d + c0 + e) : 0.f;
        }
#pragma unroll
        for (int q = 0; q < RPC; ++q) {
            float w[V];
            unpack<T>(raw[q], w);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                if (e >= ne) w[e] = 0.f;
#pragma unroll
                for (int t = 0; t < TB; ++t) acc[q][t] = fmaf(w[e], xv[t][e], acc[q][t]);
            }
        }
    }
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
    for (int q = 0; q < RPC; ++q)
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            float s = warp_sum(acc[q][t]);
            if (lane == 0) red[warp][q * TB + t] = s;
        }
    __syncthreads();
    if (threadIdx.x < RPC * TB) {
        const int q = threadIdx.x / TB, t = threadIdx.x % TB;
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < kThreads / 32; ++w) s += red[w][threadIdx.x];
        const int row = row0 + q, b = b0 + t;
        if (row < r && b < B) h[(size_t)b * r + row] = fmaxf(s, 0.f);
    }
}

// P2: each warp owns RPW consecutive rows (one row is r elements, 1-2 KB);
// lanes stride over the row's vectors; h for TB tokens sits in shared memory.
template <typename T, int RPW, int TB>
__global__ void __launch_bounds__(kThreads)
pred_up_kernel(const T *__restrict__ W, int ld, int r, int f, const float *__restrict__ h, int B,
               float *__restrict__ s) {
    constexpr int V = Vec<T>::N;
    extern __shared__ float hs[];  // [TB][rp]
    const int rp = (r + 7) & ~7;
    const int b0 = blockIdx.y * TB;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row0 = (blockIdx.x * (kThreads / 32) + warp) * RPW;
    const int nvec = (r + V - 1) / V;

    // prefetch the first vectors of this warp's rows before waiting on h
    uint4 pre[RPW];
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
        const int row = min(row0 + q, f - 1);
        pre[q] = lane < nvec ? ld_stream(W + (size_t)row * ld + lane * V) : make_uint4(0, 0, 0, 0);
    }

    pdl_wait();  // h comes from P1
    for (int i = threadIdx.x; i < TB * rp; i += kThreads) {
        const int t = i / rp, c = i % rp;
        const int b = b0 + t;
        hs[i] = (c < r && b < B) ? h[(size_t)b * r + c] : 0.f;
    }
    __syncthreads();

    float acc[RPW][TB];
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
        for (int t = 0; t < TB; ++t) acc[q][t] = 0.f;

    for (int v = lane; v < nvec; v += 32) {
        const int c0 = v * V;
        const int ne = min(V, r - c0);
        uint4 raw[RPW];
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
            const int row = min(row0 + q, f - 1);
            raw[q] = (v == lane) ? pre[q] : ld_stream(W + (size_t)row * ld + c0);
        }
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
            float w[V];
            unpack<T>(raw[q], w);
#pragma unroll
            for (int e = 0; e < V; ++e) {
                if (e >= ne) w[e] = 0.f;
#pragma unroll
                for (int t = 0; t < TB; ++t) acc[q][t] = fmaf(w[e], hs[t * rp + c0 + e], acc[q][t]);
            }
        }
    }
#pragma unroll
    for (int q = 0; q < RPW; ++q)
#pragma unroll
        for (int t = 0; t < TB; ++t) {
            const float v = warp_sum(acc[q][t]);
            const int row = row0 + q, b = b0 + t;
            if (lane == 0 && row < f && b < B) s[(size_t)b * f + row] = v;
        }
}

template <typename T>
cudaError_t run_predict(const PredictArgs &a, cudaStream_t s) {
    constexpr int RPC = 4, TB1 = 4, RPW = 4, TB2 = 4;
    const bool pdl = pdl_enabled();
    const int ldd = a.ld_down ? a.ld_down : a.d;
    const int ldu = a.ld_up ? a.ld_up : a.r;
    dim3 g1((a.r + RPC - 1) / RPC, (a.B + TB1 - 1) / TB1);
    cudaError_t e = launch(pred_down_kernel<T, RPC, TB1>, g1, dim3(kThreads), 0, s, pdl,
                           static_cast<const T *>(a.p_down), ldd, a.d, a.r, a.x, a.B, a.h);
    if (e != cudaSuccess) return e;
    const int rows_per_cta = (kThreads / 32) * RPW;
    dim3 g2((a.f + rows_per_cta - 1) / rows_per_cta, (a.B + TB2 - 1) / TB2);
    const size_t smem = sizeof(float) * TB2 * ((a.r + 7) & ~7);
    if (smem > 48 * 1024) {
        e = cudaFuncSetAttribute(pred_up_kernel<T, RPW, TB2>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch(pred_up_kernel<T, RPW, TB2>, g2, dim3(kThreads), smem, s, pdl,
                  static_cast<const T *>(a.p_up), ldu, a.r, a.f, static_cast<const float *>(a.h),
                  a.B, a.scores);
}

}  // namespace

cudaError_t launch_predict(const PredictArgs &a, cudaStream_t s) {
    switch (a.dtype) {
    case CS_F32: return run_predict<float>(a, s);
    case CS_F16: return run_predict<__half>(a, s);
    default: return run_predict<__nv_bfloat16>(a, s);
    }
}

}  // namespace cs
