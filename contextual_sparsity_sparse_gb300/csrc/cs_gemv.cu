// Streaming GEMVs over contiguous weight rows: the predictor's two maps and
// the exact-mask pre-activations.
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (SparsityPredictor: a
// bias-free down map to a small bottleneck, ReLU, a bias-free up map to one
// score per neuron; the closing sigmoid is monotone and not applied, so scores
// are logits); "Contextual Sparsity and Activation Predictors", first section
// (the exact mask needs every gate row: g_j = w_gate_j . x + b_j).
//
//   out[b, row] = epi( sum_c W[row, c] * v[b, c] ),  epi = id | relu | +bias
//
// Each CTA owns a contiguous block of rows, i.e. one contiguous byte range of
// W.  Thread 0 streams it into shared memory in chunks of ~40 KB with bulk
// async copies (one copy per chunk, so the copy engine's fixed per-copy cost
// is amortised), double-buffered, and issues the first two chunks before
// waiting on the previous kernel: the weights do not depend on it, only v
// does.  Warps then reduce whole rows from shared memory with shuffles.
#include <algorithm>
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kThreads = 256;
constexpr int kWarps = kThreads / 32;

enum { EPI_NONE = 0, EPI_RELU = 1, EPI_BIAS = 2 };

struct GemvK {
    const uint8_t *W;
    int ldb;            // row pitch in bytes (multiple of 16)
    int ncols;          // used columns
    int nrows;
    const float *v;     // [B, ncols]
    int B;
    float *out;         // [B, nrows]
    const float *bias;  // [nrows] (EPI_BIAS)
    int rows_per_cta;
    int chunk_rows;
    uint32_t *err;
};

template <typename T, int TB, int EPI>
__global__ void __launch_bounds__(kThreads) stream_gemv_kernel(const GemvK a) {
    constexpr int V = Vec<T>::N;
    extern __shared__ __align__(16) uint8_t smem[];
    __shared__ __align__(8) uint64_t full[2];
    const int ncp = (a.ncols + 7) & ~7;
    float *vs = reinterpret_cast<float *>(smem);                       // [TB][ncp]
    uint8_t *buf0 = smem + (((size_t)TB * ncp * 4 + 127) & ~size_t(127));
    const size_t chunk_bytes = (size_t)a.chunk_rows * a.ldb;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blockIdx.x * a.rows_per_cta;
    const int r1 = min(a.nrows, r0 + a.rows_per_cta);
    const int nch = r0 < r1 ? (r1 - r0 + a.chunk_rows - 1) / a.chunk_rows : 0;
    const int b0 = blockIdx.y * TB;
    const int nvec = (a.ncols * (int)sizeof(T) + 15) / 16;

    auto issue = [&](int ch) {
        const int rs = r0 + ch * a.chunk_rows;
        const int nr = min(a.chunk_rows, r1 - rs);
        const uint32_t bytes = (uint32_t)nr * (uint32_t)a.ldb;
        uint8_t *dst = buf0 + (size_t)(ch & 1) * chunk_bytes;
        mbar_arrive_expect_tx(&full[ch & 1], bytes);
        bulk_g2s(dst, a.W + (size_t)rs * a.ldb, bytes, &full[ch & 1]);
    };

    if (tid == 0) {
        mbar_init(&full[0], 1);
        mbar_init(&full[1], 1);
        mbar_fence_init();
        for (int ch = 0; ch < min(2, nch); ++ch) issue(ch);
    }

    pdl_launch_dependents();  // one wave: the next kernel may start its prologue
    pdl_wait();               // v comes from the previous kernel
    const bool v4ok = (a.ncols & 3) == 0 && (reinterpret_cast<uintptr_t>(a.v) & 15) == 0;
    for (int t = 0; t < TB; ++t) {
        const int b = b0 + t;
        float *dst = vs + t * ncp;
        if (v4ok && b < a.B) {
            const float4 *src = reinterpret_cast<const float4 *>(a.v + (size_t)b * a.ncols);
#pragma unroll 8
            for (int c = tid; c < ncp / 4; c += kThreads)
                reinterpret_cast<float4 *>(dst)[c] = c * 4 < a.ncols ? ld_dep(src + c) : make_float4(0.f, 0.f, 0.f, 0.f);
        } else {
            for (int c = tid; c < ncp; c += kThreads)
                dst[c] = (b < a.B && c < a.ncols) ? ld_dep(a.v + (size_t)b * a.ncols + c) : 0.f;
        }
    }
    __syncthreads();

    bool ok = true;
    for (int ch = 0; ch < nch; ++ch) {
        if (!mbar_wait(&full[ch & 1], (uint32_t)((ch >> 1) & 1))) {
            if (tid == 0) atomicOr(a.err, CS_DEVERR_TIMEOUT);
            ok = false;
        }
        const uint8_t *buf = buf0 + (size_t)(ch & 1) * chunk_bytes;
        const int rs = r0 + ch * a.chunk_rows;
        const int nr = min(a.chunk_rows, r1 - rs);
        for (int q = warp; q < nr; q += kWarps) {
            const uint4 *row = reinterpret_cast<const uint4 *>(buf + (size_t)q * a.ldb);
            float acc[TB];
#pragma unroll
            for (int t = 0; t < TB; ++t) acc[t] = 0.f;
            for (int v = lane; v < nvec; v += 32) {
                float w[V];
                unpack<T>(row[v], w);
                const int ne = a.ncols - v * V;
                if (ne < V) {
#pragma unroll
                    for (int e = 0; e < V; ++e) w[e] = e < ne ? w[e] : 0.f;
                }
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    const float *vv = vs + t * ncp + v * V;
#pragma unroll
                    for (int e = 0; e < V; e += 4) {
                        const float4 x4 = *reinterpret_cast<const float4 *>(vv + e);
                        acc[t] = fmaf(w[e], x4.x, acc[t]);
                        acc[t] = fmaf(w[e + 1], x4.y, acc[t]);
                        acc[t] = fmaf(w[e + 2], x4.z, acc[t]);
                        acc[t] = fmaf(w[e + 3], x4.w, acc[t]);
                    }
                }
            }
#pragma unroll
            for (int t = 0; t < TB; ++t) {
                float sum = warp_sum(acc[t]);
                const int b = b0 + t;
                if (lane == 0 && b < a.B) {
                    if (EPI == EPI_RELU) sum = fmaxf(sum, 0.f);
                    if (EPI == EPI_BIAS && a.bias) sum += a.bias[rs + q];
                    a.out[(size_t)b * a.nrows + rs + q] = sum;
                }
            }
        }
        __syncthreads();  // the buffer of chunk ch is free
        if (tid == 0 && ok && ch + 2 < nch) issue(ch + 2);
    }
    if (!ok && tid == 0) {
        // let copies already in flight land before the CTA's memory goes away
        for (int ch = 0; ch < nch; ++ch) mbar_wait(&full[ch & 1], (uint32_t)((ch >> 1) & 1), 100000000ull);
    }
}

// One token (B = 1): weights streamed straight into registers with coalesced
// 16-byte loads, v held in registers, no shared-memory staging.  A round is RU
// rows; the first round's weights are loaded before waiting on the previous
// kernel (they do not depend on it), and each round's loads are issued before
// the previous round's reductions, so loads stay in flight across them.
//   SPLIT = false (rows of at most 256 vectors): a warp per row, lane l takes
//     vectors l + 32 i (i < NV); warp w's round takes RU consecutive rows.
//   SPLIT = true (longer rows): every row is spread over the CTA, thread t
//     takes vectors t + 256 i (i < NV); per round each warp sums its share of
//     the RU rows, one barrier publishes the warp sums, and thread u adds row
//     u's eight warp sums in warp order.
// Each vector of a thread has its own accumulator, added in order at the end
// of the row, so results are bit-reproducible.
template <typename T, int EPI, bool SPLIT, int NV, int RU>
__global__ void __launch_bounds__(kThreads) gemv_reg_kernel(const GemvK a) {
    constexpr int V = Vec<T>::N;
    __shared__ float red[2][SPLIT ? RU : 1][kWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int r0 = blockIdx.x * a.rows_per_cta;
    const int r1 = min(a.nrows, r0 + a.rows_per_cta);
    const int nvec = (a.ncols * (int)sizeof(T) + 15) / 16;
    const int per_round = SPLIT ? RU : kWarps * RU;
    const int nround = r0 < r1 ? (r1 - r0 + per_round - 1) / per_round : 0;

    int vv[NV];
#pragma unroll
    for (int i = 0; i < NV; ++i) vv[i] = SPLIT ? tid + i * kThreads : lane + 32 * i;
    auto row_of = [&](int k, int u) { return SPLIT ? r0 + k * RU + u : r0 + (k * kWarps + warp) * RU + u; };

    uint4 w[RU][NV];
    auto load = [&](int k) {
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            const int row = min(row_of(k, u), r1 - 1);   // rows past the block repeat its last
            const uint4 *rp = reinterpret_cast<const uint4 *>(a.W + (size_t)row * a.ldb);
#pragma unroll
            for (int i = 0; i < NV; ++i) w[u][i] = vv[i] < nvec ? __ldg(rp + vv[i]) : make_uint4(0u, 0u, 0u, 0u);
        }
    };
    if (nround > 0) load(0);

    pdl_launch_dependents();  // one wave: the next kernel may start its prologue
    pdl_wait();               // v comes from the previous kernel

    // this thread's slice of v (zero past ncols); weights past ncols in a
    // row's last vector are zeroed in the dot product (row padding may hold
    // anything)
    float xr[NV][V];
    int ne[NV];
    const bool x4 = (reinterpret_cast<uintptr_t>(a.v) & 15) == 0;
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int c0 = vv[i] * V;
        ne[i] = a.ncols - c0;
        if (vv[i] < nvec && x4 && c0 + V <= a.ncols) {
#pragma unroll
            for (int e = 0; e < V; e += 4) {
                const float4 t = ld_dep(reinterpret_cast<const float4 *>(a.v + c0 + e));
                xr[i][e] = t.x; xr[i][e + 1] = t.y; xr[i][e + 2] = t.z; xr[i][e + 3] = t.w;
            }
        } else {
#pragma unroll
            for (int e = 0; e < V; ++e) xr[i][e] = (vv[i] < nvec && c0 + e < a.ncols) ? ld_dep(a.v + c0 + e) : 0.f;
        }
    }

    for (int k = 0; k < nround; ++k) {
        float part[RU];
#pragma unroll
        for (int u = 0; u < RU; ++u) {
            float acc[NV];
#pragma unroll
            for (int i = 0; i < NV; ++i) {
                float f[V];
                unpack<T>(w[u][i], f);
                if (ne[i] < V) {
#pragma unroll
                    for (int e = 0; e < V; ++e) f[e] = e < ne[i] ? f[e] : 0.f;
                }
                acc[i] = 0.f;
#pragma unroll
                for (int e = 0; e < V; ++e) acc[i] = fmaf(f[e], xr[i][e], acc[i]);
            }
            part[u] = acc[0];
#pragma unroll
            for (int i = 1; i < NV; ++i) part[u] += acc[i];
        }
        if (k + 1 < nround) load(k + 1);   // in flight during the reductions
#pragma unroll
        for (int u = 0; u < RU; ++u) part[u] = warp_sum(part[u]);
        if (SPLIT) {
            if (lane == 0) {
#pragma unroll
                for (int u = 0; u < RU; ++u) red[k & 1][u][warp] = part[u];
            }
            __syncthreads();
            const int row = row_of(k, tid);
            if (tid < RU && row < r1) {
                float sum = 0.f;
#pragma unroll
                for (int q = 0; q < kWarps; ++q) sum += red[k & 1][tid][q];
                if (EPI == EPI_RELU) sum = fmaxf(sum, 0.f);
                if (EPI == EPI_BIAS && a.bias) sum += a.bias[row];
                a.out[row] = sum;
            }
        } else if (lane == 0) {
#pragma unroll
            for (int u = 0; u < RU; ++u) {
                const int row = row_of(k, u);
                if (row < r1) {
                    float sum = part[u];
                    if (EPI == EPI_RELU) sum = fmaxf(sum, 0.f);
                    if (EPI == EPI_BIAS && a.bias) sum += a.bias[row];
                    a.out[row] = sum;
                }
            }
        }
    }
}

template <typename T, int EPI, bool SPLIT, int NV, int RU>
cudaError_t run_reg(const GemvK &k0, cudaStream_t s) {
    GemvK k = k0;
    int sms = device_sm_count();
    sms = sms < 1 ? 1 : sms;
    k.rows_per_cta = std::max(1, (k.nrows + 2 * sms - 1) / (2 * sms));   // two CTAs per SM
    dim3 grid((k.nrows + k.rows_per_cta - 1) / k.rows_per_cta);
    return launch(gemv_reg_kernel<T, EPI, SPLIT, NV, RU>, grid, dim3(kThreads), 0, s, pdl_enabled(), k);
}

template <typename T, int TB, int EPI>
cudaError_t run_tb(const GemvK &k0, cudaStream_t s, size_t per_cta) {
    GemvK k = k0;
    int sms = device_sm_count();
    sms = sms < 1 ? 1 : sms;
    const size_t vbytes = ((size_t)TB * ((k.ncols + 7) & ~7) * 4 + 127) & ~size_t(127);
    // two CTAs per SM: each gets per_cta (half of ~220 KB by default) for its
    // vector and two buffers
    size_t chunk_budget = per_cta > vbytes ? (per_cta - vbytes) / 2 : 0;
    chunk_budget = std::min<size_t>(chunk_budget, 48 * 1024);
    k.rows_per_cta = std::max(1, (k.nrows + 2 * sms - 1) / (2 * sms));
    k.chunk_rows = (int)std::max<size_t>(1, chunk_budget / (size_t)k.ldb);
    k.chunk_rows = std::min(k.chunk_rows, k.rows_per_cta);
    const size_t smem = vbytes + 2 * (size_t)k.chunk_rows * k.ldb;
    auto fn = stream_gemv_kernel<T, TB, EPI>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid((k.nrows + k.rows_per_cta - 1) / k.rows_per_cta, (k.B + TB - 1) / TB);
    return launch(fn, grid, dim3(kThreads), smem, s, pdl_enabled(), k);
}

constexpr size_t kGemvCta = 110 * 1024;       // two CTAs per SM

template <typename T, int EPI>
cudaError_t run_gemv(const GemvK &k, cudaStream_t s, size_t per_cta) {
    // one token: the register-streaming kernel
    const int nvec = (k.ncols * (int)sizeof(T) + 15) / 16;
    if (k.B == 1) {
        if (nvec <= 32) return run_reg<T, EPI, false, 1, 4>(k, s);
        if (nvec <= 64) return run_reg<T, EPI, false, 2, 4>(k, s);
        if (nvec <= 128) return run_reg<T, EPI, false, 4, 4>(k, s);
        if (nvec <= 256) return run_reg<T, EPI, false, 8, 2>(k, s);
        if (nvec <= 512) return run_reg<T, EPI, true, 2, 4>(k, s);
        if (nvec <= 1024) return run_reg<T, EPI, true, 4, 4>(k, s);
        if (nvec <= 2048) return run_reg<T, EPI, true, 8, 2>(k, s);
    }
    // tokens per CTA: as many as fit beside the weight buffers (weights are
    // re-streamed for each group of TB tokens)
    const size_t row_f = (size_t)((k.ncols + 7) & ~7) * 4;
    if (k.B >= 4 && 4 * row_f <= 48 * 1024) return run_tb<T, 4, EPI>(k, s, per_cta);
    if (k.B >= 2 && 2 * row_f <= 48 * 1024) return run_tb<T, 2, EPI>(k, s, per_cta);
    return run_tb<T, 1, EPI>(k, s, per_cta);
}


template <int EPI>
cudaError_t dispatch(cs_dtype dt, const GemvK &k, cudaStream_t s, size_t per_cta = kGemvCta) {
    switch (dt) {
    case CS_F32: return run_gemv<float, EPI>(k, s, per_cta);
    case CS_F16: return run_gemv<__half, EPI>(k, s, per_cta);
    default: return run_gemv<__nv_bfloat16, EPI>(k, s, per_cta);
    }
}

}  // namespace

cudaError_t launch_predict(const PredictArgs &a, cudaStream_t s) {
    const size_t es = dtype_size(a.dtype);
    GemvK k = {};
    // P1: h[b, i] = relu(sum_t P_down[i, t] x[b, t])
    k.W = static_cast<const uint8_t *>(a.p_down);
    k.ldb = (a.ld_down ? a.ld_down : a.d) * (int)es;
    k.ncols = a.d;
    k.nrows = a.r;
    k.v = a.x;
    k.B = a.B;
    k.out = a.h;
    k.err = a.err;
    cudaError_t e = dispatch<EPI_RELU>(a.dtype, k, s);
    if (e != cudaSuccess) return e;
    // P2: s[b, j] = sum_i P_up[j, i] h[b, i]
    k.W = static_cast<const uint8_t *>(a.p_up);
    k.ldb = (a.ld_up ? a.ld_up : a.r) * (int)es;
    k.ncols = a.r;
    k.nrows = a.f;
    k.v = a.h;
    k.out = a.scores;
    return dispatch<EPI_NONE>(a.dtype, k, s);
}

cudaError_t launch_gemv_batch(cs_dtype dt, const void *W, int ldb_bytes, int ncols, int nrows, const float *v,
                              int B, float *out, const float *bias, int epi, uint32_t *err, cudaStream_t s) {
    GemvK k = {};
    k.W = static_cast<const uint8_t *>(W);
    k.ldb = ldb_bytes;
    k.ncols = ncols;
    k.nrows = nrows;
    k.v = v;
    k.B = B;
    k.out = out;
    k.bias = bias;
    k.err = err;
    if (epi == 1) return dispatch<EPI_RELU>(dt, k, s);
    if (epi == 2) return dispatch<EPI_BIAS>(dt, k, s);
    return dispatch<EPI_NONE>(dt, k, s);
}

cudaError_t launch_preact(const PreactArgs &a, cudaStream_t s) {
    GemvK k = {};
    k.W = static_cast<const uint8_t *>(a.w_gate);
    k.ldb = a.ld * (int)dtype_size(a.dtype);
    k.ncols = a.d;
    k.nrows = a.f;
    k.v = a.x;
    k.B = 1;
    k.out = a.pre;
    k.bias = a.bias;
    k.err = a.err;
    return dispatch<EPI_BIAS>(a.dtype, k, s);
}

}  // namespace cs
