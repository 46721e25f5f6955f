// Gathered sparse FFN (gate GEMV + activation + down AXPY) and the dense
// pre-activation GEMV of exact-mask mode.
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (sparse_mlp_forward: only
// the chosen neurons' gate rows and down columns are read) and section
// "Kernel-Level Implementation" (one warp-uncoalesced thread per neuron in the
// page's sketch; here every row is moved whole and contiguous); section "The
// SiLU/GELU Challenge: TurboSparse" for the gated form relu(gate x) * up x.
//
// Design.  W_down is stored transposed, so each chosen neuron needs two (or
// three, gated) contiguous rows of d elements.  A persistent grid of one CTA
// per SM splits the ascending index list into contiguous chunks.  Thread 0 of
// each CTA streams the chunk's rows into a ring of shared-memory stages with
// bulk async copies (TMA engine, completion counted on an mbarrier per
// stage), so up to ~200 KB per SM is in flight with one issuing thread.  The
// 512 threads own fixed 16-byte column vectors: they dot the staged gate (and
// up) rows with x held in registers, combine the per-warp sums through shared
// memory in a fixed order, apply ReLU (and the up factor), and accumulate
// a_j * w_down_j into per-thread fp32 registers.  Each CTA writes its partial
// y; a second kernel adds the G partials per column in a fixed order (and
// applies the residual epilogue), so y is bit-reproducible run to run.
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kFfnThreads = 512;
constexpr int kFfnWarps = kFfnThreads / 32;
constexpr int kMaxStages = 16;
constexpr int kNg = 4;                    // neurons per reduction group (max)
constexpr size_t kRingBudget = 220 * 1024;

struct FfnK {
    const uint8_t *w_gate, *w_up, *w_down_t;
    const float *bias, *x, *preact;
    const int32_t *idx, *count;
    float *part;
    uint32_t *err;
    int d, f, B, dp;
    int ldb;        // row pitch in bytes
    int rb;         // bytes copied per row (d * elem rounded up to 16)
    int nst;        // ring stages
    int ng;         // neurons per group (<= kNg, <= nst / 2 when possible)
    size_t ring_off;
};

template <typename T, int TB, bool GLU, bool PRE, int MAXV>
__global__ void __launch_bounds__(kFfnThreads, 1) ffn_gather_kernel(const FfnK a) {
    constexpr int V = Vec<T>::N;
    constexpr int NROW = (PRE ? 0 : 1) + (GLU ? 1 : 0) + 1;
    constexpr bool DOTS = !PRE || GLU;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t *full = reinterpret_cast<uint64_t *>(smem);
    float *red = reinterpret_cast<float *>(smem + 128);  // [warps][kNg][TB][2]
    int *s_abort = reinterpret_cast<int *>(smem + 128 + sizeof(float) * kFfnWarps * kNg * TB * 2);
    uint8_t *ring = smem + a.ring_off;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int b0 = blockIdx.y * TB;
    const int nvec = (a.d + V - 1) / V;
    const int stage_bytes = NROW * a.rb;

    if (tid == 0) {
        for (int s = 0; s < a.nst; ++s) mbar_init(&full[s], 1);
        *s_abort = 0;
        mbar_fence_init();
    }
    __syncthreads();

    pdl_wait();  // idx, count and x come from earlier kernels

    int n = *a.count;
    if (n < 0 || n > a.f) {
        if (tid == 0 && c == 0 && blockIdx.y == 0) atomicOr(a.err, CS_DEVERR_COUNT);
        n = n < 0 ? 0 : a.f;
    }
    const int n0 = (int)((long long)n * c / G);
    const int cnt = (int)((long long)n * (c + 1) / G) - n0;
    const int32_t *my_idx = a.idx + n0;
    const uint64_t pol = policy_evict_first();

    auto issue = [&](int m) {
        const int s = m % a.nst;
        int j = __ldg(my_idx + m);
        if (j < 0 || j >= a.f) j = 0;  // consumers see the bad id and use a = 0
        uint8_t *st = ring + (size_t)s * stage_bytes;
        mbar_arrive_expect_tx(&full[s], (uint32_t)stage_bytes);
        int r = 0;
        if (!PRE) bulk_g2s_hint(st + (r++) * a.rb, a.w_gate + (size_t)j * a.ldb, a.rb, &full[s], pol);
        if (GLU) bulk_g2s_hint(st + (r++) * a.rb, a.w_up + (size_t)j * a.ldb, a.rb, &full[s], pol);
        bulk_g2s_hint(st + r * a.rb, a.w_down_t + (size_t)j * a.ldb, a.rb, &full[s], pol);
    };

    int issued = 0;
    if (tid == 0) {
        const int first = min(a.nst, cnt);
        for (int m = 0; m < first; ++m) issue(m);
        issued = first;
    }

    // x in registers: thread owns vectors v = tid + i * kFfnThreads
    float xr[TB][MAXV][V];
    float yacc[TB][MAXV][V];
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        const int b = min(b0 + t, a.B - 1);
        const bool live = b0 + t < a.B;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            const int v = tid + i * kFfnThreads;
#pragma unroll
            for (int e = 0; e < V; ++e) {
                const int col = v * V + e;
                xr[t][i][e] = (live && DOTS && v < nvec && col < a.d) ? __ldg(a.x + (size_t)b * a.d + col) : 0.f;
                yacc[t][i][e] = 0.f;
            }
        }
    }

    for (int g0 = 0; g0 < cnt; g0 += a.ng) {
        const int gn = min(a.ng, cnt - g0);
        float pg[kNg][TB], pu[kNg][TB];
#pragma unroll
        for (int q = 0; q < kNg; ++q) {
#pragma unroll
            for (int t = 0; t < TB; ++t) pg[q][t] = pu[q][t] = 0.f;
            if (q < gn) {
                const int m = g0 + q;
                const int s = m % a.nst;
                if (!mbar_wait(&full[s], (uint32_t)((m / a.nst) & 1))) {
                    atomicOr(a.err, CS_DEVERR_TIMEOUT);
                    *s_abort = 1;
                }
                if (DOTS) {
                    const uint8_t *st = ring + (size_t)s * stage_bytes;
#pragma unroll
                    for (int i = 0; i < MAXV; ++i) {
                        const int v = tid + i * kFfnThreads;
                        if (v < nvec) {
                            const int ne = min(V, a.d - v * V);
                            if (!PRE) {
                                float w[V];
                                unpack<T>(*reinterpret_cast<const uint4 *>(st + v * 16), w);
#pragma unroll
                                for (int e = 0; e < V; ++e) {
                                    const float we = e < ne ? w[e] : 0.f;
#pragma unroll
                                    for (int t = 0; t < TB; ++t) pg[q][t] = fmaf(we, xr[t][i][e], pg[q][t]);
                                }
                            }
                            if (GLU) {
                                float w[V];
                                unpack<T>(*reinterpret_cast<const uint4 *>(st + (PRE ? 0 : a.rb) + v * 16), w);
#pragma unroll
                                for (int e = 0; e < V; ++e) {
                                    const float we = e < ne ? w[e] : 0.f;
#pragma unroll
                                    for (int t = 0; t < TB; ++t) pu[q][t] = fmaf(we, xr[t][i][e], pu[q][t]);
                                }
                            }
                        }
                    }
                }
            }
        }
        if (DOTS) {
#pragma unroll
            for (int q = 0; q < kNg; ++q)
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    if (q < gn) {
                        const float sg = warp_sum(pg[q][t]);
                        const float su = GLU ? warp_sum(pu[q][t]) : 0.f;
                        if (lane == 0) {
                            red[((warp * kNg + q) * TB + t) * 2 + 0] = sg;
                            red[((warp * kNg + q) * TB + t) * 2 + 1] = su;
                        }
                    }
                }
            __syncthreads();
        }
        // activations (every thread forms them itself, same fixed order)
        float act[kNg][TB];
#pragma unroll
        for (int q = 0; q < kNg; ++q) {
#pragma unroll
            for (int t = 0; t < TB; ++t) act[q][t] = 0.f;
            if (q < gn) {
                const int j = __ldg(my_idx + g0 + q);
                const bool valid = j >= 0 && j < a.f;
                if (!valid && tid == 0) atomicOr(a.err, CS_DEVERR_INDEX);
                const int js = valid ? j : 0;
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    float g = 0.f, u = 0.f;
                    if (!PRE || GLU) {
                        for (int w = 0; w < kFfnWarps; ++w) {
                            g += red[((w * kNg + q) * TB + t) * 2 + 0];
                            u += red[((w * kNg + q) * TB + t) * 2 + 1];
                        }
                    }
                    if (PRE) g = __ldg(a.preact + js);
                    else if (a.bias) g += __ldg(a.bias + js);
                    float av = fmaxf(g, 0.f);
                    if (GLU) av *= u;
                    act[q][t] = valid ? av : 0.f;
                }
            }
        }
        // y += a_j * w_down_j
#pragma unroll
        for (int q = 0; q < kNg; ++q) {
            if (q < gn) {
                const int s = (g0 + q) % a.nst;
                const uint8_t *dn = ring + (size_t)s * stage_bytes + (NROW - 1) * a.rb;
#pragma unroll
                for (int i = 0; i < MAXV; ++i) {
                    const int v = tid + i * kFfnThreads;
                    if (v < nvec) {
                        float w[V];
                        unpack<T>(*reinterpret_cast<const uint4 *>(dn + v * 16), w);
#pragma unroll
                        for (int t = 0; t < TB; ++t)
#pragma unroll
                            for (int e = 0; e < V; ++e) yacc[t][i][e] = fmaf(act[q][t], w[e], yacc[t][i][e]);
                    }
                }
            }
        }
        __syncthreads();  // stages of this group and red[] are free again
        if (*s_abort) {
            if (tid == 0)
                for (int m = g0 + gn; m < issued; ++m)
                    mbar_wait(&full[m % a.nst], (uint32_t)((m / a.nst) & 1), 100000000ull);
            return;
        }
        if (tid == 0) {
            for (int q = 0; q < gn; ++q) {
                const int m = g0 + q + a.nst;
                if (m < cnt) { issue(m); issued = m + 1; }
            }
        }
    }

    pdl_launch_dependents();

    // partial y of this CTA
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        const int b = b0 + t;
        if (b >= a.B) break;
        float *dst = a.part + ((size_t)c * a.B + b) * a.dp;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            const int v = tid + i * kFfnThreads;
            if (v < nvec) {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    float4 o = make_float4(yacc[t][i][e], yacc[t][i][e + 1], yacc[t][i][e + 2], yacc[t][i][e + 3]);
                    *reinterpret_cast<float4 *>(dst + v * V + e) = o;
                }
            }
        }
    }
}

// y[b, col] = (resid[b, col] + scale *) sum_{c < G} part[c, b, col], c ascending
// within each of 8 warps, warps combined in order.
__global__ void __launch_bounds__(256)
ffn_reduce_kernel(const float *__restrict__ part, int G, int B, int d, int dp,
                  const float *__restrict__ resid, float scale, float *__restrict__ y) {
    __shared__ float red[8][33];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int col = blockIdx.x * 32 + lane;
    const int b = blockIdx.y;
    pdl_wait();
    float acc = 0.f;
    if (col < d) {
        const float *p = part + (size_t)b * dp + col;
        const size_t stride = (size_t)B * dp;
#pragma unroll 4
        for (int cc = warp; cc < G; cc += 8) acc += __ldg(p + cc * stride);
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && col < d) {
        float s = 0.f;
#pragma unroll
        for (int w = 0; w < 8; ++w) s += red[w][lane];
        const size_t o = (size_t)b * d + col;
        y[o] = resid ? fmaf(scale, s, resid[o]) : s;
    }
}

// Exact-mask mode: pre[j] = w_gate_j . x + bias_j for every neuron.
template <typename T, int RPW>
__global__ void __launch_bounds__(256)
preact_kernel(const T *__restrict__ W, int ld, int d, int f, const float *__restrict__ x,
              const float *__restrict__ bias, float *__restrict__ pre) {
    constexpr int V = Vec<T>::N;
    extern __shared__ float xs[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int row0 = (blockIdx.x * 8 + warp) * RPW;
    const int nvec = (d + V - 1) / V;
    pdl_wait();
    for (int i = threadIdx.x; i < nvec * V; i += 256) xs[i] = i < d ? x[i] : 0.f;
    __syncthreads();
    float acc[RPW];
#pragma unroll
    for (int q = 0; q < RPW; ++q) acc[q] = 0.f;
    for (int v = lane; v < nvec; v += 32) {
        const int ne = min(V, d - v * V);
        uint4 raw[RPW];
#pragma unroll
        for (int q = 0; q < RPW; ++q) raw[q] = ld_stream(W + (size_t)min(row0 + q, f - 1) * ld + v * V);
#pragma unroll
        for (int q = 0; q < RPW; ++q) {
            float w[V];
            unpack<T>(raw[q], w);
#pragma unroll
            for (int e = 0; e < V; ++e) acc[q] = fmaf(e < ne ? w[e] : 0.f, xs[v * V + e], acc[q]);
        }
    }
#pragma unroll
    for (int q = 0; q < RPW; ++q) {
        const float s = warp_sum(acc[q]);
        const int row = row0 + q;
        if (lane == 0 && row < f) pre[row] = s + (bias ? bias[row] : 0.f);
    }
}


template <typename T, int TB, bool GLU, bool PRE, int MAXV>
cudaError_t run_gather(const FfnArgs &a, FfnK k, size_t smem, cudaStream_t s) {
    auto fn = ffn_gather_kernel<T, TB, GLU, PRE, MAXV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    dim3 grid(a.G, (a.B + TB - 1) / TB);
    return launch(fn, grid, dim3(kFfnThreads), smem, s, pdl_enabled(), k);
}

template <typename T, int TB, bool GLU, bool PRE>
cudaError_t pick_maxv(const FfnArgs &a, const FfnK &k, size_t smem, cudaStream_t s) {
    constexpr int V = Vec<T>::N;
    const int nvec = (a.d + V - 1) / V;
    if (nvec <= kFfnThreads) return run_gather<T, TB, GLU, PRE, 1>(a, k, smem, s);
    if (nvec <= 2 * kFfnThreads) return run_gather<T, TB, GLU, PRE, 2>(a, k, smem, s);
    return run_gather<T, TB, GLU, PRE, 4>(a, k, smem, s);
}

template <typename T, int TB>
cudaError_t pick_mode(const FfnArgs &a, const FfnK &k, size_t smem, cudaStream_t s) {
    const bool glu = a.w_up != nullptr, pre = a.preact != nullptr;
    if (glu) return pre ? pick_maxv<T, TB, true, true>(a, k, smem, s) : pick_maxv<T, TB, true, false>(a, k, smem, s);
    return pre ? pick_maxv<T, TB, false, true>(a, k, smem, s) : pick_maxv<T, TB, false, false>(a, k, smem, s);
}

template <typename T>
cudaError_t run_ffn(const FfnArgs &a, cudaStream_t s) {
    const int esz = (int)sizeof(T);
    FfnK k;
    k.w_gate = static_cast<const uint8_t *>(a.w_gate);
    k.w_up = static_cast<const uint8_t *>(a.w_up);
    k.w_down_t = static_cast<const uint8_t *>(a.w_down_t);
    k.bias = a.bias;
    k.x = a.x;
    k.preact = a.preact;
    k.idx = a.idx;
    k.count = a.count;
    k.part = a.part;
    k.err = a.err;
    k.d = a.d;
    k.f = a.f;
    k.B = a.B;
    k.dp = a.dp;
    k.ldb = a.ld * esz;
    k.rb = (a.d * esz + 15) & ~15;
    const int nrow = (a.preact ? 0 : 1) + (a.w_up ? 1 : 0) + 1;
    const int tb = a.B >= 2 ? 2 : 1;
    const size_t head = 128 + sizeof(float) * kFfnWarps * kNg * tb * 2 + 16;
    k.ring_off = (head + 127) & ~size_t(127);
    int nst = (int)(kRingBudget / ((size_t)nrow * k.rb));
    nst = nst > kMaxStages ? kMaxStages : nst;
    if (nst < 1) return cudaErrorInvalidValue;
    k.nst = nst;
    k.ng = nst >= 2 * kNg ? kNg : (nst / 2 > 0 ? nst / 2 : 1);
    const size_t smem = k.ring_off + (size_t)nst * nrow * k.rb;
    cudaError_t e = tb == 2 ? pick_mode<T, 2>(a, k, smem, s) : pick_mode<T, 1>(a, k, smem, s);
    if (e != cudaSuccess) return e;
    dim3 g((a.d + 31) / 32, a.B);
    return launch(ffn_reduce_kernel, g, dim3(256), 0, s, pdl_enabled(),
                  static_cast<const float *>(a.part), a.G, a.B, a.d, a.dp, a.resid, a.scale, a.y);
}

template <typename T>
cudaError_t run_preact(const PreactArgs &a, cudaStream_t s) {
    constexpr int RPW = 4;
    constexpr int V = Vec<T>::N;
    const int rows_per_cta = 8 * RPW;
    const size_t smem = sizeof(float) * (size_t)((a.d + V - 1) / V) * V;
    auto fn = preact_kernel<T, RPW>;
    if (smem > 48 * 1024) {
        cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
    }
    return launch(fn, dim3((a.f + rows_per_cta - 1) / rows_per_cta), dim3(256), smem, s, pdl_enabled(),
                  static_cast<const T *>(a.w_gate), a.ld, a.d, a.f, a.x, a.bias, a.pre);
}

}  // namespace

// Largest d (in elements) the gather kernel takes for a dtype.
int ffn_max_d(cs_dtype t) {
    const int V = t == CS_F32 ? 4 : 8;
    return 4 * kFfnThreads * V;
}

cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s) {
    switch (a.dtype) {
    case CS_F32: return run_ffn<float>(a, s);
    case CS_F16: return run_ffn<__half>(a, s);
    default: return run_ffn<__nv_bfloat16>(a, s);
    }
}

cudaError_t launch_preact(const PreactArgs &a, cudaStream_t s) {
    switch (a.dtype) {
    case CS_F32: return run_preact<float>(a, s);
    case CS_F16: return run_preact<__half>(a, s);
    default: return run_preact<__nv_bfloat16>(a, s);
    }
}

}  // namespace cs
