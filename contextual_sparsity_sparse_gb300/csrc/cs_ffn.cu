// Gathered sparse FFN: gate GEMV + activation + down AXPY over the listed
// neurons, and the fixed-order reduction of the per-CTA partial sums.
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (sparse_mlp_forward: only
// the chosen neurons' gate rows and down columns are read) and section
// "Kernel-Level Implementation" (the page's sketch gives each neuron to one
// thread, so a warp's loads hit 32 different rows; here every row is read
// whole and coalesced); section "The SiLU/GELU Challenge: TurboSparse" for the
// gated form relu(gate x) * up x.
//
// Design.  W_down is stored transposed, so each chosen neuron needs two (or
// three, gated) contiguous rows of d elements.  A persistent grid of one CTA
// per SM splits the ascending index list into contiguous chunks.  A CTA has
// one thread per 16-byte column vector of a row (up to 1024 threads; wider
// rows give each thread MAXV vectors), and each thread gathers exactly its
// vectors of the chunk's rows with per-thread asynchronous copies (cp.async)
// into its own slots of a shared-memory ring, SG groups of NG neurons ahead.
// A thread only ever reads the slots it filled, so the ring needs no barrier.
// Per group: each thread's partial gate (and up) dot products are summed per
// warp, one block barrier publishes the warp sums, and every warp then adds
// them in a fixed shuffle order to get the activations itself, applies its
// a_j * w_down_j AXPY at once, and refills its slots.  x and the output
// accumulators live in registers (fp32).  Each CTA writes its partial y; a
// second kernel adds the G partials per column in a fixed order (and applies
// the residual epilogue), so y is bit-reproducible.
// (One-dimensional bulk copies were measured slower for rows of ~10 KB: the
// copy engine of an SM streams far below its share of HBM bandwidth.)
#include <algorithm>
#include <cstdlib>
#include <utility>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kMaxThreads = 1024;
constexpr int kMaxWarps = kMaxThreads / 32;
constexpr int kNgMax = 4;                 // neurons per group (max)
constexpr int kStageMax = 16;             // ring slots (ng * sg)
constexpr size_t kRingBudget = 200 * 1024;
constexpr int kChunkMax = 2048;           // ids per CTA (f <= kChunkMax * grid)


__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// Sum over the warps of a value that lane w (< nwarps) holds for warp w: a
// fixed xor tree, so every lane gets the same, bit-reproducible sum.
__device__ __forceinline__ float warps_total(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

template <typename T, int TB, bool GLU, bool PRE, int MAXV>
__global__ void __launch_bounds__(kMaxThreads, 1) ffn_gather_kernel(const FfnK a) {
    constexpr int V = Vec<T>::N;
    constexpr int NROW = (PRE ? 0 : 1) + (GLU ? 1 : 0) + 1;
    constexpr bool DOTS = !PRE || GLU;
    extern __shared__ __align__(16) uint4 ring[];  // [slot][NROW][nvec]
    __shared__ float red[2][kNgMax][TB][2][kMaxWarps];
    __shared__ int s_idx[kChunkMax];               // this CTA's ids, staged once
    __shared__ float s_add[kChunkMax];             // their bias (or pre-activation)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nthr = blockDim.x, nwarps = nthr >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int b0 = blockIdx.y * TB;
    const int nvec = a.nvec;
    const uint32_t row_bytes = (uint32_t)nvec * 16u;
    const uint32_t slot_bytes = NROW * row_bytes;
    const uint32_t ring_s = smem_addr(ring);

    // this thread's vectors: byte offsets within a row
    int voff[MAXV];
    bool vok[MAXV];
#pragma unroll
    for (int i = 0; i < MAXV; ++i) {
        const int v = tid + i * nthr;
        vok[i] = v < nvec;
        voff[i] = v * 16;
    }

    pdl_launch_dependents();  // one wave: the next kernel may get resident now
    pdl_wait();  // idx, count and x come from earlier kernels

    int n = ld_dep(a.count);
    if (n < 0 || n > a.f) {
        if (tid == 0 && c == 0 && blockIdx.y == 0) atomicOr(a.err, CS_DEVERR_COUNT);
        n = n < 0 ? 0 : a.f;
    }
    const int n0 = (int)((long long)n * c / G);
    const int cnt = min(kChunkMax, (int)((long long)n * (c + 1) / G) - n0);
    // stage the chunk's ids so issuing copies never waits on a global load
    for (int m = tid; m < cnt; m += nthr) s_idx[m] = ld_dep(a.idx + n0 + m);
    __syncthreads();
    // the chunk's bias (or pre-activation) values, copied once
    {
        const float *addsrc = PRE ? a.preact : a.bias;
        for (int m = tid; m < cnt; m += nthr) {
            int j = s_idx[m];
            j = (j >= 0 && j < a.f) ? j : 0;
            if (PRE) s_add[m] = ld_dep(a.preact + j);  // written by the pre-activation kernel
            else if (addsrc) cp4(smem_addr(&s_add[m]), addsrc + j);
            else s_add[m] = 0.f;
        }
    }
    const int ng = a.ng, sg = a.sg;
    const int ngroups = (cnt + ng - 1) / ng;

    // this thread's copies for group g into slots [s0, s0 + ng)
    auto issue = [&](int g, int s0) {
        if (g < ngroups) {
            const int gn = min(ng, cnt - g * ng);
            for (int q = 0; q < gn; ++q) {
                int j = s_idx[g * ng + q];
                j = (j >= 0 && j < a.f) ? j : 0;
                const size_t roff = (size_t)j * (size_t)a.ldb;
                const uint8_t *gr = a.w_gate + roff;
                const uint8_t *ur = a.w_up + roff;
                const uint8_t *dr = a.w_down_t + roff;
                const uint32_t sb = ring_s + (uint32_t)(s0 + q) * slot_bytes;
#pragma unroll
                for (int i = 0; i < MAXV; ++i) {
                    if (vok[i]) {
                        uint32_t r = sb + (uint32_t)voff[i];
                        if (!PRE) { cp16(r, gr + voff[i]); r += row_bytes; }
                        if (GLU) { cp16(r, ur + voff[i]); r += row_bytes; }
                        cp16(r, dr + voff[i]);
                    }
                }
            }
        }
        cp_async_commit();  // always commit, so group counting stays uniform
    };

    for (int g = 0; g < sg; ++g) issue(g, g * ng);  // group 0 also carries s_add

    float xr[TB][MAXV][V];
    float yacc[TB][MAXV][V];
    const bool xvec = (a.d & 3) == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        const int b = min(b0 + t, a.B - 1);
        const bool live = DOTS && b0 + t < a.B;
        const float *xb = a.x + (size_t)b * a.d;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            const int col0 = (tid + i * nthr) * V;
#pragma unroll
            for (int e = 0; e < V; ++e) yacc[t][i][e] = 0.f;
            if (live && vok[i] && xvec && col0 + V <= a.d) {
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    const float4 v4 = ld_dep(reinterpret_cast<const float4 *>(xb + col0 + e));
                    xr[t][i][e] = v4.x; xr[t][i][e + 1] = v4.y; xr[t][i][e + 2] = v4.z; xr[t][i][e + 3] = v4.w;
                }
            } else {
#pragma unroll
                for (int e = 0; e < V; ++e)
                    xr[t][i][e] = (live && vok[i] && col0 + e < a.d) ? ld_dep(xb + col0 + e) : 0.f;
            }
        }
    }

    int gs = 0;  // ring group of group g
    for (int g = 0; g < ngroups; ++g) {
        const int gn = min(ng, cnt - g * ng);
        const int s0 = gs * ng;
        const int p = g & 1;
        // this thread's copies for group g have landed (commits so far: sg
        // at the start, then one per finished group)
        if (sg == 2) cp_async_wait<1>(); else cp_async_wait<2>();
        // gate (and up) dot products: one accumulator per (neuron, vector).
        // Slots past the group's last neuron hold stale data whose sums are
        // never used.
        if (DOTS) {
            float pg[kNgMax][TB], pu[kNgMax][TB];
#pragma unroll
            for (int q = 0; q < kNgMax; ++q)
#pragma unroll
                for (int t = 0; t < TB; ++t) pg[q][t] = pu[q][t] = 0.f;
#pragma unroll
            for (int i = 0; i < MAXV; ++i) {
                if (!vok[i]) continue;
                const int v = tid + i * nthr;
                const int ne = a.d - v * V;  // < V only on a row's last vector
#pragma unroll
                for (int q = 0; q < kNgMax; ++q) {
                    if (q >= ng) continue;  // ng is uniform: no divergence
                    const uint4 *slot = ring + (size_t)(s0 + q) * NROW * nvec;
                    if (!PRE) {
                        float w[V];
                        unpack<T>(slot[v], w);
                        if (ne < V) {
#pragma unroll
                            for (int e = 0; e < V; ++e) w[e] = e < ne ? w[e] : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < V; ++e)
#pragma unroll
                            for (int t = 0; t < TB; ++t) pg[q][t] = fmaf(w[e], xr[t][i][e], pg[q][t]);
                    }
                    if (GLU) {
                        float w[V];
                        unpack<T>(slot[(PRE ? 0 : 1) * nvec + v], w);
                        if (ne < V) {
#pragma unroll
                            for (int e = 0; e < V; ++e) w[e] = e < ne ? w[e] : 0.f;
                        }
#pragma unroll
                        for (int e = 0; e < V; ++e)
#pragma unroll
                            for (int t = 0; t < TB; ++t) pu[q][t] = fmaf(w[e], xr[t][i][e], pu[q][t]);
                    }
                }
            }
#pragma unroll
            for (int q = 0; q < kNgMax; ++q)
#pragma unroll
                for (int t = 0; t < TB; ++t) {
                    if (q < gn) {
                        if (!PRE) {
                            const float sgv = warp_sum(pg[q][t]);
                            if (lane == 0) red[p][q][t][0][warp] = sgv;
                        }
                        if (GLU) {
                            const float suv = warp_sum(pu[q][t]);
                            if (lane == 0) red[p][q][t][1][warp] = suv;
                        }
                    }
                }
        }
        __syncthreads();  // the warp sums of group g (and, at g = 0, s_add) are visible
        // activations of group g, computed alike by every warp
        float av[kNgMax][TB];
#pragma unroll
        for (int q = 0; q < kNgMax; ++q) {
#pragma unroll
            for (int t = 0; t < TB; ++t) av[q][t] = 0.f;
            if (q >= gn) continue;
            const int m = g * ng + q;
            const int j = s_idx[m];
            const bool valid = j >= 0 && j < a.f;
            const float add = s_add[m];
#pragma unroll
            for (int t = 0; t < TB; ++t) {
                float gsum = 0.f, usum = 0.f;
                if (!PRE) gsum = warps_total(lane < nwarps ? red[p][q][t][0][lane] : 0.f);
                if (GLU) usum = warps_total(lane < nwarps ? red[p][q][t][1][lane] : 0.f);
                const float gv = PRE ? add : gsum + add;
                float act = gate_act(a.act, gv);
                if (GLU) act *= usum;
                av[q][t] = valid ? act : 0.f;
            }
            if (!valid && tid == 0) atomicOr(a.err, CS_DEVERR_INDEX);
        }
        // y += a_j * w_down_j over this thread's vectors
#pragma unroll
        for (int q = 0; q < kNgMax; ++q) {
            if (q < gn) {
                const uint4 *dn = ring + ((size_t)(s0 + q) * NROW + (NROW - 1)) * nvec;
#pragma unroll
                for (int i = 0; i < MAXV; ++i) {
                    if (vok[i]) {
                        float w[V];
                        unpack<T>(dn[tid + i * nthr], w);
#pragma unroll
                        for (int t = 0; t < TB; ++t)
#pragma unroll
                            for (int e = 0; e < V; ++e) yacc[t][i][e] = fmaf(av[q][t], w[e], yacc[t][i][e]);
                    }
                }
            }
        }
        // this thread's slots of group g are free: refill them
        issue(g + sg, s0);
        gs = gs + 1 == sg ? 0 : gs + 1;
    }
    cp_async_wait<0>();

    // partial y of this CTA
#pragma unroll
    for (int t = 0; t < TB; ++t) {
        const int b = b0 + t;
        if (b >= a.B) break;
        float *dst = a.part + ((size_t)c * a.B + b) * a.dp;
#pragma unroll
        for (int i = 0; i < MAXV; ++i) {
            if (vok[i]) {
                const int v = tid + i * nthr;
#pragma unroll
                for (int e = 0; e < V; e += 4) {
                    float4 o = make_float4(yacc[t][i][e], yacc[t][i][e + 1], yacc[t][i][e + 2], yacc[t][i][e + 3]);
                    *reinterpret_cast<float4 *>(dst + v * V + e) = o;
                }
            }
        }
    }
}

// y[b, col] = (resid[b, col] + scale *) sum_{c < G} part[c, b, col].  Warp w
// of 16 adds partials c = w, w + 16, ... in ascending order, every load of a
// thread in flight at once; the 16 warp sums are then added in warp order, so
// y is bit-reproducible.  Lane l of a CTA owns columns 2l, 2l + 1 of its
// 64-column slice.
constexpr int kRedWarps = 16;
constexpr int kRedUnroll = 16;   // partials per warp kept in flight (G <= 256 in one pass)

// gcount (optional, device): only the first min(G, *gcount) partials are
// added (the rest are known to be zero).
__global__ void __launch_bounds__(kRedWarps * 32)
ffn_reduce_kernel(const float *part, int G, int B, int d, int dp,
                  const float *resid, float scale, float *__restrict__ y, const int32_t *gcount) {
    __shared__ float2 red[kRedWarps][32];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int col = blockIdx.x * 64 + 2 * lane;
    const int b = blockIdx.y;
    pdl_launch_dependents();
    pdl_wait();
    if (gcount) {
        const int n = ld_dep(gcount);
        G = n < 0 ? 0 : n < G ? n : G;
    }
    float2 acc = make_float2(0.f, 0.f);
    if (col < d) {
        // col + 1 < dp (dp is a multiple of 8), so the pair load stays inside the row
        const float *p = part + (size_t)b * dp + col;
        const size_t stride = (size_t)B * dp;
        float2 t[kRedUnroll];
#pragma unroll
        for (int u = 0; u < kRedUnroll; ++u) {
            const int c = warp + kRedWarps * u;
            t[u] = c < G ? ld_dep(reinterpret_cast<const float2 *>(p + c * stride)) : make_float2(0.f, 0.f);
        }
#pragma unroll
        for (int u = 0; u < kRedUnroll; ++u) { acc.x += t[u].x; acc.y += t[u].y; }
        for (int c = warp + kRedWarps * kRedUnroll; c < G; c += kRedWarps) {
            const float2 v = ld_dep(reinterpret_cast<const float2 *>(p + c * stride));
            acc.x += v.x;
            acc.y += v.y;
        }
    }
    red[warp][lane] = acc;
    __syncthreads();
    if (warp == 0 && col < d) {
        float2 s = make_float2(0.f, 0.f);
#pragma unroll
        for (int w = 0; w < kRedWarps; ++w) { s.x += red[w][lane].x; s.y += red[w][lane].y; }
        const size_t o = (size_t)b * d + col;
        y[o] = resid ? fmaf(scale, s.x, resid[o]) : s.x;
        if (col + 1 < d) y[o + 1] = resid ? fmaf(scale, s.y, resid[o + 1]) : s.y;
    }
}

template <typename T, int TB, bool GLU, bool PRE, int MAXV>
cudaError_t run_gather(const FfnArgs &a, FfnK k, size_t smem, cudaStream_t s) {
    auto fn = ffn_gather_kernel<T, TB, GLU, PRE, MAXV>;
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // one thread per vector when a row has at most 1024 of them
    const int thr = ((k.nvec + MAXV - 1) / MAXV + 31) & ~31;
    dim3 grid(a.G, (a.B + TB - 1) / TB);
    return launch(fn, grid, dim3(thr), smem, s, pdl_enabled(), k);
}

template <typename T, int TB, bool GLU, bool PRE>
cudaError_t pick_maxv(const FfnArgs &a, const FfnK &k, size_t smem, cudaStream_t s) {
    if (k.nvec <= kMaxThreads) return run_gather<T, TB, GLU, PRE, 1>(a, k, smem, s);
    if (k.nvec <= 2 * kMaxThreads) return run_gather<T, TB, GLU, PRE, 2>(a, k, smem, s);
    if (k.nvec <= 4 * kMaxThreads) return run_gather<T, TB, GLU, PRE, 4>(a, k, smem, s);
    return run_gather<T, TB, GLU, PRE, 8>(a, k, smem, s);
}

template <typename T, int TB>
cudaError_t pick_mode(const FfnArgs &a, const FfnK &k, size_t smem, cudaStream_t s) {
    const bool glu = a.w_up != nullptr, pre = a.preact != nullptr;
    if (glu) return pre ? pick_maxv<T, TB, true, true>(a, k, smem, s) : pick_maxv<T, TB, true, false>(a, k, smem, s);
    return pre ? pick_maxv<T, TB, false, true>(a, k, smem, s) : pick_maxv<T, TB, false, false>(a, k, smem, s);
}

// The specialised one-token gather (cs_ffn1.cu) is used unless CS_GATHER1=0.
bool gather1_enabled() {
    static const bool on = [] {
        const char *v = getenv("CS_GATHER1");
        return !(v && v[0] == '0');
    }();
    return on;
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
    k.act = a.act;
    k.nvec = (a.d * esz + 15) / 16;
    const int nrow = (a.preact ? 0 : 1) + (a.w_up ? 1 : 0) + 1;
    const size_t per_neuron = (size_t)nrow * k.nvec * 16;
    // ring of sg groups of ng neurons: as deep as the budget allows
    const int nst = (int)(kRingBudget / per_neuron);
    if (nst < 2) return cudaErrorInvalidValue;
    // three ring groups keep one group in flight while two are in use
    if (nst >= 3 * kNgMax) { k.ng = kNgMax; k.sg = 3; }
    else if (nst >= 9) { k.ng = 3; k.sg = 3; }
    else if (nst >= 6) { k.ng = 2; k.sg = 3; }
    else if (nst >= 3) { k.ng = 1; k.sg = 3; }
    else { k.ng = 1; k.sg = 2; }
    static_assert(3 * kNgMax <= kStageMax, "ring slots");
    const size_t smem = (size_t)k.ng * k.sg * per_neuron;
    const int tb = a.B >= 2 ? 2 : 1;
    cudaError_t e;
    if (gather1_applies(k, a.B) && gather1_enabled())
        e = launch_gather1(a.dtype, k, smem, a.G, a.w_up != nullptr, a.preact != nullptr, s);
    else
        e = tb == 2 ? pick_mode<T, 2>(a, k, smem, s) : pick_mode<T, 1>(a, k, smem, s);
    if (e != cudaSuccess) return e;
    dim3 g((a.d + 63) / 64, a.B);
    return launch(ffn_reduce_kernel, g, dim3(kRedWarps * 32), 0, s, pdl_enabled(),
                  static_cast<const float *>(a.part), a.G, a.B, a.d, a.dp, a.resid, a.scale, a.y,
                  static_cast<const int32_t *>(nullptr));
}

}  // namespace

// Largest d (in elements) the gather kernel takes for a dtype.
int ffn_max_d(cs_dtype t) {
    const int V = t == CS_F32 ? 4 : 8;
    return 8 * kMaxThreads * V;
}

cudaError_t launch_ffn_reduce(const float *part, int G, int B, int d, int dp, const float *resid, float scale,
                              float *y, cudaStream_t s, const int32_t *gcount) {
    dim3 g((d + 63) / 64, B);
    return launch(ffn_reduce_kernel, g, dim3(kRedWarps * 32), 0, s, pdl_enabled(), part, G, B, d, dp, resid, scale, y,
                  gcount);
}

cudaError_t launch_ffn(const FfnArgs &a, cudaStream_t s) {
    if (tc_path_applies(a)) return launch_ffn_tc(a, s);
    switch (a.dtype) {
    case CS_F32: return run_ffn<float>(a, s);
    case CS_F16: return run_ffn<__half>(a, s);
    default: return run_ffn<__nv_bfloat16>(a, s);
    }
}

}  // namespace cs
