// Gathered sparse FFN for one token: the gate (and up) GEMV over the listed
// neurons, their activations, and the down-row AXPY into per-CTA partial sums
// (added in a fixed order by the FFN's reduction kernel).
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (sparse_mlp_forward: only
// the chosen neurons' rows are read), section "Kernel-Level Implementation"
// (rows are read whole and coalesced rather than one neuron per thread) and
// section "The SiLU/GELU Challenge: TurboSparse" (the gated form).
//
// Same data flow as the general gather kernel (one CTA per SM over a
// contiguous chunk of the ascending index list, one thread per 16-byte column
// vector, a per-thread cp.async ring of SG groups of NG neurons), specialised
// for the one-token case that decode runs at every layer, with everything the
// general kernel decides at run time fixed at compile time:
//  - NG neurons per group, so no neuron slot is computed or tested in vain;
//  - dot products and the down-row AXPY with packed fma.rn.f32x2 (two IEEE
//    single-precision FMAs per instruction, each rounded as fmaf);
//  - the dot products of a group reduced two at a time: one butterfly of five
//    shuffles reduces a pair of values across the warp (lane 0 ends with the
//    first sum, lane 16 with the second), and the same pairing adds the
//    per-warp sums across warps after the group's one block barrier; the
//    totals are taken from fixed lanes, so every thread uses the same bits.
// Summation orders are fixed, so results are bit-reproducible.
#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kThreads1 = 1024;
constexpr int kWarps1 = kThreads1 / 32;
constexpr int kChunk1 = 2048;   // ids per CTA (f <= 2048 * grid)

__device__ __forceinline__ void cp16(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
__device__ __forceinline__ void cp4(uint32_t dst, const void *src) {
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(dst), "l"(src) : "memory");
}

// d = a * b + c on each half (two fma.rn.f32).
__device__ __forceinline__ float2 ffma2(float2 a, float2 b, float2 c) {
    float2 d;
    asm("{\n\t.reg .b64 ra, rb, rc, rd;\n\t"
        "mov.b64 ra, {%2, %3};\n\t"
        "mov.b64 rb, {%4, %5};\n\t"
        "mov.b64 rc, {%6, %7};\n\t"
        "fma.rn.f32x2 rd, ra, rb, rc;\n\t"
        "mov.b64 {%0, %1}, rd;\n\t}"
        : "=f"(d.x), "=f"(d.y)
        : "f"(a.x), "f"(a.y), "f"(b.x), "f"(b.y), "f"(c.x), "f"(c.y));
    return d;
}

// A 16-byte vector of weights as V/2 pairs of floats.
__device__ __forceinline__ void unpack2(const uint4 &v, float2 (&o)[4], const __nv_bfloat16 *) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}
__device__ __forceinline__ void unpack2(const uint4 &v, float2 (&o)[4], const __half *) {
    const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) o[i] = __half22float2(*reinterpret_cast<const __half2 *>(&w[i]));
}
__device__ __forceinline__ void unpack2(const uint4 &v, float2 (&o)[2], const float *) {
    o[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
    o[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
}

// Sum over the warp of a (into lane 0) and of b (into lane 16); other lanes
// hold partial sums.
__device__ __forceinline__ float pair_sum(float a, float b) {
    const bool hi = threadIdx.x & 16;
    float keep = hi ? b : a;
    const float send = hi ? a : b;
    keep += __shfl_xor_sync(kFull, send, 16);
#pragma unroll
    for (int o = 8; o > 0; o >>= 1) keep += __shfl_xor_sync(kFull, keep, o);
    return keep;
}

template <typename T, bool GLU, bool PRE, int NG, int SG>
__global__ void __launch_bounds__(kThreads1, 1) ffn_gather1_kernel(const FfnK a) {
    constexpr int V = Vec<T>::N;
    constexpr int P = V / 2;                          // float pairs per vector
    constexpr int NROW = (PRE ? 0 : 1) + (GLU ? 1 : 0) + 1;
    constexpr int ND = (PRE ? 0 : 1) + (GLU ? 1 : 0); // dot products per neuron
    constexpr int NDOT = ND * NG;                     // per group
    constexpr int NPAIR = (NDOT + 1) / 2;
    constexpr int NPA = NPAIR > 0 ? NPAIR : 1;      // array extents
    extern __shared__ __align__(16) uint4 ring[];     // [SG * NG][NROW][nvec]
    __shared__ float red[2][NPA][2][kWarps1];
    __shared__ int s_idx[kChunk1];
    __shared__ float s_add[kChunk1];                  // bias (or pre-activation)

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int nwarps = blockDim.x >> 5;
    const int c = blockIdx.x, G = gridDim.x;
    const int nvec = a.nvec;
    const uint32_t row_bytes = (uint32_t)nvec * 16u;
    const uint32_t slot_bytes = NROW * row_bytes;
    const uint32_t ring_s = smem_addr(ring);
    const bool vok = tid < nvec;
    const int voff = tid * 16;

    pdl_launch_dependents();  // one wave: the next kernel may get resident now
    pdl_wait();               // idx, count and x come from earlier kernels

    int n = ld_dep(a.count);
    if (n < 0 || n > a.f) {
        if (tid == 0 && c == 0) atomicOr(a.err, CS_DEVERR_COUNT);
        n = n < 0 ? 0 : a.f;
    }
    const int n0 = (int)((long long)n * c / G);
    const int cnt = min(kChunk1, (int)((long long)n * (c + 1) / G) - n0);
    for (int m = tid; m < cnt; m += blockDim.x) s_idx[m] = ld_dep(a.idx + n0 + m);
    __syncthreads();
    for (int m = tid; m < cnt; m += blockDim.x) {
        int j = s_idx[m];
        j = (j >= 0 && j < a.f) ? j : 0;
        if (PRE) s_add[m] = ld_dep(a.preact + j);  // written by the pre-activation kernel
        else if (a.bias) cp4(smem_addr(&s_add[m]), a.bias + j);
        else s_add[m] = 0.f;
    }
    const int ngroups = (cnt + NG - 1) / NG;

    // this thread's copies for group g into slots [s0, s0 + NG)
    auto issue = [&](int g, int s0) {
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            const int m = g * NG + q;
            if (m < cnt && vok) {
                int j = s_idx[m];
                j = (j >= 0 && j < a.f) ? j : 0;
                const size_t roff = (size_t)j * (size_t)a.ldb + voff;
                uint32_t r = ring_s + (uint32_t)(s0 + q) * slot_bytes + (uint32_t)voff;
                if (!PRE) { cp16(r, a.w_gate + roff); r += row_bytes; }
                if (GLU) { cp16(r, a.w_up + roff); r += row_bytes; }
                cp16(r, a.w_down_t + roff);
            }
        }
        cp_async_commit();  // always commit, so group counting stays uniform
    };
#pragma unroll
    for (int g = 0; g < SG; ++g) issue(g, g * NG);  // group 0 also carries s_add

    // x as float pairs (zero past d), the output accumulators
    float2 xr[P], yacc[P];
    {
        const int col0 = tid * V;
        const bool xvec = (a.d & 3) == 0 && (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
        if (ND > 0 && vok && xvec && col0 + V <= a.d) {
#pragma unroll
            for (int e = 0; e < V; e += 4) {
                const float4 t = ld_dep(reinterpret_cast<const float4 *>(a.x + col0 + e));
                xr[e / 2] = make_float2(t.x, t.y);
                xr[e / 2 + 1] = make_float2(t.z, t.w);
            }
        } else {
#pragma unroll
            for (int e = 0; e < P; ++e) {
                const int c0 = col0 + 2 * e;
                xr[e].x = (ND > 0 && vok && c0 < a.d) ? ld_dep(a.x + c0) : 0.f;
                xr[e].y = (ND > 0 && vok && c0 + 1 < a.d) ? ld_dep(a.x + c0 + 1) : 0.f;
            }
        }
#pragma unroll
        for (int e = 0; e < P; ++e) yacc[e] = make_float2(0.f, 0.f);
    }
    // columns of this thread's vector past d (the row's padding, which may
    // hold anything) are masked out of the dot products
    const int ne = a.d - tid * V;

    int gs = 0;
    for (int g = 0; g < ngroups; ++g) {
        const int s0 = gs * NG;
        const int par = g & 1;
        cp_async_wait<SG - 1>();   // this thread's copies of group g have landed
        if (ND > 0) {
            // this thread's share of the group's dot products: dot[q * ND + r]
            float dot[NPA * 2];
#pragma unroll
            for (int q = 0; q < NG; ++q) {
#pragma unroll
                for (int r = 0; r < ND; ++r) {
                    float2 acc = make_float2(0.f, 0.f);
                    if (vok) {
                        float2 w[P];
                        unpack2(ring[(size_t)((s0 + q) * NROW + r) * nvec + tid], w, static_cast<const T *>(nullptr));
                        if (ne < V) {
#pragma unroll
                            for (int e = 0; e < P; ++e) {
                                w[e].x = 2 * e < ne ? w[e].x : 0.f;
                                w[e].y = 2 * e + 1 < ne ? w[e].y : 0.f;
                            }
                        }
#pragma unroll
                        for (int e = 0; e < P; ++e) acc = ffma2(w[e], xr[e], acc);
                    }
                    dot[q * ND + r] = acc.x + acc.y;
                }
            }
            if (NDOT & 1) dot[NPA * 2 - 1] = 0.f;
            // warp sums, two at a time: lane 0 holds the even one, lane 16 the odd
#pragma unroll
            for (int k = 0; k < NPAIR; ++k) {
                const float s = pair_sum(dot[2 * k], dot[2 * k + 1]);
                if ((lane & 15) == 0) red[par][k][lane >> 4][warp] = s;
            }
        }
        __syncthreads();  // the group's warp sums (and, at g = 0, s_add) are visible
        // the group's activations, from the warp sums added across warps
        float act[NG];
        if (ND > 0) {
            float tot[NPA * 2];
#pragma unroll
            for (int k = 0; k < NPAIR; ++k) {
                const float ea = lane < nwarps ? red[par][k][0][lane] : 0.f;
                const float eb = lane < nwarps ? red[par][k][1][lane] : 0.f;
                const float s = pair_sum(ea, eb);
                tot[2 * k] = __shfl_sync(kFull, s, 0);
                tot[2 * k + 1] = __shfl_sync(kFull, s, 16);
            }
#pragma unroll
            for (int q = 0; q < NG; ++q) {
                const int m = g * NG + q;
                const float gsum = PRE ? 0.f : tot[q * ND];
                const float usum = GLU ? tot[q * ND + ND - 1] : 1.f;
                const float gv = PRE ? s_add[m < cnt ? m : 0] : gsum + s_add[m < cnt ? m : 0];
                float v = gate_act(a.act, gv);
                if (GLU) v *= usum;
                act[q] = v;
            }
        } else {
#pragma unroll
            for (int q = 0; q < NG; ++q) {
                const int m = g * NG + q;
                act[q] = gate_act(a.act, s_add[m < cnt ? m : 0]);
            }
        }
        // y += a_j * w_down_j over this thread's vector
#pragma unroll
        for (int q = 0; q < NG; ++q) {
            const int m = g * NG + q;
            if (m < cnt) {
                const int j = s_idx[m];
                const bool valid = j >= 0 && j < a.f;
                if (!valid && tid == 0) atomicOr(a.err, CS_DEVERR_INDEX);
                const float av = valid ? act[q] : 0.f;
                if (vok) {
                    float2 w[P];
                    unpack2(ring[(size_t)((s0 + q) * NROW + NROW - 1) * nvec + tid], w, static_cast<const T *>(nullptr));
                    const float2 a2 = make_float2(av, av);
#pragma unroll
                    for (int e = 0; e < P; ++e) yacc[e] = ffma2(a2, w[e], yacc[e]);
                }
            }
        }
        // this thread's slots of group g are free: refill them
        issue(g + SG, s0);
        gs = gs + 1 == SG ? 0 : gs + 1;
    }
    cp_async_wait<0>();

    // partial y of this CTA
    if (vok) {
        float *dst = a.part + (size_t)c * a.dp + (size_t)tid * V;
#pragma unroll
        for (int e = 0; e < P; e += 2)
            *reinterpret_cast<float4 *>(dst + 2 * e) = make_float4(yacc[e].x, yacc[e].y, yacc[e + 1].x, yacc[e + 1].y);
    }
}

template <typename T, bool GLU, bool PRE>
cudaError_t run1(const FfnK &k, size_t smem, int G, cudaStream_t s) {
    void (*fn)(const FfnK) = nullptr;
    if (k.sg != 3) return cudaErrorNotSupported;
    switch (k.ng) {
    case 1: fn = ffn_gather1_kernel<T, GLU, PRE, 1, 3>; break;
    case 2: fn = ffn_gather1_kernel<T, GLU, PRE, 2, 3>; break;
    case 3: fn = ffn_gather1_kernel<T, GLU, PRE, 3, 3>; break;
    case 4: fn = ffn_gather1_kernel<T, GLU, PRE, 4, 3>; break;
    default: return cudaErrorNotSupported;
    }
    cudaError_t e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int thr = (k.nvec + 31) & ~31;
    return launch(fn, dim3(G), dim3(thr), smem, s, pdl_enabled(), k);
}

template <typename T>
cudaError_t run1_mode(const FfnK &k, size_t smem, int G, bool glu, bool pre, cudaStream_t s) {
    if (glu) return pre ? run1<T, true, true>(k, smem, G, s) : run1<T, true, false>(k, smem, G, s);
    return pre ? run1<T, false, true>(k, smem, G, s) : run1<T, false, false>(k, smem, G, s);
}

}  // namespace

bool gather1_applies(const FfnK &k, int B) {
    return B == 1 && k.nvec <= kThreads1 && k.sg == 3 && k.ng >= 1 && k.ng <= 4 && k.f <= 0x7fffffff;
}

cudaError_t launch_gather1(cs_dtype dt, const FfnK &k, size_t smem, int G, bool glu, bool pre, cudaStream_t s) {
    switch (dt) {
    case CS_F32: return run1_mode<float>(k, smem, G, glu, pre, s);
    case CS_F16: return run1_mode<__half>(k, smem, G, glu, pre, s);
    default: return run1_mode<__nv_bfloat16>(k, smem, G, glu, pre, s);
    }
}

}  // namespace cs
