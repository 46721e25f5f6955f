// Head-sparse attention for one decode token: only the selected heads' query
// projection, attention over the KV cache and output projection run.
//
// Sources: "Contextual Sparsity and Activation Predictors", first section (a
// small, input-dependent set of attention heads approximates the layer);
// "Contextual Sparsity: Activation-Aware LLM Inference and the Deja Vu
// Paradigm", sections "The Empirical Foundation" (20-30% of heads contribute
// per token) and "Implications for System Design" (select the heads to
// compute per token).  The heads come from the same predictor and top-k as
// the FFN's neurons (a predictor with one output per head).
//
// For each selected head h, over S cached keys / values ([H, S, d_head]):
//     q = W_q[h] x,  s_i = q . k_i / sqrt(d_head),  p = softmax(s),
//     o = sum_i p_i v_i,  y += W_o[:, h] o.
//
// GB300 mapping.  Grids span every head slot (the launch never depends on the
// device-side count): slot m < count takes head idx[m], the others skip or
// write zero partials.  The query kernel spreads each head's W_q rows over
// (slot, 8-row block) CTAs, one warp per row.  The core kernel gives each
// head (slot, column chunk) CTAs: each forms the scores of all S keys (one
// thread per key), a max-subtracted softmax with fixed-order sums and o
// (threads over (key residue, 16-byte channel vector) pairs, combined in a
// fixed order),
// then its chunk of W_o[:, h] o, four warp groups over the d_head rows added
// in order.  The chunks of one head repeat the softmax; their K and V come
// from L2 after the first.  The FFN's fixed-order reduction adds the H
// partials, so y is bit-reproducible.
#include <algorithm>

#include "cs_internal.cuh"

using namespace cs;

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnMaxS = 16384;

struct AttnK {
    const uint8_t *w_q, *w_o_t, *k, *v;
    const float *x;
    const int32_t *idx, *count;
    float *part;    // [H, dp] per-head partial outputs
    float *qbuf;    // [H, dh] queries of the slots
    uint32_t *err;
    int d, H, dh, S, dp;
    size_t row_bytes;   // d * element size
};

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

constexpr int kQRows = 8;       // query rows per CTA (one per warp)
constexpr int kOVec = 64;       // 16-byte column vectors of the output projection per CTA
constexpr int kOGroups = kAttnThreads / kOVec;

// The head of slot m, or -1 (slot beyond the count, or an id out of range).
__device__ __forceinline__ int slot_head(const AttnK &a, int m, bool flag) {
    int n = *a.count;
    if (n < 0 || n > a.H) {
        if (flag && m == 0 && threadIdx.x == 0) atomicOr(a.err, CS_DEVERR_COUNT);
        n = n < 0 ? 0 : a.H;
    }
    if (m >= n) return -1;
    const int h = a.idx[m];
    if (h < 0 || h >= a.H) {
        if (flag && threadIdx.x == 0) atomicOr(a.err, CS_DEVERR_INDEX);
        return -1;
    }
    return h;
}

// 1. q of the head in slot m, rows p*8 .. p*8+7 (one warp per row, lanes over
//    16-byte vectors of the row), scaled by 1/sqrt(d_head), into qbuf[m, :].
template <typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_q_kernel(const AttnK a) {
    constexpr int V = Vec<T>::N;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int m = blockIdx.x;
    pdl_launch_dependents();
    pdl_wait();  // the head list comes from the selection
    const int h = slot_head(a, m, blockIdx.y == 0);
    const int c = blockIdx.y * kQRows + warp;
    if (h < 0 || c >= a.dh) return;
    const int nv = a.d / V;
    const uint4 *row = reinterpret_cast<const uint4 *>(a.w_q + ((size_t)h * a.dh + c) * a.row_bytes);
    float acc = 0.f;
    for (int v = lane; v < nv; v += 32) {
        float w[V];
        unpack<T>(__ldg(row + v), w);
        const float4 *xv = reinterpret_cast<const float4 *>(a.x + (size_t)v * V);
#pragma unroll
        for (int e = 0; e < V; e += 4) {
            const float4 x4 = ld_dep(xv + e / 4);
            acc = fmaf(w[e], x4.x, acc);
            acc = fmaf(w[e + 1], x4.y, acc);
            acc = fmaf(w[e + 2], x4.z, acc);
            acc = fmaf(w[e + 3], x4.w, acc);
        }
    }
    acc = warp_sum(acc);
    if (lane == 0) a.qbuf[(size_t)m * a.dh + c] = acc * (1.f / sqrtf((float)a.dh));
}

// 2-5. For the head in slot m: scores of the S keys, softmax, o, and this
//      CTA's chunk p of kOVec column vectors of the output projection.  Every
//      chunk of a head repeats steps 2-4 (its K and V come from L2 after the
//      first), so the output projection spreads over many SMs.
template <typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_core_kernel(const AttnK a) {
    constexpr int V = Vec<T>::N;
    extern __shared__ __align__(16) float sm[];
    const int dh = a.dh, d = a.d, S = a.S;
    float *q = sm;                              // [dh]
    float *o = q + dh;                          // [dh]
    float *red = o + dh;                        // [kAttnThreads]
    float *red5 = red + kAttnThreads;           // [kOGroups][kOVec][V]
    float *s = red5 + kOGroups * kOVec * V;     // [S]
    __shared__ float wred[kAttnWarps];
    __shared__ float s_max, s_z;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = blockIdx.x, p = blockIdx.y;
    const int nv = d / V;
    const int v0 = p * kOVec, v1 = min(nv, v0 + kOVec);
    float *part = a.part + (size_t)m * a.dp;

    pdl_launch_dependents();
    pdl_wait();  // q comes from the query kernel
    const int h = slot_head(a, m, false);
    if (h < 0) {
        for (int c = v0 * V + tid; c < v1 * V; c += kAttnThreads) part[c] = 0.f;
        return;
    }
    for (int c = tid; c < dh; c += kAttnThreads) q[c] = a.qbuf[(size_t)m * dh + c];
    __syncthreads();

    // 2. scores and their maximum
    const int kv = dh / V;
    const size_t head_bytes = (size_t)S * dh * sizeof(T);
    const uint8_t *kb = a.k + (size_t)h * head_bytes;
    float lmax = -INFINITY;
    for (int i = tid; i < S; i += kAttnThreads) {
        const uint4 *kr = reinterpret_cast<const uint4 *>(kb + (size_t)i * dh * sizeof(T));
        float acc = 0.f;
        for (int v = 0; v < kv; ++v) {
            float w[V];
            unpack<T>(__ldg(kr + v), w);
#pragma unroll
            for (int e = 0; e < V; ++e) acc = fmaf(q[v * V + e], w[e], acc);
        }
        s[i] = acc;
        lmax = fmaxf(lmax, acc);
    }
    lmax = warp_max_f(lmax);
    if (lane == 0) wred[warp] = lmax;
    __syncthreads();
    if (warp == 0) {
        float v = lane < kAttnWarps ? wred[lane] : -INFINITY;
        v = warp_max_f(v);
        if (lane == 0) s_max = v;
    }
    __syncthreads();
    const float mx = s_max;

    // 3. p_i = e^(s_i - max) and their sum, in a fixed order
    float lz = 0.f;
    for (int i = tid; i < S; i += kAttnThreads) {
        const float pe = expf(s[i] - mx);
        s[i] = pe;
        lz += pe;
    }
    lz = warp_sum(lz);
    if (lane == 0) wred[warp] = lz;
    __syncthreads();
    if (warp == 0) {
        float v = lane < kAttnWarps ? wred[lane] : 0.f;
        v = warp_sum(v);
        if (lane == 0) s_z = v;
    }
    __syncthreads();
    const float inv_z = 1.f / s_z;

    // 4. o[c] = sum_i p_i v_i[c] / Z: thread (g, u) takes keys i = g (mod G)
    //    and the 16-byte vector u of channels; the G groups are added in order
    //    (d_head / V vectors per row, a power of two, so G * (d_head / V) = 256)
    {
        const int nvh = dh / V, G = kAttnThreads / nvh;
        const int u = tid % nvh, g = tid / nvh;
        const uint4 *vb = reinterpret_cast<const uint4 *>(a.v + (size_t)h * head_bytes);
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        for (int i = g; i < S; i += G) {
            float w[V];
            unpack<T>(__ldg(vb + (size_t)i * nvh + u), w);
            const float pi = s[i];
#pragma unroll
            for (int e = 0; e < V; ++e) acc[e] = fmaf(pi, w[e], acc[e]);
        }
#pragma unroll
        for (int e = 0; e < V; ++e) red5[(size_t)tid * V + e] = acc[e];   // [g][u][e]
        __syncthreads();
        if (tid < dh) {
            const int uu = tid / V, ee = tid % V;
            float t = 0.f;
            for (int gg = 0; gg < G; ++gg) t += red5[((size_t)gg * nvh + uu) * V + ee];
            o[tid] = t * inv_z;
        }
        __syncthreads();
    }

    // 5. columns [v0*V, v1*V) of this head's partial: group g sums rows
    //    c = g (mod kOGroups), then the groups are added in order
    {
        const int g = tid / kOVec, vl = tid % kOVec, v = v0 + vl;
        float acc[V];
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = 0.f;
        if (v < v1) {
            for (int c = g; c < dh; c += kOGroups) {
                const uint4 *row = reinterpret_cast<const uint4 *>(a.w_o_t + ((size_t)h * dh + c) * a.row_bytes);
                float w[V];
                unpack<T>(__ldg(row + v), w);
                const float oc = o[c];
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = fmaf(oc, w[e], acc[e]);
            }
        }
#pragma unroll
        for (int e = 0; e < V; ++e) red5[((size_t)g * kOVec + vl) * V + e] = acc[e];
        __syncthreads();
        if (g == 0 && v < v1) {
#pragma unroll
            for (int e = 0; e < V; ++e) {
                float t = 0.f;
                for (int gg = 0; gg < kOGroups; ++gg) t += red5[((size_t)gg * kOVec + vl) * V + e];
                part[(size_t)v * V + e] = t;
            }
        }
    }
}

template <typename T>
cudaError_t run_attn(const AttnK &k, cudaStream_t s) {
    constexpr int V = Vec<T>::N;
    cudaError_t e = launch(attn_q_kernel<T>, dim3(k.H, (k.dh + kQRows - 1) / kQRows), dim3(kAttnThreads), 0, s,
                           pdl_enabled(), k);
    if (e != cudaSuccess) return e;
    const size_t smem = sizeof(float) * ((size_t)2 * k.dh + kAttnThreads + (size_t)kOGroups * kOVec * V + k.S);
    auto fn = attn_core_kernel<T>;
    e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    const int nv = k.d / V;
    return launch(fn, dim3(k.H, (nv + kOVec - 1) / kOVec), dim3(kAttnThreads), smem, s, pdl_enabled(), k);
}

}  // namespace

extern "C" {

cs_status cs_sparse_attention(const cs_attn_layer *layer, const float *x, const int32_t *heads,
                              const int32_t *count, const void *k_cache, const void *v_cache, int seq_len,
                              float *y, void *ws, size_t ws_bytes, cs_stream_t stream) {
    if (!layer || !x || !heads || !count || !k_cache || !v_cache || !y) {
        set_error("cs_sparse_attention: layer, x, heads, count, k_cache, v_cache and y are required");
        return CS_ERR_INVALID;
    }
    const cs_attn_layer &L = *layer;
    if (L.dtype != CS_F32 && L.dtype != CS_F16 && L.dtype != CS_BF16) {
        set_error("cs_sparse_attention: bad dtype %d", (int)L.dtype);
        return CS_ERR_INVALID;
    }
    const int esz = (int)dtype_size(L.dtype), V = 16 / esz;
    const bool dh_ok = L.d_head >= V && L.d_head <= kAttnThreads && (L.d_head & (L.d_head - 1)) == 0;
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (L.d < V || L.d % V || L.n_heads < 1 || !dh_ok || !L.w_q || !L.w_o_t || !al16(L.w_q) || !al16(L.w_o_t) ||
        !al16(x) || !al16(k_cache) || !al16(v_cache) || (reinterpret_cast<uintptr_t>(heads) & 3u) ||
        (reinterpret_cast<uintptr_t>(count) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u) || x == y) {
        set_error("cs_sparse_attention: d a multiple of %d, d_head a power of two in [%d, %d], 16-byte aligned "
                  "weights, caches and x, and y not aliasing x", V, V, kAttnThreads);
        return CS_ERR_INVALID;
    }
    if (seq_len < 1 || seq_len > kAttnMaxS) {
        set_error("cs_sparse_attention: seq_len=%d outside [1, %d]", seq_len, kAttnMaxS);
        return seq_len < 1 ? CS_ERR_INVALID : CS_ERR_UNSUPPORTED;
    }
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) {
        set_error("cs_sparse_attention: workspace is null or not 256-byte aligned");
        return CS_ERR_WORKSPACE;
    }
    // the partial outputs use the workspace's per-CTA partial rows (one per head)
    const WsLayout WL = ws_layout(L.d, 1, 1, 1, device_sm_count());
    if (ws_bytes < WL.total) {
        set_error("cs_sparse_attention: workspace too small: %zu bytes given, %zu needed", ws_bytes, WL.total);
        return CS_ERR_WORKSPACE;
    }
    // H partial rows, then the H queries, inside the workspace's G partial rows
    const size_t q_rows = ((size_t)L.n_heads * L.d_head + WL.dp - 1) / WL.dp;
    if ((size_t)L.n_heads + q_rows > (size_t)WL.G) {
        set_error("cs_sparse_attention: %d heads of %d need more than the %d partial rows of the workspace",
                  L.n_heads, L.d_head, WL.G);
        return CS_ERR_UNSUPPORTED;
    }
    AttnK k;
    k.w_q = static_cast<const uint8_t *>(L.w_q);
    k.w_o_t = static_cast<const uint8_t *>(L.w_o_t);
    k.k = static_cast<const uint8_t *>(k_cache);
    k.v = static_cast<const uint8_t *>(v_cache);
    k.x = x;
    k.idx = heads;
    k.count = count;
    k.part = reinterpret_cast<float *>(static_cast<char *>(ws) + WL.part);
    k.qbuf = k.part + (size_t)L.n_heads * WL.dp;
    k.err = static_cast<uint32_t *>(ws);
    k.d = L.d;
    k.H = L.n_heads;
    k.dh = L.d_head;
    k.S = seq_len;
    k.dp = WL.dp;
    k.row_bytes = (size_t)L.d * esz;
    cudaStream_t s = (cudaStream_t)stream;
    cudaError_t e = L.dtype == CS_F32 ? run_attn<float>(k, s)
                    : L.dtype == CS_F16 ? run_attn<__half>(k, s)
                                        : run_attn<__nv_bfloat16>(k, s);
    if (e == cudaSuccess) e = launch_ffn_reduce(k.part, L.n_heads, 1, L.d, WL.dp, nullptr, 1.f, y, s);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_sparse_attention");
}

}  // extern "C"
