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
// GB300 mapping: four kernels chained with programmatic dependent launch.
// Grids span every head slot (the launch never depends on the device-side
// count): slot m < count takes head idx[m], the others exit or write zero
// partials.
//  1. query: (slot, block of five W_q rows) CTAs; each row is spread over the
//     CTA (thread t takes 16-byte vectors t + 256 i), x in registers, one
//     block reduction per five rows.
//  2. attend, split over the keys (flash-decoding): a (slot, split) CTA owns
//     2048 / (vectors per key) keys, i.e. 32 KB of K and 32 KB of V, all of it
//     loaded into registers before waiting for the query; it forms its
//     scores, their maximum m, l = sum e^(s - m) and the unnormalised
//     o = sum e^(s - m) v, and writes (m, l, o).
//  3. combine and project: a (slot, 64-vector column chunk) CTA merges the
//     head's splits in split order (M = max m, L = sum l e^(m - M),
//     o = sum o_s e^(m - M) / L) and applies its chunk of W_o[:, h] o (four
//     row groups added in order); a thread's first 24 rows (96 of d_head 128)
//     are loaded before the wait, so they stream in while the attend kernel
//     runs (all 32 would need registers that keep an attend CTA off the SM).
//  4. the FFN's fixed-order reduction adds the per-slot partials.
// Kernels 1-3 let their dependents launch only after their own wait, so when
// kernels 2 and 3 start the selection that wrote the head list has finished
// and they may read it, and fetch K, V and W_o rows, before their wait.  All
// sums run in fixed orders, so y is bit-reproducible.
#include <algorithm>

#include "cs_internal.cuh"

using namespace cs;

namespace {

constexpr int kAttnThreads = 256;
constexpr int kAttnWarps = kAttnThreads / 32;
constexpr int kAttnMaxS = 16384;
constexpr int kSplitVec = 2048;   // 16-byte vectors of K (and of V) per split: 8 per thread
constexpr int kKV = kSplitVec / kAttnThreads;
constexpr int kQRows = 5;         // W_q rows per query CTA (10 heads of 128 rows: 260 CTAs, one wave)
constexpr int kOVec = 64;         // 16-byte column vectors of the output projection per CTA
constexpr int kOGroups = kAttnThreads / kOVec;
constexpr int kOPre = 24;         // W_o rows per thread loaded before the wait (the registers leave room for an attend CTA)

struct AttnK {
    const uint8_t *w_q, *w_o_t, *k, *v;
    const float *x;
    const int32_t *idx, *count;
    float *part;    // [H, dp] per-slot partial outputs
    float *qbuf;    // [H, dh] queries of the slots
    float *split;   // [H, ns, dh + 2] per-split (m, l, o)
    uint32_t *err;
    int d, H, dh, S, dp;
    int nvk;        // 16-byte vectors per key (and per W_q / W_o row block column)
    int sc;         // keys per split
    int ns;         // splits
    size_t row_bytes;   // d * element size
};

__device__ __forceinline__ float warp_max_f(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(kFull, v, o));
    return v;
}

// The head of slot m, or -1 (slot beyond the count, or an id out of range).
// flag: this CTA reports a bad count or id in the error word.
__device__ __forceinline__ int slot_head(const AttnK &a, int m, bool flag) {
    int n = ld_dep(a.count);
    if (n < 0 || n > a.H) {
        if (flag && m == 0 && threadIdx.x == 0) atomicOr(a.err, CS_DEVERR_COUNT);
        n = n < 0 ? 0 : a.H;
    }
    if (m >= n) return -1;
    const int h = ld_dep(a.idx + m);
    if (h < 0 || h >= a.H) {
        if (flag && threadIdx.x == 0) atomicOr(a.err, CS_DEVERR_INDEX);
        return -1;
    }
    return h;
}

// 1. rows r0 .. r0+4 of q for the head in slot m (scaled by 1/sqrt(d_head)).
template <typename T, int NV>
__global__ void __launch_bounds__(kAttnThreads) attn_q_kernel(const AttnK a) {
    constexpr int V = Vec<T>::N;
    __shared__ float red[kQRows][kAttnWarps];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = blockIdx.y, r0 = blockIdx.x * kQRows;
    pdl_wait();               // the head list comes from the selection
    pdl_launch_dependents();  // (after the wait: dependents may read the head list)
    const int h = slot_head(a, m, blockIdx.x == 0);
    if (h < 0) return;
    const int nv = a.d / V;
    uint4 w[kQRows][NV];
#pragma unroll
    for (int u = 0; u < kQRows; ++u) {
        const int row = min(r0 + u, a.dh - 1);
        const uint4 *rp = reinterpret_cast<const uint4 *>(a.w_q + ((size_t)h * a.dh + row) * a.row_bytes);
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            const int v = tid + i * kAttnThreads;
            w[u][i] = v < nv ? __ldg(rp + v) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    float xr[NV][V];
#pragma unroll
    for (int i = 0; i < NV; ++i) {
        const int v = tid + i * kAttnThreads;
#pragma unroll
        for (int e = 0; e < V; e += 4) {
            const float4 t = v < nv ? ld_dep(reinterpret_cast<const float4 *>(a.x + (size_t)v * V + e))
                                    : make_float4(0.f, 0.f, 0.f, 0.f);
            xr[i][e] = t.x; xr[i][e + 1] = t.y; xr[i][e + 2] = t.z; xr[i][e + 3] = t.w;
        }
    }
#pragma unroll
    for (int u = 0; u < kQRows; ++u) {
        float acc[NV];
#pragma unroll
        for (int i = 0; i < NV; ++i) {
            float f[V];
            unpack<T>(w[u][i], f);
            acc[i] = 0.f;
#pragma unroll
            for (int e = 0; e < V; ++e) acc[i] = fmaf(f[e], xr[i][e], acc[i]);
        }
        float t = acc[0];
#pragma unroll
        for (int i = 1; i < NV; ++i) t += acc[i];
        t = warp_sum(t);
        if (lane == 0) red[u][warp] = t;
    }
    __syncthreads();
    if (tid < kQRows && r0 + tid < a.dh) {
        float t = 0.f;
#pragma unroll
        for (int q = 0; q < kAttnWarps; ++q) t += red[tid][q];
        a.qbuf[(size_t)m * a.dh + r0 + tid] = t * (1.f / sqrtf((float)a.dh));
    }
}

// 2. split s of the keys of the head in slot m: (max, sum, unnormalised o).
//    Thread t holds vectors e = t + 256 j (j < 8) of the split's K block and
//    of its V block: key e / nvk, channel vector t % nvk (the same for every
//    j, since nvk divides 256).
template <typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_split_kernel(const AttnK a) {
    constexpr int V = Vec<T>::N;
    __shared__ float sc[kSplitVec];               // the split's scores (at most 2048 keys)
    __shared__ float red[kAttnWarps];
    __shared__ float ored[kAttnThreads * V];      // [thread][channel] partial o
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int m = blockIdx.y, s = blockIdx.x;
    const int nvk = a.nvk, u = tid % nvk;
    const int k0 = s * a.sc;                      // first key of the split
    const int nk = min(a.sc, a.S - k0);           // keys in the split
    const int h = slot_head(a, m, false);         // the selection has finished (see above)
    uint4 kr[kKV], vr[kKV];
    if (h >= 0) {
        const size_t head = (size_t)h * a.S * nvk;          // in vectors
        const uint4 *kb = reinterpret_cast<const uint4 *>(a.k) + head + (size_t)k0 * nvk;
        const uint4 *vb = reinterpret_cast<const uint4 *>(a.v) + head + (size_t)k0 * nvk;
        const int nvec = nk * nvk;
#pragma unroll
        for (int j = 0; j < kKV; ++j) {
            const int e = tid + j * kAttnThreads;
            kr[j] = e < nvec ? __ldg(kb + e) : make_uint4(0u, 0u, 0u, 0u);
            vr[j] = e < nvec ? __ldg(vb + e) : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    pdl_wait();               // q comes from the query kernel
    pdl_launch_dependents();
    if (h < 0) return;
    float qr[V];
#pragma unroll
    for (int e = 0; e < V; ++e) qr[e] = ld_dep(a.qbuf + (size_t)m * a.dh + u * V + e);

    // scores: each key's nvk vectors lie in consecutive threads (nvk <= 32:
    // one warp; nvk = 64: two warps, added through shared memory)
    const int lpk = min(nvk, 32);
#pragma unroll
    for (int j = 0; j < kKV; ++j) {
        float f[V];
        unpack<T>(kr[j], f);
        float t = 0.f;
#pragma unroll
        for (int e = 0; e < V; ++e) t = fmaf(qr[e], f[e], t);
        for (int o = lpk >> 1; o > 0; o >>= 1) t += __shfl_xor_sync(kFull, t, o);
        const int e = tid + j * kAttnThreads, key = e / nvk;
        if (nvk <= 32) {
            if ((lane & (lpk - 1)) == 0 && key < nk) sc[key] = t;
        } else {
            // nvk = 64: warps 2w and 2w + 1 hold the halves of one key
            if (lane == 0) ored[warp + j * kAttnWarps] = t;
        }
    }
    __syncthreads();
    if (nvk > 32) {
        // key (j, w2) of the 8 x 4 keys: halves from warps 2 w2 and 2 w2 + 1
        if (tid < kKV * kAttnWarps / 2) {
            const int j = tid / (kAttnWarps / 2), w2 = tid % (kAttnWarps / 2);
            const int key = (j * kAttnThreads + w2 * 64) / 64;
            if (key < nk) sc[key] = ored[2 * w2 + j * kAttnWarps] + ored[2 * w2 + 1 + j * kAttnWarps];
        }
        __syncthreads();
    }
    // the split's maximum and e^(s - m), summed in a fixed order
    float mx = -INFINITY;
    for (int i = tid; i < nk; i += kAttnThreads) mx = fmaxf(mx, sc[i]);
    mx = warp_max_f(mx);
    if (lane == 0) red[warp] = mx;
    __syncthreads();
    mx = red[0];
#pragma unroll
    for (int q = 1; q < kAttnWarps; ++q) mx = fmaxf(mx, red[q]);
    __syncthreads();
    float lz = 0.f;
    for (int i = tid; i < nk; i += kAttnThreads) {
        const float p = expf(sc[i] - mx);
        sc[i] = p;
        lz += p;
    }
    lz = warp_sum(lz);
    if (lane == 0) red[warp] = lz;
    __syncthreads();
    // o: each thread adds its keys' p v over its channel vector, then the
    // 256 / nvk threads of one channel vector are added in thread order
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
#pragma unroll
    for (int j = 0; j < kKV; ++j) {
        const int key = (tid + j * kAttnThreads) / nvk;
        const float p = key < nk ? sc[key] : 0.f;
        float f[V];
        unpack<T>(vr[j], f);
#pragma unroll
        for (int e = 0; e < V; ++e) acc[e] = fmaf(p, f[e], acc[e]);
    }
#pragma unroll
    for (int e = 0; e < V; ++e) ored[tid * V + e] = acc[e];
    __syncthreads();
    float *out = a.split + ((size_t)m * a.ns + s) * (a.dh + 2);
    if (tid < a.dh) {
        const int uu = tid / V, ee = tid % V;
        float t = 0.f;
        for (int g = uu; g < kAttnThreads; g += nvk) t += ored[g * V + ee];
        out[2 + tid] = t;
    }
    if (tid == 0) {
        float l = 0.f;
#pragma unroll
        for (int q = 0; q < kAttnWarps; ++q) l += red[q];
        out[0] = mx;
        out[1] = l;
    }
}

// 3. merge the splits of the head in slot m, then columns [v0*V, v1*V) of
//    its partial: group g sums rows c = g (mod 4), groups added in order.
template <typename T>
__global__ void __launch_bounds__(kAttnThreads) attn_out_kernel(const AttnK a) {
    constexpr int V = Vec<T>::N;
    __shared__ float o[256];
    __shared__ float wgt[kAttnMaxS / 32];         // m_s, then e^(m_s - M), per split
    __shared__ float lsum[kAttnMaxS / 32];        // l_s per split
    __shared__ float s_inv;
    __shared__ float red5[kOGroups * kOVec * V];
    const int tid = threadIdx.x;
    const int m = blockIdx.y, p = blockIdx.x;
    const int dh = a.dh, nv = a.d / V;
    const int v0 = p * kOVec, v1 = min(nv, v0 + kOVec);
    const int g = tid / kOVec, vl = tid % kOVec, v = v0 + vl;
    float *part = a.part + (size_t)m * a.dp;
    const int h = slot_head(a, m, false);         // the selection has finished
    uint4 wpre[kOPre];
    if (h >= 0 && v < v1) {
#pragma unroll
        for (int r = 0; r < kOPre; ++r) {
            const int c = g + r * kOGroups;
            wpre[r] = c < dh ? __ldg(reinterpret_cast<const uint4 *>(a.w_o_t + ((size_t)h * dh + c) * a.row_bytes) + v)
                             : make_uint4(0u, 0u, 0u, 0u);
        }
    }
    pdl_wait();               // the splits come from the attend kernel
    pdl_launch_dependents();
    if (h < 0) {
        for (int c = v0 * V + tid; c < v1 * V; c += kAttnThreads) part[c] = 0.f;
        return;
    }
    const float *sp = a.split + (size_t)m * a.ns * (dh + 2);
    // the splits' maxima and sums, one thread per split, then M and L by warp
    // 0 in split order
    for (int s = tid; s < a.ns; s += kAttnThreads) {
        wgt[s] = ld_dep(sp + (size_t)s * (dh + 2));
        lsum[s] = ld_dep(sp + (size_t)s * (dh + 2) + 1);
    }
    __syncthreads();
    if (tid == 0) {
        float M = -INFINITY;
        for (int s = 0; s < a.ns; ++s) M = fmaxf(M, wgt[s]);
        float L = 0.f;
        for (int s = 0; s < a.ns; ++s) {
            const float w = expf(wgt[s] - M);
            wgt[s] = w;
            L += lsum[s] * w;
        }
        s_inv = 1.f / L;
    }
    __syncthreads();
    if (tid < dh) {
        float t = 0.f;
        for (int s = 0; s < a.ns; ++s) t += ld_dep(sp + (size_t)s * (dh + 2) + 2 + tid) * wgt[s];
        o[tid] = t * s_inv;
    }
    __syncthreads();
    float acc[V];
#pragma unroll
    for (int e = 0; e < V; ++e) acc[e] = 0.f;
    if (v < v1) {
#pragma unroll
        for (int r = 0; r < kOPre; ++r) {
            const int c = g + r * kOGroups;
            if (c < dh) {
                float f[V];
                unpack<T>(wpre[r], f);
                const float oc = o[c];
#pragma unroll
                for (int e = 0; e < V; ++e) acc[e] = fmaf(oc, f[e], acc[e]);
            }
        }
        // the remaining rows eight at a time, all eight loads in flight
        const uint4 *col = reinterpret_cast<const uint4 *>(a.w_o_t + (size_t)h * dh * a.row_bytes) + v;
        const size_t rstride = a.row_bytes / 16;
        for (int c0 = g + kOPre * kOGroups; c0 < dh; c0 += 8 * kOGroups) {
            uint4 wr[8];
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int c = c0 + r * kOGroups;
                wr[r] = c < dh ? __ldg(col + (size_t)c * rstride) : make_uint4(0u, 0u, 0u, 0u);
            }
#pragma unroll
            for (int r = 0; r < 8; ++r) {
                const int c = c0 + r * kOGroups;
                if (c < dh) {
                    float f[V];
                    unpack<T>(wr[r], f);
                    const float oc = o[c];
#pragma unroll
                    for (int e = 0; e < V; ++e) acc[e] = fmaf(oc, f[e], acc[e]);
                }
            }
        }
    }
#pragma unroll
    for (int e = 0; e < V; ++e) red5[((size_t)g * kOVec + vl) * V + e] = acc[e];
    __syncthreads();
    if (g == 0 && v < v1) {
#pragma unroll
        for (int e = 0; e < V; ++e) {
            float t = 0.f;
#pragma unroll
            for (int gg = 0; gg < kOGroups; ++gg) t += red5[((size_t)gg * kOVec + vl) * V + e];
            part[(size_t)v * V + e] = t;
        }
    }
}

template <typename T>
cudaError_t run_attn(const AttnK &k, cudaStream_t s) {
    constexpr int V = Vec<T>::N;
    const int nv = k.d / V;
    // slot in y: the launch order runs through every CTA of slot 0 first, so
    // the CTAs of the count selected slots come first and fill the first wave
    const dim3 gq((k.dh + kQRows - 1) / kQRows, k.H);
    cudaError_t e;
    if (nv <= kAttnThreads) e = launch(attn_q_kernel<T, 1>, gq, dim3(kAttnThreads), 0, s, pdl_enabled(), k);
    else if (nv <= 2 * kAttnThreads) e = launch(attn_q_kernel<T, 2>, gq, dim3(kAttnThreads), 0, s, pdl_enabled(), k);
    else if (nv <= 3 * kAttnThreads) e = launch(attn_q_kernel<T, 3>, gq, dim3(kAttnThreads), 0, s, pdl_enabled(), k);
    else if (nv <= 4 * kAttnThreads) e = launch(attn_q_kernel<T, 4>, gq, dim3(kAttnThreads), 0, s, pdl_enabled(), k);
    else e = launch(attn_q_kernel<T, 8>, gq, dim3(kAttnThreads), 0, s, pdl_enabled(), k);
    if (e != cudaSuccess) return e;
    e = launch(attn_split_kernel<T>, dim3(k.ns, k.H), dim3(kAttnThreads), 0, s, pdl_enabled(), k);
    if (e != cudaSuccess) return e;
    return launch(attn_out_kernel<T>, dim3((nv + kOVec - 1) / kOVec, k.H), dim3(kAttnThreads), 0, s, pdl_enabled(),
                  k);
}

}  // namespace

namespace cs {

// The launch geometry of one call: the split of the positions and where the
// partial rows, queries and split records sit inside the workspace's G x dp
// partial values (H partial rows, the H queries, then per head its splits'
// (max, sum, o)).
struct AttnGeom {
    WsLayout WL;
    int esz, nvk, sc, ns;
    size_t need;
};

static AttnGeom attn_geom(const AttnCall &c) {
    const cs_attn_layer &L = c.layer;
    AttnGeom g;
    g.WL = ws_layout(L.d, 1, 1, 1, device_sm_count());
    g.esz = (int)dtype_size(L.dtype);
    g.nvk = L.d_head * g.esz / 16;
    g.sc = kSplitVec / g.nvk;
    g.ns = (c.seq_len + g.sc - 1) / g.sc;
    g.need = (size_t)L.n_heads * g.WL.dp + (size_t)L.n_heads * L.d_head + (size_t)L.n_heads * g.ns * (L.d_head + 2);
    return g;
}

cs_status attn_check(const AttnCall &c, const char *who) {
    const cs_attn_layer &L = c.layer;
    if (L.dtype != CS_F32 && L.dtype != CS_F16 && L.dtype != CS_BF16) {
        set_error("%s: bad dtype %d", who, (int)L.dtype);
        return CS_ERR_INVALID;
    }
    const int esz = (int)dtype_size(L.dtype), V = 16 / esz;
    const bool dh_ok = L.d_head >= V && L.d_head <= kAttnThreads && (L.d_head & (L.d_head - 1)) == 0;
    auto al16 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; };
    if (L.d < V || L.d % V || L.n_heads < 1 || !dh_ok || !L.w_q || !L.w_o_t || !al16(L.w_q) || !al16(L.w_o_t) ||
        !c.k_cache || !c.v_cache || !al16(c.k_cache) || !al16(c.v_cache)) {
        set_error("%s: d a multiple of %d, d_head a power of two in [%d, %d], and 16-byte aligned weights and "
                  "caches", who, V, V, kAttnThreads);
        return CS_ERR_INVALID;
    }
    if (c.seq_len < 1 || c.seq_len > kAttnMaxS) {
        set_error("%s: seq_len=%d outside [1, %d]", who, c.seq_len, kAttnMaxS);
        return c.seq_len < 1 ? CS_ERR_INVALID : CS_ERR_UNSUPPORTED;
    }
    return CS_OK;
}

cs_status attn_check_ws(const AttnCall &c, const char *who) {
    const cs_attn_layer &L = c.layer;
    const int V = 16 / (int)dtype_size(L.dtype);
    if (!c.ws || (reinterpret_cast<uintptr_t>(c.ws) & 255u)) {
        set_error("%s: workspace is null or not 256-byte aligned", who);
        return CS_ERR_WORKSPACE;
    }
    const AttnGeom g = attn_geom(c);
    if (c.ws_bytes < g.WL.total) {
        set_error("%s: workspace too small: %zu bytes given, %zu needed", who, c.ws_bytes, g.WL.total);
        return CS_ERR_WORKSPACE;
    }
    if (g.need > (size_t)g.WL.G * g.WL.dp || L.d / V > 8 * kAttnThreads) {
        set_error("%s: %d heads of %d over %d positions (d=%d) need more than the %d x %d partial values of "
                  "the workspace, or d is too wide", who, L.n_heads, L.d_head, c.seq_len, L.d, g.WL.G, g.WL.dp);
        return CS_ERR_UNSUPPORTED;
    }
    return CS_OK;
}

cudaError_t attn_launch(const AttnCall &c, const float *x, const int32_t *heads, const int32_t *count, float *y,
                        cudaStream_t s) {
    const cs_attn_layer &L = c.layer;
    const AttnGeom g = attn_geom(c);
    AttnK k;
    k.w_q = static_cast<const uint8_t *>(L.w_q);
    k.w_o_t = static_cast<const uint8_t *>(L.w_o_t);
    k.k = static_cast<const uint8_t *>(c.k_cache);
    k.v = static_cast<const uint8_t *>(c.v_cache);
    k.x = x;
    k.idx = heads;
    k.count = count;
    k.part = reinterpret_cast<float *>(static_cast<char *>(c.ws) + g.WL.part);
    k.qbuf = k.part + (size_t)L.n_heads * g.WL.dp;
    k.split = k.qbuf + (size_t)L.n_heads * L.d_head;
    k.nvk = g.nvk;
    k.sc = g.sc;
    k.ns = g.ns;
    k.err = static_cast<uint32_t *>(c.ws);
    k.d = L.d;
    k.H = L.n_heads;
    k.dh = L.d_head;
    k.S = c.seq_len;
    k.dp = g.WL.dp;
    k.row_bytes = (size_t)L.d * g.esz;
    cudaError_t e = L.dtype == CS_F32 ? run_attn<float>(k, s)
                    : L.dtype == CS_F16 ? run_attn<__half>(k, s)
                                        : run_attn<__nv_bfloat16>(k, s);
    // the reduction adds the partial rows of the selected slots only (the
    // count is read on the device and clamped to the head count)
    if (e == cudaSuccess) e = launch_ffn_reduce(k.part, L.n_heads, 1, L.d, g.WL.dp, nullptr, 1.f, y, s, count);
    return e;
}

}  // namespace cs

extern "C" {

cs_status cs_sparse_attention(const cs_attn_layer *layer, const float *x, const int32_t *heads,
                              const int32_t *count, const void *k_cache, const void *v_cache, int seq_len,
                              float *y, void *ws, size_t ws_bytes, cs_stream_t stream) {
    if (!layer || !x || !heads || !count || !k_cache || !v_cache || !y) {
        set_error("cs_sparse_attention: layer, x, heads, count, k_cache, v_cache and y are required");
        return CS_ERR_INVALID;
    }
    const AttnCall c{*layer, k_cache, v_cache, seq_len, ws, ws_bytes};
    cs_status st = attn_check(c, "cs_sparse_attention");
    if (st != CS_OK) return st;
    if ((reinterpret_cast<uintptr_t>(x) & 15u) || (reinterpret_cast<uintptr_t>(heads) & 3u) ||
        (reinterpret_cast<uintptr_t>(count) & 3u) || (reinterpret_cast<uintptr_t>(y) & 3u) || x == y) {
        set_error("cs_sparse_attention: x 16-byte aligned, heads, count and y 4-byte aligned, and y not "
                  "aliasing x");
        return CS_ERR_INVALID;
    }
    st = attn_check_ws(c, "cs_sparse_attention");
    if (st != CS_OK) return st;
    const cudaError_t e = attn_launch(c, x, heads, count, y, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_sparse_attention");
}

}  // extern "C"
