// Batched gathered FFN on the fifth-generation tensor cores, for dense unions.
//
// Sources: "Contextual Sparsity and Activation Predictors", section "When it
// breaks" (a batch reads the union of its tokens' active sets, which grows
// dense with B); "Contextual Sparsity: Activation-Aware LLM Inference and the
// Deja Vu Paradigm", section "The Prediction Problem" (sparse_mlp_forward: the
// chosen neurons' gate rows and down columns) and section "The SiLU/GELU
// Challenge: TurboSparse" (relu(gate x) * up x).
//
// With U the union list (ascending ids, n = |U|) and X the B token rows, the
// batched FFN is two GEMMs over gathered rows:
//   H  = W_gate[U] X^T            M = n, N = B, K = d   (and W_up[U] X^T)
//   Y^T = W_down^T[U]^T A^T       M = d, N = B, K = n   (A = act(H) per token)
// Operands are fp16 / bf16 (the weights' type); accumulation is fp32 in tensor
// memory.  The fp32 activations enter each GEMM split into two rows of the
// weights' type, v = hi + lo with hi = round(v) and lo = round(v - hi), so
// W.hi + W.lo carries ~16 (bf16) or ~22 (fp16) mantissa bits of v and the
// result stays at fp32-accumulate accuracy.  Row 2b holds hi(v_b) and row
// 2b + 1 lo(v_b), so N is 2B, padded to NP (16, 32 or 64), and B <= 32.
//
// Kernels (one launch each, chained with programmatic dependent launch):
//   tc_split_kernel  X -> XS [NP, dk] (rows 2b: hi(x_b), rows 2b + 1: lo(x_b))
//   tc_gate_kernel   persistent, one CTA per SM over 128-neuron tiles of U:
//                    gathered W_gate (and W_up) rows and XS staged by per-thread
//                    cp.async into 128-byte-swizzled shared memory (K-major),
//                    tcgen05.mma issued by one thread into tensor memory, then
//                    an epilogue that reads the accumulators (tcgen05.ld), adds
//                    the bias, applies relu (times up) and writes AS [NP, kp]
//                    (hi / lo rows again)
//   tc_down_kernel   128-row tiles of d x split-K over U: gathered W_down^T
//                    rows staged as the MN-major operand (64 neurons x 128
//                    columns per stage), AS as the K-major operand; per-split
//                    partial y written for the fixed-order reduce kernel
// The gate kernel runs warp-specialised: seven producer warps copy stages in
// with per-thread cp.async and arrive on the stage's "full" mbarrier when
// their copies land (cp.async.mbarrier.arrive), and one warp issues the MMAs
// and commits them to the stage's "empty" mbarrier, which releases it to the
// producers; no block barrier per stage.  The down kernel refills a stage two
// k-blocks after its MMAs were issued, their completion tracked by
// tcgen05.commit on one mbarrier per stage.  Every wait is bounded: on a
// timeout the kernel records CS_DEVERR_TIMEOUT, stops issuing, lets its copies
// land and frees its tensor memory.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <algorithm>
#include <cstdlib>

#include "cs_internal.cuh"

namespace cs {

namespace {

constexpr int kTcThreads = 256;        // 8 warps; warps 0..3 own TMEM lanes 0..127 in the epilogues
constexpr int kTileM = 128;            // rows of an MMA tile
constexpr int kKB = 64;                // K elements per stage: one 128-byte swizzle row
constexpr int kTileBytes = kTileM * kKB * 2;   // 16 KB per 128 x 64 operand tile
constexpr size_t kTcSmemBudget = 216 * 1024;

struct TcArgs {
    const uint8_t *w_gate, *w_up, *w_down_t;
    const float *bias;
    const float *x;        // [B, d]
    const int32_t *idx;    // union ids, ascending
    const int32_t *count;  // device count
    uint16_t *xs;          // [NP, dk]
    uint16_t *as;          // [NP, kp]
    float *part;           // down GEMM: [P, 2, B, 256] stream-K partials
    float *pieces;         // gate GEMM: [P, 3, 128, NP or 2 NP] partial tile sums
    unsigned *tile_count;  // gate GEMM: [2P] arrivals per tile, zeroed by the split kernel
    uint32_t *err;
    int d, f, B, ldb, dk, kp, dp, splits, stages;
    int act;               // the gate's activation (CS_ACT_*)
};

// ---- element type helpers --------------------------------------------------
template <typename T> struct Tc;
template <> struct Tc<__half> {
    static constexpr bool kBf16 = false;
    __device__ static uint16_t bits(float v) { return __half_as_ushort(__float2half_rn(v)); }
    __device__ static float val(uint16_t b) { return __half2float(__ushort_as_half(b)); }
};
template <> struct Tc<__nv_bfloat16> {
    static constexpr bool kBf16 = true;
    __device__ static uint16_t bits(float v) { return __bfloat16_as_ushort(__float2bfloat16_rn(v)); }
    __device__ static float val(uint16_t b) { return __bfloat162float(__ushort_as_bfloat16(b)); }
};

// ---- tcgen05 / TMEM PTX ------------------------------------------------------
// Shared-memory matrix descriptor: start address, leading and stride byte
// offsets (16-byte units), descriptor version 1, 128-byte swizzle.
__device__ __forceinline__ uint64_t umma_desc(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}
// Instruction descriptor for kind::f16: fp32 accumulator, A/B fp16 or bf16,
// A K-major or MN-major, B K-major, M = 128, N = n.
__device__ __forceinline__ uint32_t umma_idesc(bool bf16, bool a_mn, int n) {
    return (1u << 4) | ((bf16 ? 1u : 0u) << 7) | ((bf16 ? 1u : 0u) << 10) | ((a_mn ? 1u : 0u) << 15) |
           ((uint32_t)(n >> 3) << 17) | ((uint32_t)(kTileM >> 4) << 24);
}
__device__ __forceinline__ void umma(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, bool acc) {
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
        "l"(a), "l"(b), "r"(idesc), "r"(acc ? 1u : 0u));
}
__device__ __forceinline__ void umma_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_addr(bar))
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void fence_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
__device__ __forceinline__ void tmem_alloc(uint32_t *dst, uint32_t cols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_addr(dst)), "r"(cols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_free(uint32_t taddr, uint32_t cols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(cols) : "memory");
}
// 8 consecutive fp32 accumulator columns of this thread's TMEM lane
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void cp16t(uint32_t dst, const void *src) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(dst), "l"(src) : "memory");
}
// offset of 16-byte chunk c of row r in a K-major 128-byte-swizzled tile
__device__ __forceinline__ uint32_t kmaj_off(int r, int c) {
    return (uint32_t)((r >> 3) * 1024 + (r & 7) * 128 + ((c ^ (r & 7)) << 4));
}
// offset of 16-byte chunk c (of 16 * MT along M) of k-row k in the MN-major
// tile: [k / 8][c / 8][k % 8][128 B], swizzled like the K-major rows
template <int MT>
__device__ __forceinline__ uint32_t mnmaj_off(int k, int c) {
    return (uint32_t)((k >> 3) * (2048 * MT) + (c >> 3) * 1024 + (k & 7) * 128 + (((c & 7) ^ (k & 7)) << 4));
}
__device__ __forceinline__ uint32_t tmem_cols(int c) {
    uint32_t n = 32;
    while ((int)n < c) n <<= 1;
    return n;
}

// ---- X -> [hi; lo] rows ------------------------------------------------------
// A thread converts 8 consecutive columns of one token (16-byte stores of
// its hi and lo rows); rows past 2B are zero.  dk = d is a multiple of 64.
template <typename T>
__global__ void tc_split_kernel(const TcArgs a, int np, int ncount) {
    pdl_launch_dependents();
    pdl_wait();
    const int gt = blockIdx.x * blockDim.x + threadIdx.x, gs = gridDim.x * blockDim.x;
    for (int i = gt; i < ncount; i += gs) a.tile_count[i] = 0u;
    const int c8 = a.dk / 8;
    const bool x4 = (reinterpret_cast<uintptr_t>(a.x) & 15) == 0;
    for (int i = gt; i < (np / 2) * c8; i += gs) {
        const int b = i / c8, c0 = (i % c8) * 8;
        uint32_t hi[4] = {0u, 0u, 0u, 0u}, lo[4] = {0u, 0u, 0u, 0u};
        if (b < a.B) {
            float v[8];
            const float *src = a.x + (size_t)b * a.d + c0;
            if (x4) {
                const float4 p = ld_dep(reinterpret_cast<const float4 *>(src));
                const float4 q = ld_dep(reinterpret_cast<const float4 *>(src + 4));
                v[0] = p.x; v[1] = p.y; v[2] = p.z; v[3] = p.w; v[4] = q.x; v[5] = q.y; v[6] = q.z; v[7] = q.w;
            } else {
#pragma unroll
                for (int e = 0; e < 8; ++e) v[e] = ld_dep(src + e);
            }
#pragma unroll
            for (int e = 0; e < 8; e += 2) {
                const uint16_t h0 = Tc<T>::bits(v[e]), h1 = Tc<T>::bits(v[e + 1]);
                const uint16_t l0 = Tc<T>::bits(v[e] - Tc<T>::val(h0)), l1 = Tc<T>::bits(v[e + 1] - Tc<T>::val(h1));
                hi[e / 2] = (uint32_t)h0 | ((uint32_t)h1 << 16);
                lo[e / 2] = (uint32_t)l0 | ((uint32_t)l1 << 16);
            }
        }
        *reinterpret_cast<uint4 *>(a.xs + (size_t)(2 * b) * a.dk + c0) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
        *reinterpret_cast<uint4 *>(a.xs + (size_t)(2 * b + 1) * a.dk + c0) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    }
}

// wait until at most n (0..6) of this thread's copy groups are pending
__device__ __forceinline__ void cp_async_wait_upto(int n) {
    switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    default: cp_async_wait<6>(); break;
    }
}

// bounded wait on a stage barrier; false after the time limit
__device__ __forceinline__ bool stage_wait(uint64_t *bar, uint32_t parity) {
    return mbar_wait(bar, parity, 1000000000ull);
}

// arrive on bar once all of this thread's earlier cp.async copies have landed
// (the barrier's expected count includes this arrival)
__device__ __forceinline__ void cp_async_arrive(uint64_t *bar) {
    asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_addr(bar)) : "memory");
}

// Gate-GEMM warp roles: warps 0 .. kProdWarps-1 copy stages in, warp
// kProdWarps issues the MMAs.
constexpr int kProdWarps = 7;
constexpr int kProd = kProdWarps * 32;

// ---- gate (and up) GEMM + activation, stream-K ----------------------------------
// Work units are (tile t of 128 union neurons, k-block of KS elements of d),
// t-major; CTA c of P takes units [U c / P, U (c+1) / P).  With at most 2P
// tiles a CTA's range touches at most three tiles ("segments"); each segment
// accumulates into its own tensor-memory set and all are read once the last
// MMA is done.  A tile covered by one CTA gets its activation at once; a tile
// shared by several CTAs has each CTA's partial sums written to a piece slot,
// and the CTA whose arrival completes the tile's counter adds the pieces in
// CTA order (so the result does not depend on who arrives last) and applies
// the bias and activation.
constexpr int kGateSegMax = 3;

// sk_start / sk_owner: see the down GEMM below
__device__ __forceinline__ long long sk_start(int c, long long U, int P);
__device__ __forceinline__ int sk_owner(long long u, long long U, int P);

// act = relu(g + bias) or silu(g + bias) (* u), written as the hi / lo rows of AS
template <typename T, bool GLU, int NP>
__device__ __forceinline__ void gate_act_out(const TcArgs &a, const float (&g)[NP], const float (&u)[NP], float bias,
                                             bool live, int p) {
#pragma unroll
    for (int b = 0; b < NP / 2; ++b) {
        if (b < a.B) {
            float act = gate_act(a.act, g[2 * b] + g[2 * b + 1] + bias);
            if (GLU) act *= u[2 * b] + u[2 * b + 1];
            act = live ? act : 0.f;
            const uint16_t hi = Tc<T>::bits(act);
            const uint16_t lo = Tc<T>::bits(act - Tc<T>::val(hi));
            a.as[(size_t)(2 * b) * a.kp + p] = hi;
            a.as[(size_t)(2 * b + 1) * a.kp + p] = lo;
        }
    }
}

template <typename T, bool GLU, int NP, int KS>
__global__ void __launch_bounds__(kTcThreads, 1) tc_gate_kernel(const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[8];    // stage landed: kProd cp.async arrivals
    __shared__ __align__(8) uint64_t empty[8];   // stage's MMAs done: one tcgen05.commit
    __shared__ uint32_t tmem_base;
    __shared__ int s_idx[kGateSegMax * kTileM];
    __shared__ int s_last[kGateSegMax];
    constexpr int KA = KS / kKB;                           // 64-element swizzle atoms per row per stage
    constexpr int kA = GLU ? 2 : 1;                        // weight tiles per stage besides X
    constexpr int kWBytes = KA * kTileBytes;               // one weight tile: [atom][128 rows][128 B]
    constexpr int kXAtom = NP * 128;                       // one X atom: [NP rows][128 B]
    constexpr int kStageBytes = kA * kWBytes + KA * kXAtom;
    constexpr int kSetCols = GLU ? 2 * NP : NP;            // accumulator columns of one segment
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.stages;
    const uint32_t base = smem_addr(dsm);
    const uint32_t sbase = (base + 1023u) & ~1023u;       // 1024-byte aligned stages
    const uint32_t ncols = tmem_cols(kGateSegMax * kSetCols);

    if (warp == 0) tmem_alloc(&tmem_base, ncols);
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], kProd);
            mbar_init(&empty[s], 1);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    pdl_launch_dependents();
    pdl_wait();  // XS, the union list, its count and the zeroed counters come from earlier kernels

    int n = *a.count;
    if (n < 0 || n > a.f) {
        if (tid == 0 && blockIdx.x == 0) atomicOr(a.err, CS_DEVERR_COUNT);
        n = n < 0 ? 0 : a.f;
    }
    const int NT = (n + kTileM - 1) / kTileM;
    const int NKB = a.dk / KS;
    const long long U = (long long)NT * NKB;
    const int P = gridDim.x, c = blockIdx.x;
    const long long u0 = U > 0 ? sk_start(c, U, P) : 0;
    const int Q = U > 0 ? (int)(sk_start(c + 1, U, P) - u0) : 0;
    const int t_first = Q > 0 ? (int)(u0 / NKB) : 0;
    const int kb_first = Q > 0 ? (int)(u0 % NKB) : 0;
    const int nseg = Q > 0 ? (int)((u0 + Q - 1) / NKB) - t_first + 1 : 0;   // <= kGateSegMax
    const int kb_end = Q > 0 ? (int)((u0 + Q - 1) % NKB) + 1 : 0;           // last segment's end

    // ids of this CTA's tiles (positions past n repeat a valid row; their
    // activations are written as 0)
    for (int i = tid; i < nseg * kTileM; i += kTcThreads) {
        const int p = (t_first + i / kTileM) * kTileM + (i % kTileM);
        int j = p < n ? a.idx[p] : (n > 0 ? a.idx[n - 1] : 0);
        if (j < 0 || j >= a.f) {
            atomicOr(a.err, CS_DEVERR_INDEX);
            j = 0;
        }
        s_idx[i] = j;
    }
    __syncthreads();

    const bool bf = Tc<T>::kBf16;
    const uint32_t idesc = umma_idesc(bf, false, NP);
    struct Cur {
        int lt, kb;   // tile relative to t_first, k-block
    };
    auto step = [&](Cur &u) {
        if (++u.kb == NKB) { u.kb = 0; ++u.lt; }
    };
    Cur ic{0, kb_first};   // unit of the next issue

    // Producers (warps 0 .. kProdWarps-1) copy unit q into stage q % S once
    // the MMAs of unit q - S have released it, and arrive on full[q % S] when
    // their copies land; the MMA warp waits for full, issues the stage's MMAs
    // and commits them to empty.  No block barrier per stage: the producers
    // run up to S stages ahead.  The lanes of a warp cover contiguous bytes of
    // a row (KS * 2 bytes per row).
    bool ok = true;
    if (warp < kProdWarps) {
        for (int q = 0; q < Q; ++q) {
            const int sq = q % S;
            // the whole warp stops together if a wait gives up
            if (q >= S && !__all_sync(kFull, stage_wait(&empty[sq], (uint32_t)((q / S - 1) & 1)))) {
                ok = false;
                break;
            }
            const uint32_t st = sbase + (uint32_t)(sq * kStageBytes);
            const size_t koff = (size_t)ic.kb * KS * 2;
            for (int i = tid; i < kTileM * 8 * KA; i += kProd) {
                const int r = i / (8 * KA), ch = i % (8 * KA);
                const uint32_t off = (uint32_t)((ch >> 3) * kTileBytes) + kmaj_off(r, ch & 7);
                const size_t roff = (size_t)s_idx[ic.lt * kTileM + r] * a.ldb + koff + ch * 16;
                cp16t(st + off, a.w_gate + roff);
                if (GLU) cp16t(st + kWBytes + off, a.w_up + roff);
            }
            const uint32_t sx = st + kA * kWBytes;
            for (int i = tid; i < NP * 8 * KA; i += kProd) {
                const int r = i / (8 * KA), ch = i % (8 * KA);
                cp16t(sx + (uint32_t)((ch >> 3) * kXAtom) + kmaj_off(r, ch & 7),
                      reinterpret_cast<const uint8_t *>(a.xs) + (size_t)r * a.dk * 2 + koff + ch * 16);
            }
            cp_async_arrive(&full[sq]);
            step(ic);
        }
    } else {
        // the MMA warp: every lane waits (so the warp stays converged), lane 0
        // issues; the copies were made visible to the tensor cores' async
        // proxy by the proxy fence after the wait
        Cur cc{0, kb_first};   // unit being multiplied
        for (int q = 0; q < Q; ++q) {
            const int sq = q % S;
            if (!__all_sync(kFull, stage_wait(&full[sq], (uint32_t)((q / S) & 1)))) { ok = false; break; }
            fence_async_smem();
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = sbase + (uint32_t)(sq * kStageBytes);
                const uint32_t sx = st + kA * kWBytes;
                const uint32_t acc = tmem + (uint32_t)(cc.lt * kSetCols);
                const bool fresh = q == 0 || cc.kb == 0;
#pragma unroll
                for (int kk = 0; kk < KS / 16; ++kk) {
                    const uint32_t ka = (uint32_t)(kk >> 2), kin = (uint32_t)((kk & 3) * 32);
                    const uint64_t bd = umma_desc(sx + ka * kXAtom + kin, 16, 1024);
                    umma(acc, umma_desc(st + ka * kTileBytes + kin, 16, 1024), bd, idesc, !(fresh && kk == 0));
                    if (GLU)
                        umma(acc + NP, umma_desc(st + kWBytes + ka * kTileBytes + kin, 16, 1024), bd, idesc,
                             !(fresh && kk == 0));
                }
                umma_commit(&empty[sq]);
            }
            __syncwarp();
            step(cc);
        }
    }
    // every decision to stop is taken by the whole block at a barrier; then
    // everyone waits for the last unit's MMAs
    ok = __syncthreads_and(ok);
    if (ok && Q > 0) ok = __syncthreads_and(stage_wait(&empty[(Q - 1) % S], (uint32_t)(((Q - 1) / S) & 1)));
    tc_fence_after();

    // segments: a whole tile -> activation now; a part -> piece slot (c, sg)
    const int r = warp * 32 + lane;  // TMEM lane = tile row (warps 0..3)
    for (int sg = 0; sg < nseg && ok; ++sg) {
        const int t = t_first + sg;
        const bool whole = (sg > 0 || kb_first == 0) && (sg < nseg - 1 || kb_end == NKB);
        if (warp < 4) {
            float g[NP], u[NP];
            const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(sg * kSetCols);
#pragma unroll
            for (int c0 = 0; c0 < NP; c0 += 8) {
                float v[8];
                tmem_ld8(lane_addr + (uint32_t)c0, v);
#pragma unroll
                for (int e = 0; e < 8; ++e) g[c0 + e] = v[e];
                if (GLU) {
                    tmem_ld8(lane_addr + (uint32_t)(NP + c0), v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) u[c0 + e] = v[e];
                }
            }
            const int p = t * kTileM + r;
            if (whole) {
                const float bias = (p < n && a.bias) ? a.bias[s_idx[sg * kTileM + r]] : 0.f;
                gate_act_out<T, GLU, NP>(a, g, u, bias, p < n, p);
            } else {
                float *piece = a.pieces + ((size_t)(c * kGateSegMax + sg) * kTileM + r) * kSetCols;
#pragma unroll
                for (int e = 0; e < NP; ++e) piece[e] = g[e];
                if (GLU) {
#pragma unroll
                    for (int e = 0; e < NP; ++e) piece[NP + e] = u[e];
                }
            }
        }
    }
    __syncthreads();  // pieces written
    if (tid == 0) {
        for (int sg = 0; sg < kGateSegMax; ++sg) s_last[sg] = 0;
        for (int sg = 0; sg < nseg && ok; ++sg) {
            const bool whole = (sg > 0 || kb_first == 0) && (sg < nseg - 1 || kb_end == NKB);
            if (whole) continue;
            const int t = t_first + sg;
            const int c_lo = sk_owner((long long)t * NKB, U, P), c_hi = sk_owner((long long)(t + 1) * NKB - 1, U, P);
            int pieces = 0;
            for (int cc2 = c_lo; cc2 <= c_hi; ++cc2) pieces += sk_start(cc2 + 1, U, P) > sk_start(cc2, U, P);
            __threadfence();
            const unsigned old = atomicAdd(a.tile_count + t, 1u);
            s_last[sg] = old == (unsigned)(pieces - 1);
        }
    }
    __syncthreads();
    for (int sg = 0; sg < nseg && ok; ++sg) {
        if (!s_last[sg]) continue;
        // the last piece of tile t arrived: add all pieces in CTA order
        __threadfence();
        const int t = t_first + sg;
        if (warp < 4) {
            float g[NP], u[NP];
#pragma unroll
            for (int e = 0; e < NP; ++e) { g[e] = 0.f; u[e] = 0.f; }
            const int c_lo = sk_owner((long long)t * NKB, U, P), c_hi = sk_owner((long long)(t + 1) * NKB - 1, U, P);
            for (int cc2 = c_lo; cc2 <= c_hi; ++cc2) {
                const long long st2 = sk_start(cc2, U, P);
                if (sk_start(cc2 + 1, U, P) == st2) continue;
                const int sg2 = t - (int)(st2 / NKB);
                const float *piece = a.pieces + ((size_t)(cc2 * kGateSegMax + sg2) * kTileM + r) * kSetCols;
#pragma unroll
                for (int e = 0; e < NP; ++e) g[e] += __ldcg(piece + e);
                if (GLU) {
#pragma unroll
                    for (int e = 0; e < NP; ++e) u[e] += __ldcg(piece + NP + e);
                }
            }
            const int p = t * kTileM + r;
            const float bias = (p < n && a.bias) ? a.bias[s_idx[sg * kTileM + r]] : 0.f;
            gate_act_out<T, GLU, NP>(a, g, u, bias, p < n, p);
        }
    }
    if (!ok && tid == 0) atomicOr(a.err, CS_DEVERR_TIMEOUT);
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_free(tmem, ncols);
    }
}

// ---- down GEMM, stream-K -> partial y per (CTA, column group) ------------------
// Work units are (column group g of 128 * MT output rows, k-block of 64 union
// neurons), g-major; CTA c of P takes units [U c / P, U (c+1) / P), so every
// CTA gets the same amount of work.  Its range covers at most two column
// groups (when there are at most P groups); for each it writes the partial
// sum of its k-blocks to slot (c, 0) or (c, 1).  tc_reduce_kernel adds, for
// every column, the slots of the CTAs that cover its group, in CTA order.
__device__ __forceinline__ long long sk_start(int c, long long U, int P) { return U * c / P; }
// the CTA whose unit range holds unit u (0 <= u < U)
__device__ __forceinline__ int sk_owner(long long u, long long U, int P) {
    int c = (int)(((u + 1) * P - 1) / U);
    c = c < 0 ? 0 : (c >= P ? P - 1 : c);
    while (c + 1 < P && sk_start(c + 1, U, P) <= u) ++c;
    while (c > 0 && sk_start(c, U, P) > u) --c;
    return c;
}

template <typename T, int NP, int MT>
__global__ void __launch_bounds__(kTcThreads, 1) tc_down_kernel(const TcArgs a) {
    extern __shared__ __align__(1024) uint8_t dsm[];
    __shared__ __align__(8) uint64_t full[8];    // stage landed: kProd cp.async arrivals
    __shared__ __align__(8) uint64_t empty[8];   // stage's MMAs done: one tcgen05.commit
    __shared__ uint32_t tmem_base;
    constexpr int kCols = kTileM * MT;                      // output rows of a column group
    constexpr int kWBytes = MT * kTileBytes;                // 64 rows x kCols columns
    constexpr int kStageBytes = kWBytes + NP * 128;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = a.stages;
    const uint32_t base = smem_addr(dsm);
    const uint32_t sbase = (base + 1023u) & ~1023u;
    constexpr int kSegCols = MT * NP;                       // accumulator columns of one segment
    const uint32_t ncols = tmem_cols(2 * kSegCols);          // two segments, read at the end

    if (warp == 0) tmem_alloc(&tmem_base, ncols);
    if (tid == 0) {
        for (int s = 0; s < S; ++s) {
            mbar_init(&full[s], kProd);
            mbar_init(&empty[s], 1);
        }
        mbar_fence_init();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base;

    pdl_launch_dependents();
    pdl_wait();  // AS comes from the gate kernel

    int n = ld_dep(a.count);
    if (n < 0 || n > a.f) n = n < 0 ? 0 : a.f;
    const int NG = (a.d + kCols - 1) / kCols;
    const int NKB = (n + kKB - 1) / kKB;
    const long long U = (long long)NG * NKB;
    const int P = gridDim.x, c = blockIdx.x;
    const long long u0 = U > 0 ? sk_start(c, U, P) : 0;
    const int Q = U > 0 ? (int)(sk_start(c + 1, U, P) - u0) : 0;
    const bool bf = Tc<T>::kBf16;
    const uint32_t idesc = umma_idesc(bf, true, NP);
    const int last = n > 0 ? ld_dep(a.idx + n - 1) : 0;
    // unit cursors (column group, k-block): one division here, then +1 steps
    struct Cur {
        int g, kb;
    };
    const Cur first = NKB > 0 ? Cur{(int)(u0 / NKB), (int)(u0 % NKB)} : Cur{0, 0};
    auto step = [&](Cur &u) {
        if (++u.kb == NKB) { u.kb = 0; ++u.g; }
    };
    // A stage row is 16 * MT chunks covered by consecutive producer lanes.
    // Warp-specialised like the gate kernel: producers (warps 0 .. 6) copy
    // unit q into stage q % S once the MMAs of unit q - S released it and
    // arrive on full[q % S] when their copies land; warp 7 issues the MMAs
    // and commits them to empty[q % S].
    constexpr int kCh = 16 * MT;
    constexpr int kPer = (kKB * kCh + kProd - 1) / kProd;   // chunks per producer thread and stage
    bool ok = true;
    int seg = 0;           // slot (and accumulator set) of the last column group
    if (warp < kProdWarps) {
        // the row ids of a stage's chunks are loaded one stage ahead, so no
        // copy waits for its id
        int jcur[kPer], jnext[kPer];
        auto row_ids = [&](bool live, int kb, int (&j)[kPer]) {
#pragma unroll
            for (int it = 0; it < kPer; ++it) {
                const int p = kb * kKB + (tid + it * kProd) / kCh;
                j[it] = (live && p < n) ? ld_dep(a.idx + p) : last;
            }
        };
        Cur ic = first, pc = first;   // unit of the next issue, and the one after it
        step(pc);
        row_ids(Q > 0, ic.kb, jcur);
        for (int q = 0; q < Q; ++q) {
            const int sq = q % S;
            if (q >= S && !__all_sync(kFull, stage_wait(&empty[sq], (uint32_t)((q / S - 1) & 1)))) {
                ok = false;
                break;
            }
            const int m0 = ic.g * kCols;
            const uint32_t st = sbase + (uint32_t)(sq * kStageBytes);
            // 64 gathered rows x kCols columns (256 * MT bytes) of W_down^T
#pragma unroll
            for (int it = 0; it < kPer; ++it) {
                const int i = tid + it * kProd;
                if (i >= kKB * kCh) break;
                const int k = i / kCh, ch = i % kCh;
                int j = jcur[it];
                j = (j >= 0 && j < a.f) ? j : 0;
                const int col = m0 + ch * 8;
                const uint32_t dst = st + mnmaj_off<MT>(k, ch);
                if (col < a.d) {
                    cp16t(dst, a.w_down_t + (size_t)j * a.ldb + (size_t)col * 2);
                } else {
                    asm volatile("st.shared.v4.u32 [%0], {%1, %1, %1, %1};" ::"r"(dst), "r"(0u) : "memory");
                }
            }
            const uint32_t sx = st + kWBytes;
            const size_t koff = (size_t)ic.kb * kKB * 2;
            for (int i = tid; i < NP * 8; i += kProd) {
                const int r = i >> 3, ch = i & 7;
                cp16t(sx + kmaj_off(r, ch), reinterpret_cast<const uint8_t *>(a.as) + (size_t)r * a.kp * 2 + koff + ch * 16);
            }
            // plain shared stores (the zero columns) are ordered before the
            // arrival by this fence; the copies by the arrival itself
            fence_async_smem();
            cp_async_arrive(&full[sq]);
            row_ids(q + 1 < Q, pc.kb, jnext);
#pragma unroll
            for (int it = 0; it < kPer; ++it) jcur[it] = jnext[it];
            step(ic);
            step(pc);
        }
    } else {
        Cur cc = first;        // unit being multiplied
        bool fresh = true;     // the next MMA starts a new accumulation
        for (int q = 0; q < Q; ++q) {
            const int sq = q % S;
            if (!__all_sync(kFull, stage_wait(&full[sq], (uint32_t)((q / S) & 1)))) { ok = false; break; }
            fence_async_smem();
            tc_fence_after();
            if (lane == 0) {
                const uint32_t st = sbase + (uint32_t)(sq * kStageBytes);
                const uint32_t sx = st + kWBytes;
                const uint32_t acc = tmem + (uint32_t)(seg * kSegCols);
                constexpr uint32_t kSbo = 2048 * MT;   // bytes between 8-row k groups
#pragma unroll
                for (int kk = 0; kk < kKB / 16; ++kk) {
                    const uint64_t bd = umma_desc(sx + kk * 32, 16, 1024);
#pragma unroll
                    for (int t = 0; t < MT; ++t)
                        umma(acc + (uint32_t)(t * NP), umma_desc(st + t * 2048 + kk * 2 * kSbo, 1024, kSbo), bd,
                             idesc, !(fresh && kk == 0));
                }
                umma_commit(&empty[sq]);
            }
            __syncwarp();
            fresh = false;
            // a range covers at most two column groups: the second accumulates
            // into the second set, so no MMA has to finish before it starts
            if (cc.kb == NKB - 1 && q < Q - 1) {
                ++seg;
                fresh = true;
            }
            step(cc);
        }
    }
    // the number of column groups the range covers (the MMA warp's seg)
    {
        __shared__ int s_seg;
        if (tid == kProd) s_seg = seg;
        ok = __syncthreads_and(ok);
        seg = s_seg;
    }
    if (ok && Q > 0) ok = __syncthreads_and(stage_wait(&empty[(Q - 1) % S], (uint32_t)(((Q - 1) / S) & 1)));
    tc_fence_after();
    // every segment's partial sums to its slot, once the last MMAs are done
    if (ok && Q > 0 && warp < 4) {
        for (int sg = 0; sg <= seg; ++sg) {
            const size_t slot = (size_t)(c * 2 + sg) * a.B;
#pragma unroll
            for (int t = 0; t < MT; ++t) {
                const int r = t * kTileM + warp * 32 + lane;
                float y[NP];
                const uint32_t lane_addr =
                    tmem + ((uint32_t)(warp * 32) << 16) + (uint32_t)(sg * kSegCols + t * NP);
#pragma unroll
                for (int c0 = 0; c0 < NP; c0 += 8) {
                    float v[8];
                    tmem_ld8(lane_addr + (uint32_t)c0, v);
#pragma unroll
                    for (int e = 0; e < 8; ++e) y[c0 + e] = v[e];
                }
#pragma unroll
                for (int b = 0; b < NP / 2; ++b)
                    if (b < a.B) a.part[(slot + b) * kCols + r] = y[2 * b] + y[2 * b + 1];
            }
        }
    }
    if (!ok && tid == 0) atomicOr(a.err, CS_DEVERR_TIMEOUT);
    cp_async_wait<0>();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_free(tmem, ncols);
    }
}

// y[b, m] = (resid[b, m] + scale *) the stream-K partials of m's column
// group, in CTA order
template <int MT>
__global__ void __launch_bounds__(256) tc_reduce_kernel(const TcArgs a, int P, const float *resid, float scale,
                                                       float *y) {
    constexpr int kCols = kTileM * MT;
    static_assert(kCols == 256, "a CTA's 256 outputs form one column group");
    constexpr int kMaxSlots = 256;      // partial slots per group: at most the CTAs (the path needs G <= 256)
    __shared__ int s_slot[kMaxSlots];   // the group's partial slots, in CTA order
    __shared__ int s_n;
    pdl_launch_dependents();
    pdl_wait();
    // a CTA's 256 outputs lie in one column group (kCols = 256): its slots
    // are found once, by one warp, instead of by every thread
    const int g = blockIdx.x * 256 / kCols, b = blockIdx.y;
    if (threadIdx.x < 32) {
        int n = *a.count;
        if (n < 0 || n > a.f) n = n < 0 ? 0 : a.f;
        const int NG = (a.d + kCols - 1) / kCols;
        const int NKB = (n + kKB - 1) / kKB;
        const long long U = (long long)NG * NKB;
        int cnt = 0;
        if (U > 0) {
            const int c_lo = sk_owner((long long)g * NKB, U, P), c_hi = sk_owner((long long)(g + 1) * NKB - 1, U, P);
            for (int c0 = c_lo; c0 <= c_hi; c0 += 32) {
                const int c = c0 + (int)threadIdx.x;
                bool has = false;
                int slot = 0;
                if (c <= c_hi) {
                    const long long st = sk_start(c, U, P);
                    has = sk_start(c + 1, U, P) != st;   // an empty range wrote no slot
                    slot = c * 2 + (g - (int)(st / NKB));
                }
                const unsigned m = __ballot_sync(kFull, has);
                if (has) {
                    const int pos = cnt + __popc(m & ((1u << threadIdx.x) - 1u));
                    if (pos < kMaxSlots) s_slot[pos] = slot;
                }
                cnt += __popc(m);
            }
        }
        if (threadIdx.x == 0) s_n = cnt < kMaxSlots ? cnt : kMaxSlots;
    }
    __syncthreads();
    const int m = blockIdx.x * 256 + threadIdx.x;
    if (m >= a.d) return;
    float sum = 0.f;
    const int ns = s_n;
    for (int i = 0; i < ns; ++i)
        sum += __ldcg(a.part + ((size_t)s_slot[i] * a.B + b) * kCols + (m - g * kCols));
    const size_t o = (size_t)b * a.d + m;
    y[o] = resid ? fmaf(scale, sum, resid[o]) : sum;
}

template <typename T, int NP>
cudaError_t run_tc(const FfnArgs &f, cudaStream_t s) {
    TcArgs a = {};
    a.w_gate = static_cast<const uint8_t *>(f.w_gate);
    a.w_up = static_cast<const uint8_t *>(f.w_up);
    a.w_down_t = static_cast<const uint8_t *>(f.w_down_t);
    a.bias = f.bias;
    a.act = f.act;
    a.x = f.x;
    a.idx = f.idx;
    a.count = f.count;
    a.xs = static_cast<uint16_t *>(f.tc_x);
    a.as = static_cast<uint16_t *>(f.tc_a);
    {
        // the gate GEMM's piece slots and tile counters follow AS in the workspace
        char *after_as = static_cast<char *>(f.tc_a) + tc_a_bytes(f.f, f.B);
        a.pieces = reinterpret_cast<float *>(after_as);
        a.tile_count = reinterpret_cast<unsigned *>(after_as + tc_pieces_bytes(f.B, f.G));
    }
    a.part = f.part;
    a.err = f.err;
    a.d = f.d;
    a.f = f.f;
    a.B = f.B;
    a.ldb = f.ld * 2;
    a.dk = f.d;  // d is a multiple of kKB on this path
    a.kp = tc_act_pitch(f.f);
    a.dp = f.dp;
    const int sms = f.G > 0 ? f.G : 1;
    const bool glu = f.w_up != nullptr;

    // 1. X -> [hi; lo]
    a.stages = 0;
    cudaError_t e = launch(tc_split_kernel<T>, dim3(std::min(4 * sms, (NP / 2 * a.dk / 8 + 255) / 256)), dim3(256), 0,
                           s, pdl_enabled(), a, NP, 2 * sms);
    if (e != cudaSuccess) return e;

    // 2. gate (and up) GEMM + activation, stream-K over (128-neuron tile,
    //    k-block) units
    {
        // gate-only layers: 256 K-elements (512 bytes of each gathered row) per
        // stage, two stages; measured 3.8% faster than 128 with four stages at
        // B = 32 and equal at B = 4 .. 16
        const bool ks256 = !glu && a.dk % 256 == 0;
        const bool ks128 = !glu && !ks256 && a.dk % 128 == 0;
        const int stage = ks256 ? 4 * (kTileBytes + NP * 128)
                        : ks128 ? 2 * (kTileBytes + NP * 128) : (glu ? 2 : 1) * kTileBytes + NP * 128;
        a.stages = std::min(8, (int)(kTcSmemBudget / stage));
        const size_t smem = (size_t)a.stages * stage + 1024;
        auto fn = ks256 ? tc_gate_kernel<T, false, NP, 256>
                        : ks128 ? tc_gate_kernel<T, false, NP, 128>
                                : (glu ? tc_gate_kernel<T, true, NP, 64> : tc_gate_kernel<T, false, NP, 64>);
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = launch(fn, dim3(sms), dim3(kTcThreads), smem, s, pdl_enabled(), a);
        if (e != cudaSuccess) return e;
    }
    // 3. down GEMM, stream-K over (256-row column group, 64-neuron k-block)
    //    units: every CTA the same share; 512 bytes of each gathered row per stage
    constexpr int MT = 2;
    {
        const int stage = MT * kTileBytes + NP * 128;
        a.stages = std::min(8, (int)(kTcSmemBudget / stage));
        const size_t smem = (size_t)a.stages * stage + 1024;
        auto fn = tc_down_kernel<T, NP, MT>;
        e = cudaFuncSetAttribute(fn, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        e = launch(fn, dim3(sms), dim3(kTcThreads), smem, s, pdl_enabled(), a);
        if (e != cudaSuccess) return e;
    }
    // 4. the partials of each column, in CTA order (+ residual epilogue)
    return launch(tc_reduce_kernel<MT>, dim3((f.d + 255) / 256, f.B), dim3(256), 0, s, pdl_enabled(), a, sms,
                  f.resid, f.scale, f.y);
}

template <typename T>
cudaError_t run_tc_np(const FfnArgs &f, cudaStream_t s) {
    const int n2 = 2 * f.B;
    if (n2 <= 16) return run_tc<T, 16>(f, s);
    if (n2 <= 32) return run_tc<T, 32>(f, s);
    return run_tc<T, 64>(f, s);
}

}  // namespace

int tc_act_pitch(int f) { return (f + kTileM - 1) / kTileM * kTileM; }

static int tc_np(int B) { return 2 * B <= 16 ? 16 : (2 * B <= 32 ? 32 : 64); }

size_t tc_x_bytes(int d, int B) { return align256((size_t)tc_np(B) * d * 2); }
size_t tc_a_bytes(int f, int B) { return align256((size_t)tc_np(B) * tc_act_pitch(f) * 2); }
// [P, 3 segments, 128 rows, 2 NP] fp32 (gate and up halves)
size_t tc_pieces_bytes(int B, int P) { return align256((size_t)P * kGateSegMax * kTileM * 2 * tc_np(B) * 4); }

size_t tc_workspace_bytes(int d, int f, int B) {
    if (B < 2 || B > kTcMaxB) return 0;
    int sms = device_sm_count();
    sms = sms < 1 ? 1 : sms;
    return tc_x_bytes(d, B) + tc_a_bytes(f, B) + tc_pieces_bytes(B, sms) + align256((size_t)2 * sms * 4);
}

bool tc_path_applies(const FfnArgs &f) {
    if (!f.tc_x || !f.tc_a || f.preact) return false;
    if (f.dtype == CS_F32 || f.B < tc_min_batch() || f.B > kTcMaxB) return false;
    if (f.d % kKB != 0 || (f.ld * 2) % 16 != 0) return false;
    // down GEMM: stream-K partials (2 slots x 256 columns per CTA and token)
    // fit the workspace's partial-sum region, and a CTA's range spans <= 2
    // column groups; gate GEMM: at most 2P tiles, so a range spans <= 3 tiles
    if (f.d < 512 || (f.d + 255) / 256 > f.G || f.G > 256) return false;
    if ((f.f + kTileM - 1) / kTileM > 2 * f.G) return false;
    return true;
}

int tc_min_batch() {
    static const int v = [] {
        const char *e = getenv("CS_TC_MIN_B");
        const int b = e ? atoi(e) : kTcDefaultMinB;
        return b < 2 ? 2 : b;
    }();
    return v;
}

cudaError_t launch_ffn_tc(const FfnArgs &f, cudaStream_t s) {
    return f.dtype == CS_F16 ? run_tc_np<__half>(f, s) : run_tc_np<__nv_bfloat16>(f, s);
}

}  // namespace cs
