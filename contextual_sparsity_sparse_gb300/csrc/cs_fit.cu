// Fitting a predictor's up map to its layer (setup, not on the decode path).
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "The Prediction Problem" (a small predictor trained
// to reproduce which neurons the layer activates); "Contextual Sparsity and
// Activation Predictors", section "Precision, recall, and which error hurts"
// (the predictor's recall decides the quality).
//
// With P_down fixed, P_up is the ridge regression of the gate pre-activations
// onto the bottleneck features over N calibration inputs:
//     P_up = G^T H (H^T H + lam I)^-1,  H = [relu(P_down x_n)]_n  (N x r),
//                                       G = [W_gate x_n + b]_n    (N x f).
//   1. H and G: the streaming GEMV kernels over the N tokens (fp32).
//   2. H^T H and H^T G: a tiled product with fp32 inputs and fp64 sums.
//   3. H^T H + lam I = L L^T: one CTA, right-looking Cholesky in fp64.
//   4. For each neuron j, (L L^T) p_j = (H^T G)[:, j]: one warp per neuron,
//      forward then backward substitution in shared memory, fp64.
//   5. P_up in the predictor's dtype.
// The call waits for its stream at the end (it reports a matrix that is not
// positive definite), so it belongs to setup, not to a captured graph.
#include <algorithm>
#include <type_traits>

#include "cs_internal.cuh"

using namespace cs;

namespace {

constexpr int kGT = 64;     // output tile of the Gram products
constexpr int kGK = 16;     // tokens per step
constexpr int kFitMaxR = 2048;
constexpr uint32_t kNotSpd = 0x100u;   // private flag in the scratch error word

// C[i, j] = sum_n X[n, i] * Y[n, j] for i < M, j < Nc: X [N, ldx], Y [N, ldy]
// fp32, fp64 sums; stored at C[i * ldc + j], or C[j * ldc + i] with trans.
// 16 x 16 threads, each a 4 x 4 block of the 64 x 64 tile.
__global__ void __launch_bounds__(256) gram_kernel(const float *__restrict__ X, int ldx, const float *__restrict__ Y,
                                                   int ldy, int N, int M, int Nc, double *__restrict__ C, int ldc,
                                                   bool trans) {
    __shared__ float xs[kGK][kGT], ys[kGK][kGT];
    const int i0 = blockIdx.y * kGT, j0 = blockIdx.x * kGT;
    const int tid = threadIdx.x, ti = tid >> 4, tj = tid & 15;
    double acc[4][4];
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) acc[p][q] = 0.0;
    for (int n0 = 0; n0 < N; n0 += kGK) {
        for (int e = tid; e < kGK * kGT; e += 256) {
            const int kk = e / kGT, c = e % kGT, n = n0 + kk;
            xs[kk][c] = (n < N && i0 + c < M) ? X[(size_t)n * ldx + i0 + c] : 0.f;
            ys[kk][c] = (n < N && j0 + c < Nc) ? Y[(size_t)n * ldy + j0 + c] : 0.f;
        }
        __syncthreads();
#pragma unroll 4
        for (int kk = 0; kk < kGK; ++kk) {
            double a[4], b[4];
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                a[q] = xs[kk][ti * 4 + q];
                b[q] = ys[kk][tj * 4 + q];
            }
#pragma unroll
            for (int p = 0; p < 4; ++p)
#pragma unroll
                for (int q = 0; q < 4; ++q) acc[p][q] = fma(a[p], b[q], acc[p][q]);
        }
        __syncthreads();
    }
#pragma unroll
    for (int p = 0; p < 4; ++p)
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const int i = i0 + ti * 4 + p, j = j0 + tj * 4 + q;
            if (i < M && j < Nc) C[trans ? (size_t)j * ldc + i : (size_t)i * ldc + j] = acc[p][q];
        }
}

// A <- A + lam I, then its lower triangle becomes L with A = L L^T (row-major
// r x r, in place).  A non-positive pivot sets kNotSpd and continues with 1.
__global__ void __launch_bounds__(1024) cholesky_kernel(double *__restrict__ A, int r, double lam,
                                                        uint32_t *__restrict__ err) {
    __shared__ double piv;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5, nw = blockDim.x >> 5;
    for (int i = tid; i < r; i += blockDim.x) A[(size_t)i * r + i] += lam;
    __syncthreads();
    for (int k = 0; k < r; ++k) {
        if (tid == 0) {
            double v = A[(size_t)k * r + k];
            if (!(v > 0.0)) {
                atomicOr(err, kNotSpd);
                v = 1.0;
            }
            v = sqrt(v);
            A[(size_t)k * r + k] = v;
            piv = v;
        }
        __syncthreads();
        const double p = piv;
        for (int i = k + 1 + tid; i < r; i += blockDim.x) A[(size_t)i * r + k] /= p;
        __syncthreads();
        // trailing update of the lower triangle: warp per row, lanes along it
        for (int i = k + 1 + warp; i < r; i += nw) {
            const double lik = A[(size_t)i * r + k];
            for (int j = k + 1 + lane; j <= i; j += 32) A[(size_t)i * r + j] -= lik * A[(size_t)j * r + k];
        }
        __syncthreads();
    }
}

__device__ __forceinline__ double warp_sum_d(double v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(kFull, v, o);
    return v;
}

// For each row j of B [f, r]: solve (L L^T) p = B[j, :] in place.  One warp
// per row; its right-hand side lives in shared memory meanwhile.
constexpr int kSolveWarps = 8;
__global__ void __launch_bounds__(kSolveWarps * 32) chol_solve_kernel(const double *__restrict__ L, int r,
                                                                      double *__restrict__ B, int f) {
    extern __shared__ double ysm[];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    double *y = ysm + (size_t)warp * r;
    for (int j = blockIdx.x * kSolveWarps + warp; j < f; j += gridDim.x * kSolveWarps) {
        double *b = B + (size_t)j * r;
        for (int i = lane; i < r; i += 32) y[i] = b[i];
        __syncwarp();
        // L y = b
        for (int i = 0; i < r; ++i) {
            const double *Li = L + (size_t)i * r;
            double s = 0.0;
            for (int k = lane; k < i; k += 32) s = fma(Li[k], y[k], s);
            s = warp_sum_d(s);
            const double yi = (y[i] - s) / Li[i];
            __syncwarp();
            if (lane == 0) y[i] = yi;
            __syncwarp();
        }
        // L^T p = y, eliminating one unknown at a time from the top rows
        for (int i = r - 1; i >= 0; --i) {
            const double *Li = L + (size_t)i * r;
            const double xi = y[i] / Li[i];
            __syncwarp();
            if (lane == 0) y[i] = xi;
            for (int k = lane; k < i; k += 32) y[k] = fma(-Li[k], xi, y[k]);
            __syncwarp();
        }
        for (int i = lane; i < r; i += 32) b[i] = y[i];
        __syncwarp();
    }
}

template <typename T>
__global__ void to_storage_kernel(const double *__restrict__ src, int rows, int cols, T *__restrict__ dst, int ld) {
    const size_t n = (size_t)rows * cols;
    for (size_t e = (size_t)blockIdx.x * blockDim.x + threadIdx.x; e < n; e += (size_t)gridDim.x * blockDim.x) {
        const size_t i = e / cols, c = e % cols;
        const float v = (float)src[e];
        if constexpr (sizeof(T) == 4) dst[i * ld + c] = v;
        else if constexpr (std::is_same<T, __half>::value) dst[i * ld + c] = __float2half_rn(v);
        else dst[i * ld + c] = __float2bfloat16_rn(v);
    }
}

struct FitLayout {
    size_t err, h, g, a, b, total;
};

FitLayout fit_layout(int f, int r, int N) {
    FitLayout L;
    size_t off = 0;
    L.err = off; off += 256;
    L.h = off;   off += align256(sizeof(float) * (size_t)N * r);
    L.g = off;   off += align256(sizeof(float) * (size_t)N * f);
    L.a = off;   off += align256(sizeof(double) * (size_t)r * r);
    L.b = off;   off += align256(sizeof(double) * (size_t)f * r);
    L.total = off;
    return L;
}

}  // namespace

extern "C" {

size_t cs_fit_scratch_size(int d, int f, int r, int N) {
    if (d < 1 || f < 1 || r < 1 || N < 1) return 0;
    return fit_layout(f, r, N).total;
}

cs_status cs_fit_predictor(const cs_ffn_layer *layer, cs_predictor *pred, const float *X, int N, double lambda,
                           void *scratch, size_t scratch_bytes, cs_stream_t stream) {
    if (!layer || !pred || !X || N < 1 || !(lambda >= 0.0) || (reinterpret_cast<uintptr_t>(X) & 15u)) {
        set_error("cs_fit_predictor: layer, pred and X (16-byte aligned) are required, N >= 1, lambda >= 0");
        return CS_ERR_INVALID;
    }
    const cs_ffn_layer &Ly = *layer;
    const int d = Ly.d, f = Ly.f, r = pred->r;
    const int ld = Ly.ld ? Ly.ld : Ly.d;
    const int ldd = pred->ld_down ? pred->ld_down : pred->d, ldu = pred->ld_up ? pred->ld_up : pred->r;
    const bool dt_ok = (Ly.dtype == CS_F32 || Ly.dtype == CS_F16 || Ly.dtype == CS_BF16) &&
                       (pred->dtype == CS_F32 || pred->dtype == CS_F16 || pred->dtype == CS_BF16);
    if (!dt_ok || d < 1 || f < 1 || r < 1 || pred->d != d || pred->f != f || ld < d || ldd < d || ldu < r ||
        (ld * dtype_size(Ly.dtype)) % 16 || (ldd * dtype_size(pred->dtype)) % 16 || !Ly.w_gate || !pred->p_down ||
        !pred->p_up || (reinterpret_cast<uintptr_t>(Ly.w_gate) & 15u) ||
        (reinterpret_cast<uintptr_t>(pred->p_down) & 15u) || (reinterpret_cast<uintptr_t>(pred->p_up) & 3u) ||
        (reinterpret_cast<uintptr_t>(Ly.bias) & 3u)) {
        set_error("cs_fit_predictor: the predictor must match the layer (d, f), with valid strides and pointers");
        return CS_ERR_INVALID;
    }
    // (N <= 65535 keeps the GEMV's token-group grid dimension in range)
    if (r > kFitMaxR || N > 65535 || (long long)N * std::max(f, r) > (1ll << 31)) {
        set_error("cs_fit_predictor: r=%d or N=%d beyond the supported maximum (r <= %d, N <= 65535, "
                  "N * f < 2^31)", r, N, kFitMaxR);
        return CS_ERR_UNSUPPORTED;
    }
    const FitLayout FL = fit_layout(f, r, N);
    if (!scratch || (reinterpret_cast<uintptr_t>(scratch) & 255u) || scratch_bytes < FL.total) {
        set_error("cs_fit_predictor: scratch null, misaligned or smaller than cs_fit_scratch_size (%zu bytes)",
                  FL.total);
        return CS_ERR_WORKSPACE;
    }
    cudaStream_t s = (cudaStream_t)stream;
    char *sc = static_cast<char *>(scratch);
    uint32_t *err = reinterpret_cast<uint32_t *>(sc + FL.err);
    float *H = reinterpret_cast<float *>(sc + FL.h);
    float *G = reinterpret_cast<float *>(sc + FL.g);
    double *A = reinterpret_cast<double *>(sc + FL.a);
    double *Bm = reinterpret_cast<double *>(sc + FL.b);
    cudaError_t e = cudaMemsetAsync(err, 0, 4, s);
    // 1. features and targets
    if (e == cudaSuccess)
        e = launch_gemv_batch(pred->dtype, pred->p_down, ldd * (int)dtype_size(pred->dtype), d, r, X, N, H, nullptr,
                              1, err, s);
    if (e == cudaSuccess)
        e = launch_gemv_batch(Ly.dtype, Ly.w_gate, ld * (int)dtype_size(Ly.dtype), d, f, X, N, G, Ly.bias, 2, err,
                              s);
    if (e != cudaSuccess) return cuda_fail(e, "cs_fit_predictor(features)");
    // 2. H^T H [r, r] and (H^T G)^T [f, r]
    gram_kernel<<<dim3((r + kGT - 1) / kGT, (r + kGT - 1) / kGT), 256, 0, s>>>(H, r, H, r, N, r, r, A, r, false);
    gram_kernel<<<dim3((f + kGT - 1) / kGT, (r + kGT - 1) / kGT), 256, 0, s>>>(H, r, G, f, N, r, f, Bm, r, true);
    // 3. Cholesky of H^T H + lam I
    cholesky_kernel<<<1, 1024, 0, s>>>(A, r, lambda, err);
    // 4. one solve per neuron
    const size_t smem = sizeof(double) * (size_t)kSolveWarps * r;
    e = cudaFuncSetAttribute(chol_solve_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return cuda_fail(e, "cs_fit_predictor(solve attribute)");
    const int sms = std::max(1, device_sm_count());
    const int grid = std::min((f + kSolveWarps - 1) / kSolveWarps, 8 * sms);
    chol_solve_kernel<<<grid, kSolveWarps * 32, smem, s>>>(A, r, Bm, f);
    // 5. P_up in the predictor's dtype
    const int cgrid = 4 * sms;
    void *pu = const_cast<void *>(pred->p_up);
    if (pred->dtype == CS_F32) to_storage_kernel<float><<<cgrid, 256, 0, s>>>(Bm, f, r, static_cast<float *>(pu), ldu);
    else if (pred->dtype == CS_F16) to_storage_kernel<__half><<<cgrid, 256, 0, s>>>(Bm, f, r, static_cast<__half *>(pu), ldu);
    else to_storage_kernel<__nv_bfloat16><<<cgrid, 256, 0, s>>>(Bm, f, r, static_cast<__nv_bfloat16 *>(pu), ldu);
    e = cudaGetLastError();
    if (e != cudaSuccess) return cuda_fail(e, "cs_fit_predictor(launch)");
    uint32_t flags = 0;
    e = cudaMemcpyAsync(&flags, err, 4, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "cs_fit_predictor");
    if (flags & kNotSpd) {
        set_error("cs_fit_predictor: H^T H + lambda I is not positive definite; raise lambda or N");
        return CS_ERR_INVALID;
    }
    if (flags) {
        set_error("cs_fit_predictor: a kernel reported error bits 0x%x", flags);
        return CS_ERR_CUDA;
    }
    return CS_OK;
}

}  // extern "C"
