// Frequency-sorted neuron layout (setup, not on the decode path).
//
// Sources: "Contextual Sparsity: Activation-Aware LLM Inference and the Deja
// Vu Paradigm", section "Kernel-Level Implementation" (neurons pre-sorted by
// how often they fire, so the rows that are read together sit together);
// "Contextual Sparsity and Activation Predictors", section "Static locality:
// hot and cold neurons" (a small set of neurons fires for most inputs).
//
// With the rows sorted hottest first, a selection with a hot prefix of H
// neurons takes rows 0 .. H-1 always and predicts only the tail, so the
// predictor's up map shrinks to f - H rows.  cs_permute_rows reorders the
// rows of one matrix (one CTA per destination row, 16-byte copies when every
// address and the row length allow, element copies otherwise);
// cs_hot_order computes the order on the host.
#include <algorithm>
#include <cmath>
#include <numeric>
#include <vector>

#include "cs_internal.cuh"

namespace {

constexpr int kPermThreads = 128;

__global__ void __launch_bounds__(kPermThreads)
permute_rows_kernel(const uint8_t *__restrict__ src, int src_rows, size_t src_pitch,
                    const int32_t *__restrict__ perm, int rows, uint8_t *__restrict__ dst,
                    size_t dst_pitch, int row_bytes, int esz, bool vec16) {
    for (int i = blockIdx.x; i < rows; i += gridDim.x) {
        const int p = __ldg(perm + i);
        const bool ok = p >= 0 && p < src_rows;
        const uint8_t *s = src + (size_t)(ok ? p : 0) * src_pitch;
        uint8_t *d = dst + (size_t)i * dst_pitch;
        if (vec16) {
            for (int o = threadIdx.x * 16; o < row_bytes; o += kPermThreads * 16)
                *reinterpret_cast<uint4 *>(d + o) =
                    ok ? __ldg(reinterpret_cast<const uint4 *>(s + o)) : make_uint4(0u, 0u, 0u, 0u);
        } else if (esz == 4) {
            for (int o = threadIdx.x * 4; o < row_bytes; o += kPermThreads * 4)
                *reinterpret_cast<uint32_t *>(d + o) = ok ? __ldg(reinterpret_cast<const uint32_t *>(s + o)) : 0u;
        } else {
            for (int o = threadIdx.x * 2; o < row_bytes; o += kPermThreads * 2)
                *reinterpret_cast<uint16_t *>(d + o) =
                    ok ? __ldg(reinterpret_cast<const unsigned short *>(s + o)) : (uint16_t)0;
        }
    }
}

}  // namespace

using namespace cs;

extern "C" {

cs_status cs_permute_rows(const void *src, int src_rows, int ld_src, const int32_t *perm, int rows, int cols,
                          cs_dtype dtype, void *dst, int ld_dst, cs_stream_t stream) {
    if (dtype != CS_F32 && dtype != CS_F16 && dtype != CS_BF16) {
        set_error("cs_permute_rows: bad dtype %d", (int)dtype);
        return CS_ERR_INVALID;
    }
    const int esz = (int)dtype_size(dtype);
    if (!src || !dst || !perm || src_rows < 1 || rows < 0 || cols < 1 || ld_src < cols || ld_dst < cols ||
        (reinterpret_cast<uintptr_t>(src) % esz) || (reinterpret_cast<uintptr_t>(dst) % esz) ||
        (reinterpret_cast<uintptr_t>(perm) & 3u)) {
        set_error("cs_permute_rows: src, dst and perm are required (element-aligned); src_rows, cols >= 1; "
                  "ld_src, ld_dst >= cols");
        return CS_ERR_INVALID;
    }
    const size_t sp = (size_t)ld_src * esz, dp = (size_t)ld_dst * esz;
    const uint8_t *s8 = static_cast<const uint8_t *>(src);
    uint8_t *d8 = static_cast<uint8_t *>(dst);
    if (s8 < d8 + (size_t)rows * dp && d8 < s8 + (size_t)src_rows * sp) {
        set_error("cs_permute_rows: src and dst overlap");
        return CS_ERR_INVALID;
    }
    if (rows == 0) return CS_OK;
    const int row_bytes = cols * esz;
    const bool vec16 = row_bytes % 16 == 0 && sp % 16 == 0 && dp % 16 == 0 &&
                       (reinterpret_cast<uintptr_t>(src) & 15u) == 0 && (reinterpret_cast<uintptr_t>(dst) & 15u) == 0;
    int sms = device_sm_count();
    const int grid = std::min(rows, 8 * (sms > 0 ? sms : 1));
    permute_rows_kernel<<<grid, kPermThreads, 0, (cudaStream_t)stream>>>(s8, src_rows, sp, perm, rows, d8, dp,
                                                                         row_bytes, esz, vec16);
    cudaError_t e = cudaGetLastError();
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_permute_rows");
}

cs_status cs_hot_order(const float *freq, int f, int32_t *perm) {
    if (f < 0 || (f > 0 && (!freq || !perm))) {
        set_error("cs_hot_order: f >= 0, and freq and perm are required when f > 0");
        return CS_ERR_INVALID;
    }
    std::vector<int32_t> o((size_t)f);
    std::iota(o.begin(), o.end(), 0);
    // most frequent first; NaN as the lowest frequency; ties by lower id
    auto key = [&](int32_t j) { return std::isnan(freq[j]) ? -INFINITY : freq[j]; };
    std::stable_sort(o.begin(), o.end(), [&](int32_t a, int32_t b) {
        const float ka = key(a), kb = key(b);
        if (ka != kb) return ka > kb;
        return std::isnan(freq[a]) < std::isnan(freq[b]);
    });
    std::copy(o.begin(), o.end(), perm);
    return CS_OK;
}

}  // extern "C"
