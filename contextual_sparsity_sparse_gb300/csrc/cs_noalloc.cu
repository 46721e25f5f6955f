// Workspace-free variant of the gathered sparse FFN.
//
// Some callers cannot allocate device memory: a plugin or callback that runs
// inside a host framework which owns every device allocation and hands it no
// allocator, or a latency-critical path where a cudaMalloc (which may
// synchronise the device) is not allowed.  This entry point lets them run the
// gathered FFN without a workspace.  The per-CTA partial sums, which
// cs_sparse_ffn keeps in the caller's workspace, live here in a file-scope
// device array instead.  There is no counterpart of this in the method's
// sources; it only changes where the scratch memory comes from.
#include <cuda.h>

#include <mutex>

#include "cs_internal.cuh"

namespace {

// Fixed scratch capacity: 2^21 fp32 partial sums (8 MiB per GPU that loads the
// library, held until the process exits).  A call needs
// (SM count) * B * roundup(d, 8) of them.
constexpr size_t kNoAllocFloats = size_t(1) << 21;

__device__ __align__(256) float g_noalloc_part[kNoAllocFloats];
__device__ __align__(256) uint32_t g_noalloc_err[64];

// The arrays' device addresses differ per CUDA context (each context loads its
// own copy of the module), so they are looked up once per context and cached
// under that context's handle.  The current context is read through the
// driver entry point that the runtime exposes, so the library does not link
// the driver library itself.
struct Slot {
    CUcontext ctx;
    float *part;
    uint32_t *err;
};
constexpr int kSlots = 64;

std::mutex g_mu;
Slot g_slots[kSlots] = {};
int g_nslots = 0;

using CtxGetCurrentFn = CUresult (*)(CUcontext *);

// The current context, or null when it cannot be read.
CUcontext current_context() {
    static CtxGetCurrentFn fn = [] {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess) {
            cudaGetLastError();
            return static_cast<CtxGetCurrentFn>(nullptr);
        }
        return reinterpret_cast<CtxGetCurrentFn>(p);
    }();
    CUcontext c = nullptr;
    if (!fn || fn(&c) != CUDA_SUCCESS) return nullptr;
    return c;
}

// The arrays' addresses in the current context.
cudaError_t scratch_addresses(float **part, uint32_t **err) {
    const CUcontext ctx = current_context();
    std::lock_guard<std::mutex> lock(g_mu);
    if (ctx) {
        for (int i = 0; i < g_nslots; ++i)
            if (g_slots[i].ctx == ctx) {
                *part = g_slots[i].part;
                *err = g_slots[i].err;
                return cudaSuccess;
            }
    }
    cudaError_t e = cudaGetSymbolAddress(reinterpret_cast<void **>(part), g_noalloc_part);
    if (e != cudaSuccess) return e;
    e = cudaGetSymbolAddress(reinterpret_cast<void **>(err), g_noalloc_err);
    if (e != cudaSuccess) return e;
    // without a readable context every call looks the addresses up again
    if (ctx && g_nslots < kSlots) g_slots[g_nslots++] = Slot{ctx, *part, *err};
    return cudaSuccess;
}

}  // namespace

using namespace cs;

extern "C" cs_status cs_sparse_ffn_noalloc(const cs_ffn_layer *layer, const float *x, int B,
                                           const int32_t *idx, const int32_t *count, float *y,
                                           cs_stream_t stream) {
    int ld = 0;
    cs_status st = validate_layer(layer, &ld);
    if (st != CS_OK) return st;
    auto al4 = [](const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; };
    if (B < 1 || !x || !y || !idx || !count || !al4(x) || !al4(y) || !al4(idx) || !al4(count) || x == y) {
        set_error("cs_sparse_ffn_noalloc: B >= 1 and distinct, 4-byte aligned x, y, idx, count are required");
        return CS_ERR_INVALID;
    }
    const int G = device_sm_count() > 0 ? device_sm_count() : 1;
    const int dp = (layer->d + 7) & ~7;
    const size_t need = (size_t)G * (size_t)B * (size_t)dp;
    if (need > kNoAllocFloats) {
        set_error("cs_sparse_ffn_noalloc: needs %zu partial sums (%d SMs x B=%d x %d), more than the fixed %zu",
                  need, G, B, dp, kNoAllocFloats);
        return CS_ERR_UNSUPPORTED;
    }
    float *part = nullptr;
    uint32_t *err = nullptr;
    cudaError_t e = scratch_addresses(&part, &err);
    if (e != cudaSuccess) return cuda_fail(e, "cs_sparse_ffn_noalloc(symbol address)");
    FfnArgs a;
    a.d = layer->d; a.f = layer->f; a.ld = ld; a.B = B; a.dtype = layer->dtype;
    a.w_gate = layer->w_gate; a.w_up = layer->w_up; a.w_down_t = layer->w_down_t; a.bias = layer->bias;
    a.x = x; a.idx = idx; a.count = count; a.preact = nullptr; a.y = y;
    a.resid = nullptr; a.scale = 1.f; a.act = layer->act;
    a.err = err;     // device-side error bits are not reported by this entry point
    a.part = part;   // every partial row is fully rewritten, so nothing needs clearing
    a.G = G; a.dp = dp;
    // tc_x / tc_a stay null: the tensor-core path needs workspace buffers, so
    // every batch runs on the CUDA-core gather kernel
    e = launch_ffn(a, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_sparse_ffn_noalloc");
}
