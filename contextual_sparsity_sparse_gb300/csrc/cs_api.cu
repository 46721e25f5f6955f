// Host side of the C ABI declared in include/cs.h: argument validation,
// workspace layout and dispatch to the kernels.  No entry point allocates
// device memory; every buffer is the caller's.
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <utility>

#include "cs_internal.cuh"

namespace cs {

int ffn_max_d(cs_dtype t);
cudaError_t launch_transpose(const void *src, cs_dtype st, int rows, int cols, int ld_src, void *dst,
                             cs_dtype dt, int ld_dst, cudaStream_t s);

namespace {
thread_local std::string g_last_error;
}

void set_error(const char *fmt, ...) {
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_last_error = buf;
}

cs_status cuda_fail(cudaError_t e, const char *what) {
    set_error("%s: %s", what, cudaGetErrorString(e));
    return CS_ERR_CUDA;
}

bool pdl_enabled() {
    static const bool on = [] {
        const char *v = getenv("CS_PDL");
        return !(v && v[0] == '0');
    }();
    return on;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

size_t dtype_size(cs_dtype t) { return t == CS_F32 ? 4 : 2; }

WsLayout ws_layout(int d, int f, int r, int B, int num_sms) {
    WsLayout L;
    L.G = num_sms > 0 ? num_sms : 1;
    L.dp = (d + 7) & ~7;
    size_t off = kControlBytes;
    L.err = 0;
    L.part = off;      off += align256(sizeof(float) * (size_t)L.G * B * L.dp);
    L.h = off;         off += align256(sizeof(float) * (size_t)B * r);
    L.st_x = off;      off += align256(sizeof(float) * (size_t)L.dp);
    L.st_scores = off; off += align256(sizeof(float) * (size_t)f);
    L.st_pre = off;    off += align256(sizeof(float) * (size_t)f);
    L.st_idx = off;    off += align256(sizeof(int32_t) * 2 * (size_t)f);
    L.st_count = off;  off += 256;
    L.st_h = off;      off += align256(sizeof(float) * (size_t)r);
    L.io_y = off;      off += align256(sizeof(float) * (size_t)L.dp);
    L.io_x = off;      off += align256(sizeof(float) * (size_t)L.dp);
    L.tc = off;        off += tc_workspace_bytes(d, f, B);
    L.total = off;
    return L;
}

}  // namespace cs

using namespace cs;

namespace {

bool al16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool al4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }
bool dtype_ok(cs_dtype t) { return t == CS_F32 || t == CS_F16 || t == CS_BF16; }

#define CS_CHECK(cond, ...)                       \
    do {                                          \
        if (!(cond)) {                            \
            set_error(__VA_ARGS__);               \
            return CS_ERR_INVALID;                \
        }                                         \
    } while (0)

cs_status check_ws(void *ws, size_t ws_bytes, int d, int f, int r, int B, WsLayout *out) {
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) {
        set_error("workspace is null or not 256-byte aligned");
        return CS_ERR_WORKSPACE;
    }
    *out = ws_layout(d, f, r, B, device_sm_count());
    if (ws_bytes < out->total) {
        set_error("workspace too small: %zu bytes given, %zu needed", ws_bytes, out->total);
        return CS_ERR_WORKSPACE;
    }
    return CS_OK;
}

cs_status check_layer(const cs_ffn_layer *L, int *ld_out) {
    CS_CHECK(L, "layer is null");
    CS_CHECK(L->d >= 1 && L->f >= 1, "layer: d and f must be >= 1 (d=%d f=%d)", L->d, L->f);
    CS_CHECK(dtype_ok(L->dtype), "layer: bad dtype %d", (int)L->dtype);
    CS_CHECK(L->act == CS_ACT_RELU || L->act == CS_ACT_SILU, "layer: bad activation %d", (int)L->act);
    const int ld = L->ld ? L->ld : L->d;
    const size_t es = dtype_size(L->dtype);
    CS_CHECK(ld >= L->d, "layer: ld %d < d %d", ld, L->d);
    CS_CHECK((ld * es) % 16 == 0, "layer: ld * element size must be a multiple of 16 bytes");
    CS_CHECK(L->w_gate && L->w_down_t, "layer: w_gate and w_down_t are required");
    CS_CHECK(al16(L->w_gate) && al16(L->w_down_t) && al16(L->w_up), "layer: weights must be 16-byte aligned");
    CS_CHECK(!L->bias || al4(L->bias), "layer: bias must be 4-byte aligned");
    if (L->f > 2048 * (device_sm_count() > 0 ? device_sm_count() : 1)) {
        set_error("layer: f=%d exceeds the supported maximum (2048 per SM)", L->f);
        return CS_ERR_UNSUPPORTED;
    }
    if (L->d > ffn_max_d(L->dtype)) {
        set_error("layer: d=%d exceeds the supported maximum %d", L->d, ffn_max_d(L->dtype));
        return CS_ERR_UNSUPPORTED;
    }
    *ld_out = ld;
    return CS_OK;
}

cs_status check_pred(const cs_predictor *P) {
    CS_CHECK(P, "predictor is null");
    CS_CHECK(P->d >= 1 && P->r >= 1 && P->f >= 1, "predictor: d, r, f must be >= 1");
    CS_CHECK(dtype_ok(P->dtype), "predictor: bad dtype %d", (int)P->dtype);
    const size_t es = dtype_size(P->dtype);
    const int ldd = P->ld_down ? P->ld_down : P->d;
    const int ldu = P->ld_up ? P->ld_up : P->r;
    CS_CHECK(ldd >= P->d && ldu >= P->r, "predictor: row stride smaller than the row");
    CS_CHECK((ldd * es) % 16 == 0 && (ldu * es) % 16 == 0,
             "predictor: row strides must be multiples of 16 bytes");
    CS_CHECK(P->p_down && P->p_up && al16(P->p_down) && al16(P->p_up),
             "predictor: weights must be non-null and 16-byte aligned");
    if (P->r > 8192) {
        set_error("predictor: r=%d exceeds the supported maximum 8192", P->r);
        return CS_ERR_UNSUPPORTED;
    }
    return CS_OK;
}

}  // namespace

cs_status cs::validate_layer(const cs_ffn_layer *layer, int *ld_out) { return check_layer(layer, ld_out); }

extern "C" {

const char *cs_version(void) { return "contextual_sparsity_sparse_gb300 0.1 (sm_103a)"; }

const char *cs_status_string(cs_status s) {
    switch (s) {
    case CS_OK: return "ok";
    case CS_ERR_INVALID: return "invalid argument";
    case CS_ERR_CUDA: return "CUDA error";
    case CS_ERR_UNSUPPORTED: return "unsupported";
    case CS_ERR_TIMEOUT: return "device wait timed out";
    case CS_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char *cs_last_error(void) { return g_last_error.c_str(); }

size_t cs_workspace_size(int d, int f, int r, int B) {
    if (d < 1 || f < 1 || r < 0 || B < 1) return 0;
    return ws_layout(d, f, r < 1 ? 1 : r, B, device_sm_count()).total;
}

cs_status cs_workspace_init(void *ws, size_t ws_bytes, cs_stream_t stream) {
    if (!ws || ws_bytes < 256 || (reinterpret_cast<uintptr_t>(ws) & 255u)) {
        set_error("workspace is null, misaligned or smaller than 256 bytes");
        return CS_ERR_WORKSPACE;
    }
    if (ws_bytes < kControlBytes) {
        set_error("workspace smaller than its control region (%zu bytes)", kControlBytes);
        return CS_ERR_WORKSPACE;
    }
    cudaError_t e = cudaMemsetAsync(ws, 0, kControlBytes, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_workspace_init");
}

cs_status cs_get_device_error(void *ws, cs_stream_t stream, int clear, uint32_t *code_out) {
    CS_CHECK(ws && code_out, "cs_get_device_error: null argument");
    uint32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, ws, sizeof v, cudaMemcpyDeviceToHost, (cudaStream_t)stream);
    if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
    if (e != cudaSuccess) return cuda_fail(e, "cs_get_device_error");
    *code_out = v;
    if (clear) {
        e = cudaMemsetAsync(ws, 0, sizeof v, (cudaStream_t)stream);
        if (e == cudaSuccess) e = cudaStreamSynchronize((cudaStream_t)stream);
        if (e != cudaSuccess) return cuda_fail(e, "cs_get_device_error(clear)");
    }
    return CS_OK;
}

cs_status cs_pack_transpose(const void *src, cs_dtype src_dtype, int rows, int cols, int ld_src,
                            void *dst, cs_dtype dst_dtype, int ld_dst, cs_stream_t stream) {
    CS_CHECK(src && dst, "cs_pack_transpose: null pointer");
    CS_CHECK(dtype_ok(src_dtype) && dtype_ok(dst_dtype), "cs_pack_transpose: bad dtype");
    CS_CHECK(rows >= 0 && cols >= 0, "cs_pack_transpose: negative size");
    CS_CHECK(ld_src >= cols && ld_dst >= rows, "cs_pack_transpose: stride smaller than the row");
    CS_CHECK(src != dst, "cs_pack_transpose: in-place transpose is not supported");
    if (rows == 0 || cols == 0) return CS_OK;
    cudaError_t e = launch_transpose(src, src_dtype, rows, cols, ld_src, dst, dst_dtype, ld_dst,
                                     (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_pack_transpose");
}

cs_status cs_predict(const cs_predictor *pred, const float *x, int B, float *scores, void *ws,
                     size_t ws_bytes, cs_stream_t stream) {
    cs_status st = check_pred(pred);
    if (st != CS_OK) return st;
    CS_CHECK(x && scores && al4(x) && al4(scores), "cs_predict: x and scores must be non-null fp32 arrays");
    CS_CHECK(B >= 1, "cs_predict: B must be >= 1");
    WsLayout L;
    st = check_ws(ws, ws_bytes, pred->d, pred->f, pred->r, B, &L);
    if (st != CS_OK) return st;
    PredictArgs a;
    a.d = pred->d; a.r = pred->r; a.f = pred->f; a.B = B;
    a.dtype = pred->dtype; a.ld_down = pred->ld_down; a.ld_up = pred->ld_up;
    a.p_down = pred->p_down; a.p_up = pred->p_up;
    a.x = x;
    a.h = reinterpret_cast<float *>(static_cast<char *>(ws) + L.h);
    a.scores = scores;
    a.err = static_cast<uint32_t *>(ws);
    cudaError_t e = launch_predict(a, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_predict");
}

cs_status cs_select(const float *scores, int B, int f, const cs_select_params *params, int32_t *idx,
                    int32_t *count, uint32_t *mask, void *ws, size_t ws_bytes, cs_stream_t stream) {
    CS_CHECK(params, "cs_select: params is null");
    CS_CHECK(scores && idx && count && al4(scores) && al4(idx) && al4(count) && al4(mask),
             "cs_select: scores, idx and count are required (4-byte aligned)");
    CS_CHECK(B >= 1 && f >= 1, "cs_select: B and f must be >= 1");
    CS_CHECK(params->mode == CS_SEL_TOPK || params->mode == CS_SEL_THRESHOLD,
             "cs_select: mode must be CS_SEL_TOPK or CS_SEL_THRESHOLD (exact mode is cs_exact_ffn)");
    CS_CHECK(params->hot >= 0 && params->hot % 32 == 0 && params->hot <= (1 << 30) - f,
             "cs_select: hot must be a non-negative multiple of 32 (got %d)", params->hot);
    if (f > kSelectMaxF) {
        set_error("cs_select: f=%d exceeds the supported maximum %d", f, kSelectMaxF);
        return CS_ERR_UNSUPPORTED;
    }
    (void)ws;
    (void)ws_bytes;
    SelectArgs a;
    a.scores = scores; a.B = B; a.f = f;
    a.kind = params->mode == CS_SEL_TOPK ? SEL_TOPK : SEL_THRESHOLD;
    a.k = params->k; a.tau = params->tau;
    a.hot = params->hot;
    a.idx = idx; a.ld_idx = params->hot + f; a.count = count; a.mask = mask;
    cudaError_t e = launch_select(a, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_select");
}

cs_status cs_sparse_ffn(const cs_ffn_layer *layer, const float *x, int B, const int32_t *idx,
                        const int32_t *count, float *y, void *ws, size_t ws_bytes, cs_stream_t stream) {
    int ld = 0;
    cs_status st = check_layer(layer, &ld);
    if (st != CS_OK) return st;
    CS_CHECK(B >= 1, "cs_sparse_ffn: B must be >= 1");
    CS_CHECK(x && y && idx && count && al4(x) && al4(y) && al4(idx) && al4(count),
             "cs_sparse_ffn: x, y, idx and count are required (4-byte aligned)");
    CS_CHECK(x != y, "cs_sparse_ffn: y must not alias x");
    WsLayout L;
    st = check_ws(ws, ws_bytes, layer->d, layer->f, 1, B, &L);
    if (st != CS_OK) return st;
    FfnArgs a;
    a.d = layer->d; a.f = layer->f; a.ld = ld; a.B = B; a.dtype = layer->dtype;
    a.w_gate = layer->w_gate; a.w_up = layer->w_up; a.w_down_t = layer->w_down_t; a.bias = layer->bias;
    a.x = x; a.idx = idx; a.count = count; a.preact = nullptr; a.y = y;
    a.resid = nullptr; a.scale = 1.f; a.act = layer->act;
    a.err = static_cast<uint32_t *>(ws);
    a.part = reinterpret_cast<float *>(static_cast<char *>(ws) + L.part);
    a.G = L.G; a.dp = L.dp;
    if (tc_workspace_bytes(a.d, a.f, B) > 0) {
        a.tc_x = static_cast<char *>(ws) + L.tc;
        a.tc_a = static_cast<char *>(ws) + L.tc + tc_x_bytes(a.d, B);
    }
    cudaError_t e = launch_ffn(a, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_sparse_ffn");
}

cs_status cs_exact_ffn(const cs_ffn_layer *layer, const float *x, float *preact, int32_t *idx,
                       int32_t *count, uint32_t *mask, float *y, float tau, void *ws, size_t ws_bytes,
                       cs_stream_t stream) {
    int ld = 0;
    cs_status st = check_layer(layer, &ld);
    if (st != CS_OK) return st;
    CS_CHECK(x && preact && idx && count && y && al4(x) && al4(preact) && al4(idx) && al4(count) &&
                 al4(y) && al4(mask),
             "cs_exact_ffn: x, preact, idx, count and y are required (4-byte aligned)");
    CS_CHECK(x != y, "cs_exact_ffn: y must not alias x");
    CS_CHECK(tau >= 0.f, "cs_exact_ffn: tau must be >= 0");
    if (layer->f > kSelectMaxF) {
        set_error("cs_exact_ffn: f=%d exceeds the supported maximum %d", layer->f, kSelectMaxF);
        return CS_ERR_UNSUPPORTED;
    }
    WsLayout L;
    st = check_ws(ws, ws_bytes, layer->d, layer->f, 1, 1, &L);
    if (st != CS_OK) return st;
    cudaStream_t s = (cudaStream_t)stream;
    PreactArgs p;
    p.d = layer->d; p.f = layer->f; p.ld = ld; p.dtype = layer->dtype;
    p.w_gate = layer->w_gate; p.bias = layer->bias; p.x = x; p.pre = preact;
    p.err = static_cast<uint32_t *>(ws);
    cudaError_t e = launch_preact(p, s);
    if (e != cudaSuccess) return cuda_fail(e, "cs_exact_ffn(preact)");
    SelectArgs sa;
    sa.scores = preact; sa.B = 1; sa.f = layer->f; sa.k = 0; sa.tau = tau;
    sa.kind = layer->act == CS_ACT_SILU ? SEL_SILU_MAG : SEL_POSITIVE;
    sa.idx = idx; sa.ld_idx = layer->f; sa.count = count; sa.mask = mask;
    e = launch_select(sa, s);
    if (e != cudaSuccess) return cuda_fail(e, "cs_exact_ffn(select)");
    FfnArgs a;
    a.d = layer->d; a.f = layer->f; a.ld = ld; a.B = 1; a.dtype = layer->dtype;
    a.w_gate = layer->w_gate; a.w_up = layer->w_up; a.w_down_t = layer->w_down_t; a.bias = layer->bias;
    a.x = x; a.idx = idx; a.count = count; a.preact = preact; a.y = y;
    a.resid = nullptr; a.scale = 1.f; a.act = layer->act;
    a.err = static_cast<uint32_t *>(ws);
    a.part = reinterpret_cast<float *>(static_cast<char *>(ws) + L.part);
    a.G = L.G; a.dp = L.dp;
    e = launch_ffn(a, s);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_exact_ffn(ffn)");
}

cs_status cs_union_mask(const uint32_t *masks, int B, int f, uint32_t *umask, int32_t *uidx,
                        int32_t *ucount, void *ws, size_t ws_bytes, cs_stream_t stream) {
    CS_CHECK(masks && umask && uidx && ucount && al4(masks) && al4(umask) && al4(uidx) && al4(ucount),
             "cs_union_mask: null or misaligned pointer");
    CS_CHECK(B >= 1 && f >= 1, "cs_union_mask: B and f must be >= 1");
    (void)ws;
    (void)ws_bytes;
    UnionArgs a;
    a.masks = masks; a.B = B; a.f = f; a.umask = umask; a.uidx = uidx; a.ucount = ucount;
    cudaError_t e = launch_union(a, (cudaStream_t)stream);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_union_mask");
}

}  // extern "C"
