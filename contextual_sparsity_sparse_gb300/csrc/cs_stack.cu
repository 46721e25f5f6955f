// Layer stack on the residual stream, with look-ahead prediction.
//
// Source: "Contextual Sparsity and Activation Predictors", section "The
// predictor and its budget": the residual stream changes slowly between
// blocks (x_{l+1} = x_l + f_l(x_l)), so the sparsity of layer l+1 can be
// predicted from the input of layer l and the prediction run asynchronously,
// off the critical path.  Section "When it breaks" notes the approximation is
// weakest in early layers.
//
// GB300 mapping.  Stream P runs predictor + selection of layer l+1 from x_l
// while stream M runs layer l's gathered FFN, which writes
// x_{l+1} = x_l + c * FFN_l(x_l) into the other half of a ping-pong pair.
// Dependencies are CUDA events; the whole L-layer fork/join is captured once
// into a CUDA graph (per distinct argument set) and replayed, so a decode step
// costs one graph launch instead of ~4L kernel launches.
//
// The same machinery serves cs_decode_layer, one layer's step for one token
// (predictor, selection, gathered FFN; y without the residual): its five
// kernels become one cached graph.
//
// x / y in page-locked host memory are read and written by the graph itself:
// a small copy kernel at each end of the graph reaches the host buffer through
// its device mapping (GB300's host memory sits behind NVLink-C2C), and the
// cached graph's two copy nodes are pointed at each call's buffers by a node
// parameter update, so no copy-engine transfer is issued per call.  Without a
// device mapping the buffers are staged by copies around the graph launch.
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <string>
#include <unordered_map>
#include <utility>
#include <vector>

#include "cs_internal.cuh"

namespace cs {
int ffn_max_d(cs_dtype t);
}

using namespace cs;

namespace {

struct StackPlan {
    const cs_ffn_layer *layers;
    const cs_predictor *preds;
    int L, d, f, r;
    float *x;
    float scale;
    cs_select_params sel;
    cs_stack_mode mode;
    char *ws;
    WsLayout lay;
    int32_t *trace_count, *trace_idx;
    bool layer_only = false;  // single-layer step: y = FFN(x), no residual
    float *y = nullptr;       // its output
    // device mappings of the caller's page-locked host x (read into p.x
    // first) and host y (or the stack's x, written from p.y / p.x last)
    const float *io_src = nullptr;
    float *io_dst = nullptr;
    // one token's head-sparse attention instead of the FFN layers: the
    // predictor scores the heads, the selection picks them (into
    // trace_idx / trace_count when given), y = the attention
    const AttnCall *attn = nullptr;
};

constexpr int kIoThreads = 256;

struct IoCopy {
    const float *src;
    float *dst;
    int n;
};

dim3 io_grid(int n) { return dim3((unsigned)((n + 4 * kIoThreads - 1) / (4 * kIoThreads))); }

// dst[0, n) = src[0, n), four floats per thread (16-byte accesses when both
// ends allow them).  DIR 0 is the graph's first node (host x in), DIR 1 its
// last (y, or the stack's x, out); the two instantiations tell the nodes apart.
template <int DIR>
__global__ void __launch_bounds__(kIoThreads) io_copy_kernel(const IoCopy a) {
    pdl_launch_dependents();
    pdl_wait();  // DIR 1 reads what the reduction wrote
    const int i = (blockIdx.x * kIoThreads + threadIdx.x) * 4;
    if (i >= a.n) return;
    const bool v16 = ((reinterpret_cast<uintptr_t>(a.src) | reinterpret_cast<uintptr_t>(a.dst)) & 15u) == 0;
    if (v16 && i + 4 <= a.n) {
        *reinterpret_cast<float4 *>(a.dst + i) = ld_dep(reinterpret_cast<const float4 *>(a.src + i));
    } else {
        for (int j = i; j < a.n && j < i + 4; ++j) a.dst[j] = ld_dep(a.src + j);
    }
}

cudaError_t launch_io(int dir, const IoCopy &a, cudaStream_t s) {
    return launch(dir == 0 ? io_copy_kernel<0> : io_copy_kernel<1>, io_grid(a.n), dim3(kIoThreads), 0, s,
                  pdl_enabled(), a);
}

struct Bufs {
    float *xb[2];
    float *h, *scores, *pre, *part;
    int32_t *idx_slot[2], *cnt_slot[2];
    uint32_t *err;
};

Bufs bufs_of(const StackPlan &p) {
    Bufs b;
    b.xb[0] = p.x;
    b.xb[1] = reinterpret_cast<float *>(p.ws + p.lay.st_x);
    b.h = reinterpret_cast<float *>(p.ws + p.lay.st_h);
    b.scores = reinterpret_cast<float *>(p.ws + p.lay.st_scores);
    b.pre = reinterpret_cast<float *>(p.ws + p.lay.st_pre);
    b.part = reinterpret_cast<float *>(p.ws + p.lay.part);
    int32_t *slots = reinterpret_cast<int32_t *>(p.ws + p.lay.st_idx);
    b.idx_slot[0] = slots;
    b.idx_slot[1] = slots + p.f;
    int32_t *cnt = reinterpret_cast<int32_t *>(p.ws + p.lay.st_count);
    b.cnt_slot[0] = cnt;
    b.cnt_slot[1] = cnt + 1;
    b.err = reinterpret_cast<uint32_t *>(p.ws);
    return b;
}

void sel_out(const StackPlan &p, const Bufs &b, int l, int32_t **idx, int32_t **cnt) {
    if (p.trace_idx) *idx = p.trace_idx + (size_t)l * p.f;
    else *idx = b.idx_slot[l & 1];
    if (p.trace_count) *cnt = p.trace_count + l;
    else *cnt = b.cnt_slot[l & 1];
}

cudaError_t predict_select(const StackPlan &p, const Bufs &b, int l, const float *xin, cudaStream_t s) {
    const cs_predictor &P = p.preds[l];
    PredictArgs a;
    a.d = P.d; a.r = P.r; a.f = P.f; a.B = 1; a.dtype = P.dtype;
    a.ld_down = P.ld_down; a.ld_up = P.ld_up; a.p_down = P.p_down; a.p_up = P.p_up;
    a.x = xin; a.h = b.h; a.scores = b.scores; a.err = b.err;
    cudaError_t e = launch_predict(a, s);
    if (e != cudaSuccess) return e;
    // the predictor scores neurons hot .. f-1; the selection adds 0 .. hot-1
    SelectArgs sa;
    sa.scores = b.scores; sa.B = 1; sa.f = p.f - p.sel.hot;
    sa.kind = p.sel.mode == CS_SEL_TOPK ? SEL_TOPK : SEL_THRESHOLD;
    sa.k = p.sel.k; sa.tau = p.sel.tau; sa.hot = p.sel.hot;
    sel_out(p, b, l, &sa.idx, &sa.count);
    sa.ld_idx = p.f; sa.mask = nullptr;
    return launch_select(sa, s);
}

cudaError_t ffn_step(const StackPlan &p, const Bufs &b, int l, const float *xin, float *xout,
                     const float *preact, cudaStream_t s) {
    const cs_ffn_layer &Ly = p.layers[l];
    FfnArgs a;
    a.d = Ly.d; a.f = Ly.f; a.ld = Ly.ld ? Ly.ld : Ly.d; a.B = 1; a.dtype = Ly.dtype;
    a.w_gate = Ly.w_gate; a.w_up = Ly.w_up; a.w_down_t = Ly.w_down_t; a.bias = Ly.bias;
    a.act = Ly.act;
    a.x = xin;
    int32_t *idx, *cnt;
    sel_out(p, b, l, &idx, &cnt);
    a.idx = idx; a.count = cnt;
    a.preact = preact;
    a.y = xout;
    a.resid = p.layer_only ? nullptr : xin;
    a.scale = p.layer_only ? 1.f : p.scale;
    a.err = b.err; a.part = b.part; a.G = p.lay.G; a.dp = p.lay.dp;
    return launch_ffn(a, s);
}

cudaError_t exact_step(const StackPlan &p, const Bufs &b, int l, const float *xin, float *xout,
                       cudaStream_t s) {
    const cs_ffn_layer &Ly = p.layers[l];
    PreactArgs pa;
    pa.d = Ly.d; pa.f = Ly.f; pa.ld = Ly.ld ? Ly.ld : Ly.d; pa.dtype = Ly.dtype;
    pa.w_gate = Ly.w_gate; pa.bias = Ly.bias; pa.x = xin; pa.pre = b.pre; pa.err = b.err;
    cudaError_t e = launch_preact(pa, s);
    if (e != cudaSuccess) return e;
    SelectArgs sa;
    // the magnitude cut |act(g)| > tau (g > 0 for relu at tau = 0)
    sa.scores = b.pre; sa.B = 1; sa.f = p.f; sa.k = 0; sa.tau = p.sel.tau;
    sa.kind = Ly.act == CS_ACT_SILU ? SEL_SILU_MAG : SEL_POSITIVE;
    sel_out(p, b, l, &sa.idx, &sa.count);
    sa.ld_idx = p.f; sa.mask = nullptr;
    e = launch_select(sa, s);
    if (e != cudaSuccess) return e;
    return ffn_step(p, b, l, xin, xout, b.pre, s);
}

struct Events {
    std::vector<cudaEvent_t> ev;
    ~Events() {
        for (cudaEvent_t e : ev) cudaEventDestroy(e);
    }
    cudaError_t make(int n) {
        ev.resize(n, nullptr);
        for (int i = 0; i < n; ++i) {
            cudaError_t e = cudaEventCreateWithFlags(&ev[i], cudaEventDisableTiming);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
};

#define TRY(x)                                  \
    do {                                        \
        cudaError_t e_ = (x);                   \
        if (e_ != cudaSuccess) return e_;       \
    } while (0)

// Enqueue the whole stack.  s_pred is only touched in look-ahead mode.
cudaError_t enqueue_stack(const StackPlan &p, cudaStream_t sm, cudaStream_t sp, Events &E) {
    const Bufs b = bufs_of(p);
    const int L = p.L;
    if (p.io_src) TRY(launch_io(0, IoCopy{p.io_src, p.x, p.d}, sm));
    if (p.sel.mode == CS_SEL_EXACT) {
        for (int l = 0; l < L; ++l) TRY(exact_step(p, b, l, b.xb[l & 1], b.xb[(l + 1) & 1], sm));
    } else if (p.mode == CS_STACK_SEQUENTIAL || sp == sm) {
        if (p.mode == CS_STACK_SEQUENTIAL) {
            for (int l = 0; l < L; ++l) {
                TRY(predict_select(p, b, l, b.xb[l & 1], sm));
                TRY(ffn_step(p, b, l, b.xb[l & 1], b.xb[(l + 1) & 1], nullptr, sm));
            }
        } else {
            // look-ahead semantics on one stream: layer l+1's set from x_l
            TRY(predict_select(p, b, 0, b.xb[0], sm));
            for (int l = 0; l < L; ++l) {
                if (l + 1 < L) TRY(predict_select(p, b, l + 1, b.xb[l & 1], sm));
                TRY(ffn_step(p, b, l, b.xb[l & 1], b.xb[(l + 1) & 1], nullptr, sm));
            }
        }
    } else {
        // events: 0 fork, 1 join, 2..2+L sel[l], 2+L..2+2L+1 x[l]
        TRY(E.make(2 + L + L + 1));
        cudaEvent_t ev_fork = E.ev[0], ev_join = E.ev[1];
        auto ev_sel = [&](int l) { return E.ev[2 + l]; };
        auto ev_x = [&](int l) { return E.ev[2 + L + l]; };
        TRY(cudaEventRecord(ev_fork, sm));
        TRY(cudaStreamWaitEvent(sp, ev_fork, 0));
        TRY(predict_select(p, b, 0, b.xb[0], sp));
        TRY(cudaEventRecord(ev_sel(0), sp));
        for (int l = 0; l < L; ++l) {
            if (l + 1 < L) {
                if (l > 0) TRY(cudaStreamWaitEvent(sp, ev_x(l), 0));
                TRY(predict_select(p, b, l + 1, b.xb[l & 1], sp));
                TRY(cudaEventRecord(ev_sel(l + 1), sp));
            }
            TRY(cudaStreamWaitEvent(sm, ev_sel(l), 0));
            TRY(ffn_step(p, b, l, b.xb[l & 1], b.xb[(l + 1) & 1], nullptr, sm));
            TRY(cudaEventRecord(ev_x(l + 1), sm));
        }
        TRY(cudaEventRecord(ev_join, sp));
        TRY(cudaStreamWaitEvent(sm, ev_join, 0));
    }
    if (p.io_dst) return launch_io(1, IoCopy{b.xb[L & 1], p.io_dst, p.d}, sm);
    if (L & 1)
        TRY(cudaMemcpyAsync(p.x, b.xb[1], sizeof(float) * (size_t)p.d, cudaMemcpyDeviceToDevice, sm));
    return cudaSuccess;
}

// Enqueue one token's head-sparse attention: y = attention(x, select(P(x))).
cudaError_t enqueue_attention(const StackPlan &p, cudaStream_t s) {
    const Bufs b = bufs_of(p);
    if (p.io_src) TRY(launch_io(0, IoCopy{p.io_src, p.x, p.d}, s));
    const cs_predictor &P = p.preds[0];
    PredictArgs a;
    a.d = P.d; a.r = P.r; a.f = P.f; a.B = 1; a.dtype = P.dtype;
    a.ld_down = P.ld_down; a.ld_up = P.ld_up; a.p_down = P.p_down; a.p_up = P.p_up;
    a.x = p.x; a.h = b.h; a.scores = b.scores; a.err = b.err;
    TRY(launch_predict(a, s));
    SelectArgs sa;
    sa.scores = b.scores; sa.B = 1; sa.f = p.f;
    sa.kind = p.sel.mode == CS_SEL_TOPK ? SEL_TOPK : SEL_THRESHOLD;
    sa.k = p.sel.k; sa.tau = p.sel.tau; sa.hot = 0;
    sel_out(p, b, 0, &sa.idx, &sa.count);
    sa.ld_idx = p.f; sa.mask = nullptr;
    TRY(launch_select(sa, s));
    TRY(attn_launch(*p.attn, p.x, sa.idx, sa.count, p.y, s));
    if (p.io_dst) TRY(launch_io(1, IoCopy{p.y, p.io_dst, p.d}, s));
    return cudaSuccess;
}

// Enqueue one layer's step for one token: y = FFN(x, select(P(x))).
cudaError_t enqueue_layer(const StackPlan &p, cudaStream_t s) {
    const Bufs b = bufs_of(p);
    if (p.io_src) TRY(launch_io(0, IoCopy{p.io_src, p.x, p.d}, s));
    if (p.sel.mode == CS_SEL_EXACT) TRY(exact_step(p, b, 0, p.x, p.y, s));
    else {
        TRY(predict_select(p, b, 0, p.x, s));
        TRY(ffn_step(p, b, 0, p.x, p.y, nullptr, s));
    }
    if (p.io_dst) TRY(launch_io(1, IoCopy{p.y, p.io_dst, p.d}, s));
    return cudaSuccess;
}

struct CacheEntry {
    cudaGraphExec_t exec = nullptr;
    cudaGraph_t graph = nullptr;      // kept while its copy nodes are updated
    cudaGraphNode_t io_node[2] = {nullptr, nullptr};
    IoCopy io_args[2] = {};
    int device = -1;
};

// Set when a captured graph's copy nodes could not be found (its kernel
// nodes do not report their functions): host I/O then uses copies.
bool g_io_nodes_unusable = false;

// CS_GRAPH_IO=0 stages host x / y with copies around the graph launch
// instead of the graph's own copy kernels (read at every call).
bool graph_io_enabled() {
    const char *v = getenv("CS_GRAPH_IO");
    return !(v && v[0] == '0');
}

std::mutex g_mu;
std::unordered_map<std::string, CacheEntry> g_cache;
constexpr size_t kMaxCached = 64;

std::string plan_key(const StackPlan &p, cudaStream_t sp, int dev) {
    std::string k;
    auto put = [&](const void *v, size_t n) { k.append(static_cast<const char *>(v), n); };
    put(&dev, sizeof dev);
    put(&p.L, sizeof p.L);
    const bool attn = p.attn != nullptr;
    put(&attn, sizeof attn);
    if (attn) {
        put(&p.attn->layer, sizeof p.attn->layer);
        put(&p.attn->k_cache, sizeof p.attn->k_cache);
        put(&p.attn->v_cache, sizeof p.attn->v_cache);
        put(&p.attn->seq_len, sizeof p.attn->seq_len);
    } else {
        put(p.layers, sizeof(cs_ffn_layer) * p.L);
    }
    if (p.sel.mode != CS_SEL_EXACT) put(p.preds, sizeof(cs_predictor) * p.L);
    put(&p.x, sizeof p.x);
    put(&p.scale, sizeof p.scale);
    put(&p.sel, sizeof p.sel);
    put(&p.mode, sizeof p.mode);
    put(&p.ws, sizeof p.ws);
    put(&p.trace_count, sizeof p.trace_count);
    put(&p.trace_idx, sizeof p.trace_idx);
    put(&p.layer_only, sizeof p.layer_only);
    put(&p.y, sizeof p.y);
    const bool same = sp == nullptr;
    put(&same, sizeof same);
    // the copy nodes' host addresses change per call; only their presence
    // shapes the graph
    const bool io[2] = {p.io_src != nullptr, p.io_dst != nullptr};
    put(io, sizeof io);
    return k;
}

void destroy_entry(CacheEntry &ce) {
    if (ce.exec) cudaGraphExecDestroy(ce.exec);
    if (ce.graph) cudaGraphDestroy(ce.graph);
    ce.exec = nullptr;
    ce.graph = nullptr;
}

void clear_cache_locked() {
    for (auto &kv : g_cache) destroy_entry(kv.second);
    g_cache.clear();
}

// The copy nodes of a captured graph and their current arguments.
cudaError_t find_io_nodes(CacheEntry &ce) {
    size_t n = 0;
    TRY(cudaGraphGetNodes(ce.graph, nullptr, &n));
    std::vector<cudaGraphNode_t> nodes(n);
    TRY(cudaGraphGetNodes(ce.graph, nodes.data(), &n));
    const void *fn[2] = {reinterpret_cast<const void *>(io_copy_kernel<0>),
                         reinterpret_cast<const void *>(io_copy_kernel<1>)};
    for (size_t i = 0; i < n; ++i) {
        cudaGraphNodeType t;
        TRY(cudaGraphNodeGetType(nodes[i], &t));
        if (t != cudaGraphNodeTypeKernel) continue;
        cudaKernelNodeParams kp = {};
        TRY(cudaGraphKernelNodeGetParams(nodes[i], &kp));
        for (int dir = 0; dir < 2; ++dir) {
            if (kp.func == fn[dir] && kp.kernelParams) {
                ce.io_node[dir] = nodes[i];
                ce.io_args[dir] = *static_cast<const IoCopy *>(kp.kernelParams[0]);
            }
        }
    }
    return cudaSuccess;
}

// Point the cached graph's copy nodes at this call's host buffers.
cudaError_t update_io(CacheEntry &ce, const StackPlan &p) {
    const float *src[2] = {p.io_src, nullptr};
    float *dst[2] = {nullptr, p.io_dst};
    for (int dir = 0; dir < 2; ++dir) {
        if (!ce.io_node[dir]) continue;
        IoCopy a = ce.io_args[dir];
        if (dir == 0) a.src = src[0];
        else a.dst = dst[1];
        if (a.src == ce.io_args[dir].src && a.dst == ce.io_args[dir].dst) continue;
        cudaKernelNodeParams kp = {};
        kp.func = dir == 0 ? reinterpret_cast<void *>(io_copy_kernel<0>) : reinterpret_cast<void *>(io_copy_kernel<1>);
        kp.gridDim = io_grid(a.n);
        kp.blockDim = dim3(kIoThreads);
        kp.sharedMemBytes = 0;
        void *args[] = {&a};
        kp.kernelParams = args;
        kp.extra = nullptr;
        TRY(cudaGraphExecKernelNodeSetParams(ce.exec, ce.io_node[dir], &kp));
        ce.io_args[dir] = a;
    }
    return cudaSuccess;
}

// A predictor scoring f outputs from d inputs through rank r, with valid
// pointers, pitches and dtype.
bool pred_ok(const cs_predictor &P, int d, int f, int r) {
    const int ldd = P.ld_down ? P.ld_down : P.d, ldu = P.ld_up ? P.ld_up : P.r;
    const size_t ep = dtype_size(P.dtype);
    return !(P.d != d || P.f != f || P.r != r || P.r < 1 || !P.p_down || !P.p_up || ldd < d || ldu < r ||
             (ldd * ep) % 16 || (ldu * ep) % 16 || (reinterpret_cast<uintptr_t>(P.p_down) & 15u) ||
             (reinterpret_cast<uintptr_t>(P.p_up) & 15u) || P.r > 8192 ||
             (P.dtype != CS_F32 && P.dtype != CS_F16 && P.dtype != CS_BF16));
}

// Shape and layout checks shared by the stack and the single-layer step.
cs_status check_models(const cs_ffn_layer *layers, const cs_predictor *preds, int L, bool exact,
                       int hot, const char *who) {
    const int d = layers[0].d, f = layers[0].f, r = exact ? 1 : preds[0].r;
    const cs_dtype dt = layers[0].dtype;
    if (d < 1 || f < 1 || (dt != CS_F32 && dt != CS_F16 && dt != CS_BF16)) {
        set_error("%s: layer 0 has a bad shape or dtype", who);
        return CS_ERR_INVALID;
    }
    if (!exact && hot >= f) {
        set_error("%s: the hot prefix (%d) must leave a tail of neurons to predict (f = %d)", who, hot, f);
        return CS_ERR_INVALID;
    }
    for (int l = 0; l < L; ++l) {
        const cs_ffn_layer &Ly = layers[l];
        const int ld = Ly.ld ? Ly.ld : Ly.d;
        const size_t es = dtype_size(Ly.dtype);
        if (Ly.d != d || Ly.f != f || Ly.dtype != dt || ld < d || (ld * es) % 16 ||
            (Ly.act != CS_ACT_RELU && Ly.act != CS_ACT_SILU) ||
            !Ly.w_gate || !Ly.w_down_t || (reinterpret_cast<uintptr_t>(Ly.w_gate) & 15u) ||
            (reinterpret_cast<uintptr_t>(Ly.w_down_t) & 15u) || (reinterpret_cast<uintptr_t>(Ly.w_up) & 15u) ||
            (reinterpret_cast<uintptr_t>(Ly.bias) & 3u)) {
            set_error("%s: layer %d has a different shape or an invalid layout", who, l);
            return CS_ERR_INVALID;
        }
        if (!exact) {
            if (!pred_ok(preds[l], d, f - hot, r)) {
                set_error("%s: predictor %d does not match the layers or is invalid (it must score the "
                          "f - hot = %d tail neurons)", who, l, f - hot);
                return CS_ERR_INVALID;
            }
        }
    }
    if (d > ffn_max_d(dt) || f > kSelectMaxF) {
        set_error("%s: d=%d or f=%d beyond the supported maximum", who, d, f);
        return CS_ERR_UNSUPPORTED;
    }
    return CS_OK;
}

cs_status check_params(const cs_select_params *params, const char *who) {
    if (!params) {
        set_error("%s: params is null", who);
        return CS_ERR_INVALID;
    }
    if (params->mode != CS_SEL_TOPK && params->mode != CS_SEL_THRESHOLD && params->mode != CS_SEL_EXACT) {
        set_error("%s: bad selection mode", who);
        return CS_ERR_INVALID;
    }
    if (params->hot < 0 || params->hot % 32 || (params->mode == CS_SEL_EXACT && params->hot)) {
        set_error("%s: hot must be a non-negative multiple of 32, and 0 in exact mode", who);
        return CS_ERR_INVALID;
    }
    if (params->mode == CS_SEL_EXACT && !(params->tau >= 0.f)) {
        set_error("%s: the exact mode's magnitude cut tau must be >= 0", who);
        return CS_ERR_INVALID;
    }
    return CS_OK;
}

// Enqueue the plan directly when the caller is capturing (or on the legacy
// stream), else replay its cached graph, capturing it on first use.
// With copy nodes (p.io_src / p.io_dst), *io_refused is set instead when the
// nodes of a captured graph cannot be located; the caller then stages its
// host buffers with copies.
template <typename Enq>
cs_status run_cached(const StackPlan &p, cudaStream_t sm, cudaStream_t sp_key, const char *who, Enq enq,
                     bool *io_refused = nullptr) {
    cudaStreamCaptureStatus cap = cudaStreamCaptureStatusNone;
    if (sm) {
        cudaError_t e = cudaStreamIsCapturing(sm, &cap);
        if (e != cudaSuccess) return cuda_fail(e, who);
    }
    if (cap == cudaStreamCaptureStatusActive || !sm) {
        cudaError_t e = enq();
        return e == cudaSuccess ? CS_OK : cuda_fail(e, who);
    }
    int dev = 0;
    cudaGetDevice(&dev);
    const std::string key = plan_key(p, sp_key, dev);
    std::lock_guard<std::mutex> lock(g_mu);
    const bool io = p.io_src || p.io_dst;
    if (io && g_io_nodes_unusable) {
        *io_refused = true;
        return CS_OK;
    }
    auto it = g_cache.find(key);
    if (it == g_cache.end()) {
        if (g_cache.size() >= kMaxCached) clear_cache_locked();
        cudaGraph_t graph = nullptr;
        cudaError_t e = cudaStreamBeginCapture(sm, cudaStreamCaptureModeThreadLocal);
        if (e != cudaSuccess) return cuda_fail(e, who);
        const cudaError_t ee = enq();
        e = cudaStreamEndCapture(sm, &graph);
        if (ee != cudaSuccess) {
            if (graph) cudaGraphDestroy(graph);
            return cuda_fail(ee, who);
        }
        if (e != cudaSuccess) return cuda_fail(e, who);
        CacheEntry ce;
        ce.device = dev;
        ce.graph = graph;
        e = cudaGraphInstantiate(&ce.exec, graph, 0);
        if (e == cudaSuccess && io) e = find_io_nodes(ce);
        if (e != cudaSuccess) {
            destroy_entry(ce);
            return cuda_fail(e, who);
        }
        if (io && ((p.io_src && !ce.io_node[0]) || (p.io_dst && !ce.io_node[1]))) {
            destroy_entry(ce);
            g_io_nodes_unusable = true;
            *io_refused = true;
            return CS_OK;
        }
        if (!io) {
            cudaGraphDestroy(ce.graph);
            ce.graph = nullptr;
        }
        it = g_cache.emplace(key, ce).first;
    }
    cudaError_t e = io ? update_io(it->second, p) : cudaSuccess;
    if (e == cudaSuccess) e = cudaGraphLaunch(it->second.exec, sm);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, who);
}

// Where a pointer given for x or y lives: device (or managed) memory is used
// in place, page-locked host memory is staged through the workspace, and
// pageable host memory is refused (its copies cannot be asynchronous).
cs_status io_kind(const void *ptr, bool *host, void **mapped, const char *who, const char *what) {
    cudaPointerAttributes at = {};
    cudaError_t e = cudaPointerGetAttributes(&at, ptr);
    *mapped = nullptr;
    if (e != cudaSuccess) {
        cudaGetLastError();
        set_error("%s: %s: %s", who, what, cudaGetErrorString(e));
        return CS_ERR_INVALID;
    }
    if (at.type == cudaMemoryTypeHost) {
        *host = true;
        *mapped = at.devicePointer;   // null when the memory is not mapped
        return CS_OK;
    }
    if (at.type == cudaMemoryTypeDevice || at.type == cudaMemoryTypeManaged) {
        *host = false;
        return CS_OK;
    }
    set_error("%s: %s is pageable host memory; use device or page-locked host memory", who, what);
    return CS_ERR_INVALID;
}

}  // namespace

extern "C" {

cs_status cs_decode_stack(const cs_ffn_layer *layers, const cs_predictor *preds, int L, float *x,
                          float resid_scale, const cs_select_params *params, cs_stack_mode mode,
                          cs_stream_t s_main, cs_stream_t s_pred, void *ws, size_t ws_bytes,
                          int32_t *trace_count, int32_t *trace_idx) {
    const char *who = "cs_decode_stack";
    if (L < 1 || !layers || !params || !x || (reinterpret_cast<uintptr_t>(x) & 3u)) {
        set_error("cs_decode_stack: L >= 1, layers, params and x are required");
        return CS_ERR_INVALID;
    }
    cs_status st = check_params(params, who);
    if (st != CS_OK) return st;
    if (mode != CS_STACK_SEQUENTIAL && mode != CS_STACK_LOOKAHEAD) {
        set_error("cs_decode_stack: bad stack mode");
        return CS_ERR_INVALID;
    }
    const bool exact = params->mode == CS_SEL_EXACT;
    if (!exact && !preds) {
        set_error("cs_decode_stack: predictors are required unless the selection is exact");
        return CS_ERR_INVALID;
    }
    st = check_models(layers, preds, L, exact, params->hot, who);
    if (st != CS_OK) return st;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) {
        set_error("cs_decode_stack: workspace is null or not 256-byte aligned");
        return CS_ERR_WORKSPACE;
    }
    bool x_host = false;
    void *xm = nullptr;
    st = io_kind(x, &x_host, &xm, who, "x");
    if (st != CS_OK) return st;
    const int d = layers[0].d, f = layers[0].f, r = exact ? 1 : preds[0].r;
    StackPlan p;
    p.layers = layers; p.preds = preds; p.L = L; p.d = d; p.f = f; p.r = r;
    p.scale = resid_scale; p.sel = *params; p.mode = mode;
    p.ws = static_cast<char *>(ws);
    p.lay = ws_layout(d, f, r, 1, device_sm_count());
    p.trace_count = trace_count; p.trace_idx = trace_idx;
    if (ws_bytes < p.lay.total) {
        set_error("cs_decode_stack: workspace too small: %zu bytes given, %zu needed", ws_bytes, p.lay.total);
        return CS_ERR_WORKSPACE;
    }
    // a host x goes through the workspace's staging row
    p.x = x_host ? reinterpret_cast<float *>(p.ws + p.lay.io_x) : x;

    cudaStream_t sm = (cudaStream_t)s_main;
    cudaStream_t sp = (cudaStream_t)s_pred;
    const bool two = mode == CS_STACK_LOOKAHEAD && !exact && sp && sp != sm;
    auto enq = [&]() {
        Events E;
        return enqueue_stack(p, sm, two ? sp : sm, E);
    };
    if (x_host && xm && graph_io_enabled()) {
        // the graph's first and last nodes read and write it in place
        p.io_src = static_cast<const float *>(xm);
        p.io_dst = static_cast<float *>(xm);
        bool refused = false;
        st = run_cached(p, sm, two ? sp : nullptr, who, enq, &refused);
        if (st != CS_OK || !refused) return st;
        p.io_src = nullptr;
        p.io_dst = nullptr;
    }
    const size_t x_bytes = sizeof(float) * (size_t)d;
    if (x_host) {
        cudaError_t e = cudaMemcpyAsync(p.x, x, x_bytes, cudaMemcpyHostToDevice, sm);
        if (e != cudaSuccess) return cuda_fail(e, "cs_decode_stack(x copy in)");
    }
    st = run_cached(p, sm, two ? sp : nullptr, who, enq);
    if (st != CS_OK || !x_host) return st;
    cudaError_t e = cudaMemcpyAsync(x, p.x, x_bytes, cudaMemcpyDeviceToHost, sm);
    return e == cudaSuccess ? CS_OK : cuda_fail(e, "cs_decode_stack(x copy out)");
}

cs_status cs_decode_layer(const cs_ffn_layer *layer, const cs_predictor *pred, const float *x, float *y,
                          const cs_select_params *params, void *ws, size_t ws_bytes, cs_stream_t stream,
                          int32_t *idx, int32_t *count) {
    const char *who = "cs_decode_layer";
    if (!layer || !params || !x || !y || (reinterpret_cast<uintptr_t>(x) & 3u) ||
        (reinterpret_cast<uintptr_t>(y) & 3u) || (!idx) != (!count) || (reinterpret_cast<uintptr_t>(idx) & 3u) ||
        (reinterpret_cast<uintptr_t>(count) & 3u)) {
        set_error("cs_decode_layer: layer, params, x and y are required (4-byte aligned); idx and count "
                  "are given together or not at all");
        return CS_ERR_INVALID;
    }
    cs_status st = check_params(params, who);
    if (st != CS_OK) return st;
    const bool exact = params->mode == CS_SEL_EXACT;
    if (!exact && !pred) {
        set_error("cs_decode_layer: a predictor is required unless the selection is exact");
        return CS_ERR_INVALID;
    }
    st = check_models(layer, pred, 1, exact, params->hot, who);
    if (st != CS_OK) return st;
    if (!ws || (reinterpret_cast<uintptr_t>(ws) & 255u)) {
        set_error("cs_decode_layer: workspace is null or not 256-byte aligned");
        return CS_ERR_WORKSPACE;
    }
    bool x_host = false, y_host = false;
    void *xm = nullptr, *ym = nullptr;
    st = io_kind(x, &x_host, &xm, who, "x");
    if (st != CS_OK) return st;
    st = io_kind(y, &y_host, &ym, who, "y");
    if (st != CS_OK) return st;

    const int d = layer->d, f = layer->f, r = exact ? 1 : pred->r;
    StackPlan p;
    p.layers = layer; p.preds = pred; p.L = 1; p.d = d; p.f = f; p.r = r;
    p.scale = 1.f; p.sel = *params; p.mode = CS_STACK_SEQUENTIAL;
    p.ws = static_cast<char *>(ws);
    p.lay = ws_layout(d, f, r, 1, device_sm_count());
    p.trace_count = count; p.trace_idx = idx;
    p.layer_only = true;
    if (ws_bytes < p.lay.total) {
        set_error("cs_decode_layer: workspace too small: %zu bytes given, %zu needed", ws_bytes, p.lay.total);
        return CS_ERR_WORKSPACE;
    }
    // host x and y go through the stack's ping-pong buffer and the y staging
    // buffer
    p.x = x_host ? reinterpret_cast<float *>(p.ws + p.lay.st_x) : const_cast<float *>(x);
    p.y = y_host ? reinterpret_cast<float *>(p.ws + p.lay.io_y) : y;

    cudaStream_t s = (cudaStream_t)stream;
    auto enq = [&]() { return enqueue_layer(p, s); };
    if ((x_host || y_host) && (!x_host || xm) && (!y_host || ym) && graph_io_enabled()) {
        // the graph's first and last nodes read x and write y in place
        p.io_src = x_host ? static_cast<const float *>(xm) : nullptr;
        p.io_dst = y_host ? static_cast<float *>(ym) : nullptr;
        bool refused = false;
        st = run_cached(p, s, nullptr, who, enq, &refused);
        if (st != CS_OK || !refused) return st;
        p.io_src = nullptr;
        p.io_dst = nullptr;
    }
    const size_t xy_bytes = sizeof(float) * (size_t)d;
    if (x_host) {
        cudaError_t e = cudaMemcpyAsync(p.x, x, xy_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cs_decode_layer(x copy)");
    }
    st = run_cached(p, s, nullptr, who, enq);
    if (st != CS_OK) return st;
    if (y_host) {
        cudaError_t e = cudaMemcpyAsync(y, p.y, xy_bytes, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "cs_decode_layer(y copy)");
    }
    return CS_OK;
}

cs_status cs_decode_attention(const cs_attn_layer *layer, const cs_predictor *pred, const float *x, float *y,
                              const cs_select_params *params, const void *k_cache, const void *v_cache,
                              int seq_len, void *ws, size_t ws_bytes, cs_stream_t stream, int32_t *heads,
                              int32_t *count) {
    const char *who = "cs_decode_attention";
    if (!layer || !pred || !params || !x || !y || x == y || (reinterpret_cast<uintptr_t>(x) & 3u) ||
        (reinterpret_cast<uintptr_t>(y) & 3u) || (!heads) != (!count) ||
        (reinterpret_cast<uintptr_t>(heads) & 3u) || (reinterpret_cast<uintptr_t>(count) & 3u)) {
        set_error("cs_decode_attention: layer, pred, params, x and y are required (4-byte aligned, y not x); "
                  "heads and count are given together or not at all");
        return CS_ERR_INVALID;
    }
    cs_status st = check_params(params, who);
    if (st != CS_OK) return st;
    if (params->mode == CS_SEL_EXACT || params->hot != 0) {
        set_error("cs_decode_attention: the heads are chosen by top-k or a threshold on the predictor's "
                  "scores, without a hot prefix");
        return CS_ERR_INVALID;
    }
    const AttnCall c{*layer, k_cache, v_cache, seq_len, ws, ws_bytes};
    st = attn_check(c, who);
    if (st != CS_OK) return st;
    const int d = layer->d, H = layer->n_heads;
    if (pred->d != d || pred->f != H) {
        set_error("cs_decode_attention: the predictor must score the %d heads from the d = %d inputs", H, d);
        return CS_ERR_INVALID;
    }
    st = attn_check_ws(c, who);
    if (st != CS_OK) return st;
    if (!pred_ok(*pred, d, H, pred->r)) {
        set_error("cs_decode_attention: the predictor must score the %d heads from the d = %d inputs, with "
                  "16-byte aligned weights and pitches", H, d);
        return CS_ERR_INVALID;
    }
    bool x_host = false, y_host = false;
    void *xm = nullptr, *ym = nullptr;
    st = io_kind(x, &x_host, &xm, who, "x");
    if (st != CS_OK) return st;
    st = io_kind(y, &y_host, &ym, who, "y");
    if (st != CS_OK) return st;
    if (!x_host && (reinterpret_cast<uintptr_t>(x) & 15u)) {
        set_error("cs_decode_attention: a device x must be 16-byte aligned");
        return CS_ERR_INVALID;
    }

    StackPlan p;
    p.layers = nullptr; p.preds = pred; p.L = 1; p.d = d; p.f = H; p.r = pred->r;
    p.scale = 1.f; p.sel = *params; p.mode = CS_STACK_SEQUENTIAL;
    p.ws = static_cast<char *>(ws);
    p.lay = ws_layout(d, H, pred->r, 1, device_sm_count());
    p.trace_count = count; p.trace_idx = heads;
    p.layer_only = true;
    p.attn = &c;
    if (ws_bytes < p.lay.total) {
        set_error("cs_decode_attention: workspace too small: %zu bytes given, %zu needed", ws_bytes, p.lay.total);
        return CS_ERR_WORKSPACE;
    }
    // host x and y go through the workspace's x row and y staging row
    p.x = x_host ? reinterpret_cast<float *>(p.ws + p.lay.st_x) : const_cast<float *>(x);
    p.y = y_host ? reinterpret_cast<float *>(p.ws + p.lay.io_y) : y;

    cudaStream_t s = (cudaStream_t)stream;
    auto enq = [&]() { return enqueue_attention(p, s); };
    if ((x_host || y_host) && (!x_host || xm) && (!y_host || ym) && graph_io_enabled()) {
        p.io_src = x_host ? static_cast<const float *>(xm) : nullptr;
        p.io_dst = y_host ? static_cast<float *>(ym) : nullptr;
        bool refused = false;
        st = run_cached(p, s, nullptr, who, enq, &refused);
        if (st != CS_OK || !refused) return st;
        p.io_src = nullptr;
        p.io_dst = nullptr;
    }
    const size_t xy_bytes = sizeof(float) * (size_t)d;
    if (x_host) {
        cudaError_t e = cudaMemcpyAsync(p.x, x, xy_bytes, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "cs_decode_attention(x copy)");
    }
    st = run_cached(p, s, nullptr, who, enq);
    if (st != CS_OK) return st;
    if (y_host) {
        cudaError_t e = cudaMemcpyAsync(y, p.y, xy_bytes, cudaMemcpyDeviceToHost, s);
        if (e != cudaSuccess) return cuda_fail(e, "cs_decode_attention(y copy)");
    }
    return CS_OK;
}

cs_status cs_stack_release(void) {
    std::lock_guard<std::mutex> lock(g_mu);
    clear_cache_locked();
    return CS_OK;
}

}  // extern "C"
