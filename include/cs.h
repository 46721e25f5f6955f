/*
 * cs.h -- C ABI of the contextual-sparsity sparse FFN library (GB300, sm_103a).
 *
 * The method (sources are web pages, cited by title and section):
 *  [P1] "Contextual Sparsity and Activation Predictors"
 *  [P2] "Contextual Sparsity: Activation-Aware LLM Inference and the Deja Vu
 *       Paradigm"
 *  [P3] "Activation sparsity" (wikillm concept page)
 *
 * A per-layer low-rank predictor scores every FFN neuron; a top-k or threshold
 * selection turns the scores into an ascending list of active neurons; only
 * those neurons' gate (and up) rows and their columns of W_down are read:
 *     y = sum_{j in A} relu(w_gate_j . x + b_j) * (w_up_j . x) * W_down[:, j].
 *
 * Conventions for every call
 *  - Pointers named as device buffers must be device memory of the current
 *    CUDA device (cudaMalloc / torch).  Struct headers are host memory.  The
 *    caller owns every buffer; the library allocates nothing on these calls.
 *  - Calls are asynchronous and stream-ordered on the stream given (NULL =
 *    legacy default stream).  CS_OK means "validated and enqueued".
 *  - Argument errors are reported synchronously and nothing is enqueued.
 *    Errors found on the device (an index out of range, a bad count) set bits
 *    in the workspace error word (see cs_get_device_error); the kernels skip
 *    or clamp the offending item instead of dereferencing it.
 *  - Weights are neuron-major: row j of w_gate, w_up and w_down_t belongs to
 *    neuron j (w_down_t is W_down transposed, so each neuron's down vector is
 *    a contiguous row).  Rows have a stride of `ld` elements; ld * elem_size
 *    must be a multiple of 16 bytes and every base pointer 16-byte aligned.
 *    Padding elements beyond d are never used.
 *  - x, scores, pre-activations and y are fp32; weights are fp32, fp16 or
 *    bf16; all dot products accumulate in fp32.
 *  - No exception crosses this boundary.  Thread safety: calls on different
 *    workspaces may run concurrently; one workspace serves one stream at a
 *    time.
 */
#ifndef CS_H
#define CS_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *cs_stream_t; /* the same type as cudaStream_t */

typedef enum cs_status {
    CS_OK = 0,
    CS_ERR_INVALID = 1,     /* bad argument; nothing was enqueued              */
    CS_ERR_CUDA = 2,        /* a CUDA runtime call failed (see cs_last_error)  */
    CS_ERR_UNSUPPORTED = 3, /* valid, but outside the supported sizes          */
    CS_ERR_TIMEOUT = 4,     /* a bounded device wait gave up                   */
    CS_ERR_WORKSPACE = 5    /* workspace missing, misaligned or too small      */
} cs_status;

/* Bits of the device error word (cs_get_device_error). */
#define CS_DEVERR_INDEX   0x1u /* a neuron id outside [0, f) was skipped        */
#define CS_DEVERR_COUNT   0x2u /* a count outside [0, f] was clamped            */
#define CS_DEVERR_TIMEOUT 0x4u /* a bounded wait inside a kernel gave up        */

typedef enum cs_dtype { CS_F32 = 0, CS_F16 = 1, CS_BF16 = 2 } cs_dtype;

typedef enum cs_sel_mode {
    CS_SEL_TOPK = 0,      /* the k best scores, lower id wins ties [P2 "The Prediction Problem"] */
    CS_SEL_THRESHOLD = 1, /* scores >= tau [P3 "Implementation sketch", predict_active]          */
    CS_SEL_EXACT = 2      /* |act(gate pre-activation)| > tau (relu, 0: g > 0), no predictor [P1] */
} cs_sel_mode;

typedef enum cs_stack_mode {
    CS_STACK_SEQUENTIAL = 0, /* layer l's set predicted from x_l                             */
    CS_STACK_LOOKAHEAD = 1   /* layer l+1's set predicted from x_l on a second stream [P1]    */
} cs_stack_mode;

/*
 * Low-rank predictor of one layer, [P2] "The Prediction Problem"
 * (SparsityPredictor): scores = P_up relu(P_down x), both maps bias-free.
 * The page's final sigmoid is monotone and is not applied: scores are logits.
 *   p_down: [r, ld_down] device, row i = i-th bottleneck unit (ld_down >= d)
 *   p_up:   [f, ld_up]   device, row j = neuron j (ld_up >= r)
 * ld_* = 0 means dense rows (d and r).
 */
typedef struct cs_predictor {
    int d, r, f;
    cs_dtype dtype;
    int ld_down, ld_up;
    const void *p_down;
    const void *p_up;
} cs_predictor;

/*
 * The gate's activation: CS_ACT_RELU, relu(g) = max(g, 0); CS_ACT_SILU,
 * silu(g) = g / (1 + e^-g), for SiLU-family models, which are only
 * functionally sparse ([P2] "The Empirical Foundation": outputs non-zero but
 * too small to matter; "The SiLU/GELU Challenge: TurboSparse").
 */
typedef enum cs_act { CS_ACT_RELU = 0, CS_ACT_SILU = 1 } cs_act;

/*
 * One FFN layer, neuron-major.  w_up == NULL gives the gate-only FFN
 * (a_j = act(g_j)); otherwise the gated FFN of [P2] "The SiLU/GELU Challenge:
 * TurboSparse" (a_j = act(g_j) * (w_up_j . x): ReLUfied SwiGLU with relu,
 * SwiGLU with silu).  g_j = w_gate_j . x + bias_j (bias may be NULL).  All
 * three matrices share dtype and ld.
 */
typedef struct cs_ffn_layer {
    int d, f;
    cs_dtype dtype;
    int ld;
    const void *w_gate;   /* [f, ld] device                       */
    const void *w_up;     /* [f, ld] device or NULL               */
    const void *w_down_t; /* [f, ld] device; row j = W_down[:, j] */
    const float *bias;    /* [f] device fp32 or NULL              */
    cs_act act;           /* the gate's activation                */
} cs_ffn_layer;

/*
 * Selection: k for CS_SEL_TOPK (clamped to [0, f]); tau for CS_SEL_THRESHOLD
 * (and, for CS_SEL_EXACT in cs_decode_stack / cs_decode_layer, the magnitude
 * cut |act(g_j)| > tau, tau >= 0; see cs_exact_ffn).
 * hot: size of an always-on prefix for a frequency-sorted layout ([P2]
 * "Kernel-Level Implementation", neurons pre-sorted by how often they fire;
 * [P1] "Static locality: hot and cold neurons").  Neurons 0 .. hot-1 are
 * always taken and only the tail is scored and selected (k and tau apply to
 * the tail).  0 for a plain selection; otherwise a multiple of 32.  Not
 * allowed with CS_SEL_EXACT.
 */
typedef struct cs_select_params {
    cs_sel_mode mode;
    int k;
    float tau;
    int hot;
} cs_select_params;

/* ------------------------------------------------------------ utilities */

const char *cs_version(void);
const char *cs_status_string(cs_status s);
/* Text of the last error on this host thread ("" if none). */
const char *cs_last_error(void);

/*
 * Workspace bytes for calls with model width d, f neurons, predictor rank r
 * and up to B tokens per call, on the current device (the size depends on its
 * SM count).  One workspace serves every call below, including
 * cs_decode_stack.  The workspace is caller-owned device memory, 256-byte
 * aligned, and must be initialised once with cs_workspace_init.
 */
size_t cs_workspace_size(int d, int f, int r, int B);
cs_status cs_workspace_init(void *ws, size_t ws_bytes, cs_stream_t stream);

/*
 * Reads (and with clear != 0 also resets) the device error word.  Waits for
 * `stream`; this is the only call that synchronises.
 */
cs_status cs_get_device_error(void *ws, cs_stream_t stream, int clear, uint32_t *code_out);

/*
 * Layout step for a frequency-sorted layout ([P2] "Kernel-Level
 * Implementation": neurons pre-sorted by firing frequency; [P1] "Static
 * locality: hot and cold neurons"): dst[i, :] = src[perm[i], :] for
 * i < rows, `cols` elements of `dtype` per row.  Apply the same perm to the
 * rows of w_gate, w_up, w_down_t and the bias (cols = 1, fp32), and perm + H
 * (rows = f - H) to p_up for a hot prefix of H neurons; y is unchanged up to
 * summation order.  src [src_rows, ld_src] and dst [rows, ld_dst] are
 * device memory and must not overlap; perm [rows] int32 device.  A perm
 * entry outside [0, src_rows) gives a zero row.
 */
cs_status cs_permute_rows(const void *src, int src_rows, int ld_src, const int32_t *perm, int rows, int cols,
                          cs_dtype dtype, void *dst, int ld_dst, cs_stream_t stream);

/*
 * The frequency-sorted order on the host: perm[i] = the neuron of rank i,
 * most frequent first, equal frequencies by lower id (NaN counts as the
 * lowest frequency).  freq [f] and perm [f] are host memory (may be NULL
 * when f == 0); synchronous.
 */
cs_status cs_hot_order(const float *freq, int f, int32_t *perm);

/*
 * Layout step: dst[c, r] = src[r, c] with dtype conversion (round to nearest
 * even).  Turns a user's W_down [d, f] into w_down_t [f, ld_dst].  src is
 * [rows, ld_src], dst is [cols, ld_dst]; both device.  Neuron-major rows
 * keep each neuron's data contiguous ([P2] "Kernel-Level Implementation":
 * indexing into row-major weights breaks coalescing).
 */
cs_status cs_pack_transpose(const void *src, cs_dtype src_dtype, int rows, int cols, int ld_src,
                            void *dst, cs_dtype dst_dtype, int ld_dst, cs_stream_t stream);

/* ------------------------------------------------------------- hot path */

/*
 * Predictor, [P2] "The Prediction Problem": scores[b, j] = sum_i P_up[j, i] *
 * relu(sum_t P_down[i, t] x[b, t]).
 *   x:      [B, d] fp32 device;   scores: [B, f] fp32 device (output).
 * B >= 1.
 */
cs_status cs_predict(const cs_predictor *pred, const float *x, int B, float *scores,
                     void *ws, size_t ws_bytes, cs_stream_t stream);

/*
 * Selection per token row, [P2] "The Prediction Problem" (top-k) and [P3]
 * "Implementation sketch" (threshold).  With H = params->hot:
 *   scores: [B, f] fp32 device -- the scores of neurons H .. H + f - 1.
 *   idx:    [B, H + f] int32 device (output): row b holds count[b] ascending
 *           ids, 0 .. H-1 first.
 *   count:  [B] int32 device (output): H + the tail's count.
 *   mask:   [B, ceil((H + f)/32)] uint32 device or NULL (output): bit j%32 of
 *           word j/32 set iff neuron j is selected.
 * TOPK: the min(k, f) best scores; higher score first, equal scores by lower
 * id, -0 == +0, NaN below every number.  THRESHOLD: {j : s_j >= tau}, NaN
 * never passes.  mode CS_SEL_EXACT is not a score selection: use
 * cs_exact_ffn.  f <= 49152; H a non-negative multiple of 32.
 */
cs_status cs_select(const float *scores, int B, int f, const cs_select_params *params,
                    int32_t *idx, int32_t *count, uint32_t *mask,
                    void *ws, size_t ws_bytes, cs_stream_t stream);

/*
 * Gathered sparse FFN, [P2] "The Prediction Problem" (sparse_mlp_forward):
 * for every token b, y[b] = sum_{m < count} a_{b, idx[m]} * w_down_t[idx[m], :]
 * with a_{b,j} = relu(w_gate_j . x_b + bias_j) (* w_up_j . x_b).  All B tokens
 * use the same list (batch union semantics, [P1] "When it breaks").
 *   x: [B, d] fp32 device;  y: [B, d] fp32 device (output, may not alias x).
 *   idx: [>= count] int32 device, ascending;  count: int32 device scalar.
 * The list stays on the device; no host synchronisation.  The reduction over
 * neurons runs in a fixed order, so results are bit-reproducible.
 */
cs_status cs_sparse_ffn(const cs_ffn_layer *layer, const float *x, int B, const int32_t *idx,
                        const int32_t *count, float *y, void *ws, size_t ws_bytes,
                        cs_stream_t stream);

/*
 * Exact-mask FFN for one token ([P1] first section: knowing which neurons are
 * inactive means computing every gate row).  Computes all pre-activations
 * g_j = w_gate_j . x + bias_j, selects A = {j : |act(g_j)| > tau} (the
 * functional-sparsity cut of [P2] "The Empirical Foundation"; for relu at
 * tau = 0 the exact mask {j : g_j > 0}), then
 * y = sum_{j in A} act(g_j) (* w_up_j . x) w_down_t[j, :].
 *   preact: [f] fp32 device (output);  idx: [f] int32 device (output);
 *   count: int32 device (output);  mask: [ceil(f/32)] uint32 device or NULL;
 *   y: [d] fp32 device (output);  tau >= 0.  The selection decides in fp32.
 */
cs_status cs_exact_ffn(const cs_ffn_layer *layer, const float *x, float *preact, int32_t *idx,
                       int32_t *count, uint32_t *mask, float *y, float tau,
                       void *ws, size_t ws_bytes, cs_stream_t stream);

/*
 * Batch union, [P1] "When it breaks": umask = OR of the B token masks;
 * uidx = its set bits ascending; ucount = |U|.
 *   masks: [B, ceil(f/32)] uint32 device;  umask: [ceil(f/32)] uint32 device;
 *   uidx: [f] int32 device;  ucount: int32 device scalar.
 * Bits at positions >= f in the last word are ignored.
 */
cs_status cs_union_mask(const uint32_t *masks, int B, int f, uint32_t *umask, int32_t *uidx,
                        int32_t *ucount, void *ws, size_t ws_bytes, cs_stream_t stream);

/*
 * Layer stack on the residual stream, [P1] "The predictor and its budget":
 * x_{l+1} = x_l + resid_scale * FFN_l(x_l, A_l) for l = 0..L-1, batch 1.
 *   SEQUENTIAL: A_l = select(P_l(x_l)).
 *   LOOKAHEAD:  A_l = select(P_l(x_{l-1})) (A_0 from x_0): the predictor and
 *               selection of layer l+1 run on s_pred while layer l's FFN runs
 *               on s_main.
 *   params->mode == CS_SEL_EXACT: A_l = {j : |act(g_j)| > params->tau} at x_l
 *               (g_j > 0 for relu at tau = 0); preds unused.
 *   x: [d] fp32, input x_0 and output x_L: device memory, or page-locked
 *      host memory (cudaHostAlloc, cudaHostRegister, torch pin_memory).  A
 *      host x is read by the graph's first kernel and written by its last
 *      through the buffer's device mapping (with asynchronous copies on s_main
 *      around the graph when it has none); x holds x_L once s_main has passed
 *      this call.  Pageable host memory is refused (CS_ERR_INVALID).
 *   layers, preds: host arrays of L structs (same d, f, r and dtype).
 *   trace_count: [L] int32 device or NULL; trace_idx: [L, f] int32 device or
 *   NULL -- per-layer selected counts and ascending ids.
 * The whole sequence is captured into a CUDA graph on the first call for a
 * given set of arguments and replayed afterwards (unless s_main is already
 * capturing, in which case the kernels are enqueued into the caller's
 * capture); a host x's address may change from call to call without a new
 * capture (the graph's two copy kernels are re-pointed).  The workspace must hold
 * cs_workspace_size(d, f, r, 1) bytes.
 */
cs_status cs_decode_stack(const cs_ffn_layer *layers, const cs_predictor *preds, int L, float *x,
                          float resid_scale, const cs_select_params *params, cs_stack_mode mode,
                          cs_stream_t s_main, cs_stream_t s_pred, void *ws, size_t ws_bytes,
                          int32_t *trace_count, int32_t *trace_idx);

/*
 * One decode step of one layer for one token, [P2] "The Prediction Problem"
 * (predictor, top-k, then the FFN over the chosen neurons only) and [P3]
 * "Implementation sketch" (predict the active set, then run the FFN on it):
 *     A = select(P(x)),  y = FFN(x, A)   (no residual).
 *   params->mode == CS_SEL_EXACT: A = {j : |act(g_j)| > params->tau} at x (g_j > 0
 *      for relu at tau = 0); pred may be NULL.
 *   x: [d] fp32 input;  y: [d] fp32 output.  Each may be device memory or
 *      page-locked host memory (cudaHostAlloc, cudaHostRegister, torch
 *      pin_memory).  A host x is read by the graph's first kernel and a
 *      host y written by its last, through the buffers' device mappings
 *      (staged with asynchronous copies on `stream` when they have none), so
 *      a host y holds the result once the stream has passed this call.
 *      Pageable host memory is refused (CS_ERR_INVALID).
 *   idx: [f] int32 device or NULL; count: int32 device scalar or NULL (both
 *      or neither) -- the selected ids, ascending, and their number.
 * The kernels are captured into a CUDA graph on the first call for a given
 * set of arguments and replayed afterwards; host addresses may change from
 * call to call without a new capture (the graph's copy kernels are
 * re-pointed).  A stream that is already capturing, or the legacy stream
 * (NULL), gets the kernels enqueued directly.  The workspace must hold
 * cs_workspace_size(d, f, r, 1) bytes.  This call uses the same workspace
 * regions as cs_decode_stack, so the two must not overlap on one workspace.
 */
cs_status cs_decode_layer(const cs_ffn_layer *layer, const cs_predictor *pred, const float *x, float *y,
                          const cs_select_params *params, void *ws, size_t ws_bytes, cs_stream_t stream,
                          int32_t *idx, int32_t *count);

/*
 * Attention weights of one layer for head-sparse decoding ([P1] first
 * section: a small, input-dependent set of heads; [P2] "The Empirical
 * Foundation": 20-30% of heads contribute per token; [P2] "Implications for
 * System Design": select the heads to compute per token).  Head h owns rows
 * h*d_head .. h*d_head + d_head - 1 of both matrices:
 *   w_q:   [n_heads * d_head, d] device, the query projection;
 *   w_o_t: [n_heads * d_head, d] device, the output projection transposed
 *          (row h*d_head + c is column h*d_head + c of W_o).
 * d a multiple of 16 / element size; d_head a power of two from 16 / element
 * size to 256; 16-byte aligned pointers.
 */
typedef struct cs_attn_layer {
    int d, n_heads, d_head;
    cs_dtype dtype;
    const void *w_q;
    const void *w_o_t;
} cs_attn_layer;

/*
 * Head-sparse attention for one token over a KV cache.  For each of the
 * count[0] heads listed in heads (ascending ids from cs_select over a
 * predictor with one output per head):
 *     q = W_q[h] x,  s_i = q . k_{h,i} / sqrt(d_head),  p = softmax(s),
 *     o = sum_i p_i v_{h,i},  y = sum_h W_o[:, h] o      (fp32 throughout).
 *   x: [d] fp32 device (16-byte aligned);  y: [d] fp32 device (output).
 *   k_cache, v_cache: [n_heads, seq_len, d_head] device in layer->dtype.
 *   1 <= seq_len <= 16384; n_heads <= the workspace's partial rows (the SM
 *   count).  The workspace is any cs_workspace_size(d, ...) workspace.
 * Ids outside [0, n_heads) are skipped and flagged (CS_DEVERR_INDEX); a count
 * outside [0, n_heads] is clamped and flagged (CS_DEVERR_COUNT).
 */
cs_status cs_sparse_attention(const cs_attn_layer *layer, const float *x, const int32_t *heads,
                              const int32_t *count, const void *k_cache, const void *v_cache, int seq_len,
                              float *y, void *ws, size_t ws_bytes, cs_stream_t stream);

/*
 * One token's head-sparse attention step in one call, [P1] first section (a
 * small, input-dependent set of heads) and [P2] "Implications for System
 * Design" (predict the heads, compute only those):
 *     H_sel = select(P(x)),  y = cs_sparse_attention(x, H_sel).
 *   pred: rank r, d = layer->d inputs, f = layer->n_heads outputs (one score
 *      per head).
 *   params: CS_SEL_TOPK or CS_SEL_THRESHOLD over the head scores, hot = 0
 *      (else CS_ERR_INVALID).
 *   x, y: [d] fp32, device memory (x 16-byte aligned) or page-locked host
 *      memory, read and written as in cs_decode_layer; y must not be x.
 *   k_cache, v_cache, seq_len: as cs_sparse_attention.
 *   heads: [n_heads] int32 device or NULL; count: int32 device scalar or NULL
 *      (both or neither) -- the chosen heads, ascending, and their number.
 * Predictor, selection and attention are captured into one CUDA graph per
 * argument set and replayed, as in cs_decode_layer (same capture and
 * host-buffer rules).  The workspace must hold cs_workspace_size(d, n_heads,
 * r, 1) bytes and meet cs_sparse_attention's bound on partial values; it
 * uses the same regions as cs_decode_layer and cs_decode_stack.
 */
cs_status cs_decode_attention(const cs_attn_layer *layer, const cs_predictor *pred, const float *x, float *y,
                              const cs_select_params *params, const void *k_cache, const void *v_cache,
                              int seq_len, void *ws, size_t ws_bytes, cs_stream_t stream, int32_t *heads,
                              int32_t *count);

/*
 * Fits a predictor's up map to its layer, [P2] "The Prediction Problem" (the
 * predictor is trained to reproduce which neurons the layer activates) and
 * [P1] "Precision, recall, and which error hurts".  With pred->p_down fixed,
 * pred->p_up is overwritten with the ridge regression of the gate
 * pre-activations g(x) = w_gate x + bias onto the bottleneck features
 * h(x) = relu(p_down x) over N calibration inputs:
 *     P_up = G^T H (H^T H + lambda I)^-1,  H = [h(x_n)] (N x r),  G = [g(x_n)] (N x f),
 * H and G in fp32, H^T H and H^T G summed in fp64, the solve in fp64, the
 * result rounded to pred->dtype.
 *   X: [N, d] fp32 device (16-byte aligned).  lambda >= 0 (absolute; the
 *   diagonal of H^T H grows with N).  pred->d and pred->f must equal the
 *   layer's; r <= 2048; N <= 65535.  scratch: cs_fit_scratch_size(d, f, r, N) device
 *   bytes, 256-byte aligned.
 * A setup call: it waits for `stream` before returning, and returns
 * CS_ERR_INVALID if H^T H + lambda I is not positive definite.
 */
size_t cs_fit_scratch_size(int d, int f, int r, int N);
cs_status cs_fit_predictor(const cs_ffn_layer *layer, cs_predictor *pred, const float *X, int N, double lambda,
                           void *scratch, size_t scratch_bytes, cs_stream_t stream);

/* Drops every cached stack and layer graph (waits for nothing; call when idle). */
cs_status cs_stack_release(void);

/*
 * cs_sparse_ffn without a workspace, for callers that cannot allocate device
 * memory (for example a plugin running inside a host framework that owns all
 * device allocations and gives it no allocator, or a path where a cudaMalloc
 * may not be issued).  The method's sources have no counterpart of this call.
 * Same arguments as cs_sparse_ffn minus the workspace.  It always runs the
 * CUDA-core gather kernel, so its y is bit-identical to cs_sparse_ffn's
 * wherever cs_sparse_ffn takes that kernel too (every fp32 layer, and every
 * batch below the tensor-core threshold of 4 tokens).  Where cs_sparse_ffn
 * takes the tensor-core path (fp16 / bf16, d a multiple of 64, 4 <= B <= 32)
 * the two agree within the library's tolerance (max |difference| / max |y|
 * below 2e-3) but not bit for bit.
 *
 * Scratch: a fixed device array inside the library (2^21 fp32 values, 8 MiB,
 * held by every GPU that loads the library until the process exits).  A call
 * needs (SM count) * B * roundup(d, 8) values; larger calls return
 * CS_ERR_UNSUPPORTED without enqueuing anything.  The call allocates nothing.
 * The first call in a CUDA context looks up the array's device address in
 * that context (cached per context afterwards), so make that first call
 * before any stream capture begins.
 * Every call shares the one array and it keeps the last call's contents
 * (each call rewrites all of what it reads): calls that overlap on the GPU,
 * on different streams or from different threads, race and must be ordered
 * by the caller.  Device-side error bits (bad ids, which are skipped as in
 * cs_sparse_ffn) are not reported by this entry point.
 */
cs_status cs_sparse_ffn_noalloc(const cs_ffn_layer *layer, const float *x, int B, const int32_t *idx,
                                const int32_t *count, float *y, cs_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* CS_H */
