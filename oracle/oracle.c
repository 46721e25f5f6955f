/*
 * CPU oracle for the contextual-sparsity feed-forward decode step.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * CPU-baseline leg of the benchmark load this file's library.  It shares no
 * code, header or table with the CUDA library, and the CUDA library never
 * calls it.
 *
 * Everything is the plain definition, evaluated in fp64 in ascending index
 * order with no blocking or fusion.  fp16 and bf16 weights are decoded from
 * their bit patterns by the decoders below.  Selection decisions are taken on
 * fp32 scores (the precision the scores are produced in), as the caller
 * passes them.
 *
 * Sources (web pages; section names as printed on them):
 *  [P1] "Contextual Sparsity and Activation Predictors"
 *  [P2] "Contextual Sparsity: Activation-Aware LLM Inference and the Deja Vu
 *       Paradigm"
 *  [P3] "Activation sparsity" (wikillm concept page)
 *
 * Parity pins for every function are in tests/test_oracle_*.py: closed forms
 * (permutation weights, the identity predictor), hand-worked fixtures in
 * tests/golden/, brute force on tiny inputs and exact invariants.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { ORC_F32 = 0, ORC_F16 = 1, ORC_BF16 = 2 };

/* ---------------------------------------------------------------- decoding */

/* IEEE binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int m = h & 0x3FF;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-14 * 2^-10 */
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(m | 0x400), e - 25);    /* (1024+m) * 2^(e-15-10) */
    return sign ? -v : v;
}

/* bfloat16: the upper 16 bits of an IEEE binary32. */
static double decode_bf16(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static double elem(const void *base, int dtype, size_t i)
{
    switch (dtype) {
    case ORC_F32: return (double)((const float *)base)[i];
    case ORC_F16: return decode_f16(((const uint16_t *)base)[i]);
    default:      return decode_bf16(((const uint16_t *)base)[i]);
    }
}

double orc_decode(const void *base, int dtype, long i) { return elem(base, dtype, (size_t)i); }
void orc_decode_array(const void *base, int dtype, long n, double *out)
{
    for (long i = 0; i < n; i++)
        out[i] = elem(base, dtype, (size_t)i);
}

/* -------------------------------------------------------------- predictor */

/*
 * Low-rank predictor, [P2] "The Prediction Problem" (SparsityPredictor):
 * two bias-free linear maps with a ReLU between them,
 *     h_i = max(0, sum_t P_down[i,t] x_t),   s_j = sum_i P_up[j,i] h_i.
 * The page ends with a sigmoid.  It is monotone, so it does not change a
 * top-k set; the scores here are the logits and a threshold lives on that
 * scale ([P3] "Implementation sketch": the threshold is on the predictor's
 * own score scale).
 */
void orc_predict(int d, int r, int f, int dtype,
                 const void *p_down, long ld_down, const void *p_up, long ld_up,
                 const double *x, double *h, double *s)
{
    #pragma omp parallel for schedule(static)
    for (int i = 0; i < r; i++) {
        double acc = 0.0;
        for (int t = 0; t < d; t++)
            acc += elem(p_down, dtype, (size_t)i * ld_down + t) * x[t];
        h[i] = acc > 0.0 ? acc : 0.0;
    }
    #pragma omp parallel for schedule(static)
    for (int j = 0; j < f; j++) {
        double acc = 0.0;
        for (int i = 0; i < r; i++)
            acc += elem(p_up, dtype, (size_t)j * ld_up + i) * h[i];
        s[j] = acc;
    }
}

/* ------------------------------------------------------------------- FFN */

typedef struct {
    int d, f, dtype;
    long ld;
    const void *w_gate;    /* [f, ld] row j = gate row of neuron j          */
    const void *w_up;      /* [f, ld] or NULL (gate-only ReLU FFN)          */
    const void *w_down_t;  /* [f, ld] row j = column j of W_down            */
    const float *bias;     /* [f] or NULL                                    */
    int act;               /* ORC_ACT_RELU or ORC_ACT_SILU                   */
} orc_layer;

enum { ORC_ACT_RELU = 0, ORC_ACT_SILU = 1 };

/*
 * The gate's activation: relu(g) = max(g, 0), or silu(g) = g / (1 + e^-g)
 * ([P2] "The SiLU/GELU Challenge: TurboSparse": down(silu(gate x) * up x);
 * [P2] "The Empirical Foundation": SiLU layers are only functionally sparse).
 */
static double gate_act(int act, double g)
{
    if (act == ORC_ACT_SILU)
        return g / (1.0 + exp(-g));
    return g > 0.0 ? g : 0.0;
}

/* Gate pre-activation g_j = w_gate_j . x + b_j. */
static double preact_j(const orc_layer *L, const double *x, int j)
{
    double acc = 0.0;
    for (int t = 0; t < L->d; t++)
        acc += elem(L->w_gate, L->dtype, (size_t)j * L->ld + t) * x[t];
    if (L->bias)
        acc += (double)L->bias[j];
    return acc;
}

/*
 * Neuron activation a_j = act(w_gate_j . x + b_j) * (w_up_j . x if the layer
 * has an up projection, else 1), act = relu or silu.  ReLU gate-only FFN:
 * [P2] "The Empirical Foundation" (ReLU layers) and [P1] first section;
 * ReLUfied SwiGLU and SwiGLU: [P2] "The SiLU/GELU Challenge: TurboSparse"
 * (down(act(gate x) * up x)).
 */
static double act_j(const orc_layer *L, const double *x, int j)
{
    double g = preact_j(L, x, j);
    double a = gate_act(L->act, g);
    if (L->w_up) {
        double u = 0.0;
        for (int t = 0; t < L->d; t++)
            u += elem(L->w_up, L->dtype, (size_t)j * L->ld + t) * x[t];
        a *= u;
    }
    return a;
}

void orc_preact(const orc_layer *L, const double *x, double *pre)
{
    #pragma omp parallel for schedule(static)
    for (int j = 0; j < L->f; j++)
        pre[j] = preact_j(L, x, j);
}

/*
 * Gathered sparse FFN, [P2] "The Prediction Problem" (sparse_mlp_forward):
 * take the gate rows and down columns of the listed neurons only,
 *     y = sum_{m} a_{idx[m]} * W_down[:, idx[m]].
 * W_down is stored transposed, so column j of W_down is row j of w_down_t.
 * Terms are added in list order (ascending neuron id for every list this
 * library produces).  Out-of-range ids are a caller error: returns -1.
 */
int orc_ffn(const orc_layer *L, const double *x, const int32_t *idx, int n, double *y)
{
    for (int m = 0; m < n; m++)
        if (idx[m] < 0 || idx[m] >= L->f)
            return -1;
    double *a = (double *)malloc(sizeof(double) * (size_t)(n > 0 ? n : 1));
    if (!a)
        return -2;
    #pragma omp parallel for schedule(static)
    for (int m = 0; m < n; m++)
        a[m] = act_j(L, x, idx[m]);
    #pragma omp parallel for schedule(static)
    for (int i = 0; i < L->d; i++) {
        double acc = 0.0;
        for (int m = 0; m < n; m++)
            acc += a[m] * elem(L->w_down_t, L->dtype, (size_t)idx[m] * L->ld + i);
        y[i] = acc;
    }
    free(a);
    return 0;
}

/* Dense FFN: every neuron, ascending. */
int orc_dense_ffn(const orc_layer *L, const double *x, double *y)
{
    int32_t *all = (int32_t *)malloc(sizeof(int32_t) * (size_t)(L->f > 0 ? L->f : 1));
    if (!all)
        return -2;
    for (int j = 0; j < L->f; j++)
        all[j] = j;
    int rc = orc_ffn(L, x, all, L->f, y);
    free(all);
    return rc;
}

/* ------------------------------------------------------------- selection */

/*
 * Ranking rule for top-k (the pages' topk leaves ties open; see the design
 * notes): larger score first; equal scores by lower neuron id; NaN ranks
 * below every number; -0 and +0 are equal.
 */
typedef struct { float s; int32_t j; } scored;

static int ranks_before(const scored *a, const scored *b)
{
    int an = isnan(a->s), bn = isnan(b->s);
    if (an != bn)
        return bn;                       /* a number beats a NaN */
    if (!an && a->s != b->s)
        return a->s > b->s;
    return a->j < b->j;
}

static int cmp_rank(const void *pa, const void *pb)
{
    const scored *a = (const scored *)pa, *b = (const scored *)pb;
    if (ranks_before(a, b)) return -1;
    if (ranks_before(b, a)) return 1;
    return 0;
}

static int cmp_i32(const void *pa, const void *pb)
{
    int32_t a = *(const int32_t *)pa, b = *(const int32_t *)pb;
    return (a > b) - (a < b);
}

/*
 * Top-k selection, [P2] "The Prediction Problem" (scores.topk(k)) and [P1]
 * "The predictor and its budget" (the top-k scores form the predicted set):
 * sort all neurons by the ranking rule, keep the first min(k, f), and return
 * them in ascending neuron order.  Returns the count.
 */
int orc_select_topk(const float *s, int f, int k, int32_t *idx)
{
    if (k < 0) k = 0;
    if (k > f) k = f;
    scored *v = (scored *)malloc(sizeof(scored) * (size_t)(f > 0 ? f : 1));
    if (!v)
        return -2;
    for (int j = 0; j < f; j++) { v[j].s = s[j]; v[j].j = j; }
    qsort(v, (size_t)f, sizeof(scored), cmp_rank);
    for (int m = 0; m < k; m++)
        idx[m] = v[m].j;
    free(v);
    qsort(idx, (size_t)k, sizeof(int32_t), cmp_i32);
    return k;
}

/*
 * Threshold selection, [P3] "Implementation sketch" (predict_active returns
 * scores >= threshold): {j : s_j >= tau}, ascending.  NaN never passes.
 */
int orc_select_threshold(const float *s, int f, float tau, int32_t *idx)
{
    int n = 0;
    for (int j = 0; j < f; j++)
        if (s[j] >= tau)
            idx[n++] = j;
    return n;
}

/*
 * Exact mask: the neurons whose gate pre-activation is positive, i.e. the
 * ones ReLU lets through ([P1] first section: knowing whether a neuron is
 * inactive means computing its gate row).  Strictly greater than zero.
 */
int orc_select_positive(const float *pre, int f, int32_t *idx)
{
    int n = 0;
    for (int j = 0; j < f; j++)
        if (pre[j] > 0.0f)
            idx[n++] = j;
    return n;
}

/*
 * Hot-prefix selection ([P2] "Kernel-Level Implementation": neurons sorted by
 * how often they fire; [P1] "Static locality: hot and cold neurons": a few
 * neurons fire for most inputs).  With the layout sorted hottest first, the
 * first `hot` neurons are always taken and only the tail is predicted:
 * s_tail holds the scores of neurons hot .. hot + f_tail - 1.  The result is
 * 0 .. hot-1 followed by hot + (the tail's own selection: top-k or
 * threshold), ascending.  Returns the count.
 */
int orc_select_hot(const float *s_tail, int f_tail, int hot, int mode, int k, float tau, int32_t *idx)
{
    if (hot < 0 || f_tail < 0)
        return -1;
    for (int j = 0; j < hot; j++)
        idx[j] = j;
    int n = mode == 0 ? orc_select_topk(s_tail, f_tail, k, idx + hot)
                      : orc_select_threshold(s_tail, f_tail, tau, idx + hot);
    if (n < 0)
        return n;
    for (int m = 0; m < n; m++)
        idx[hot + m] += hot;
    return hot + n;
}

/*
 * Magnitude selection for functional sparsity ([P2] "The Empirical
 * Foundation": under SiLU, neurons whose outputs are non-zero but too small to
 * matter): {j : |act(g_j)| > tau} from the fp32 gate pre-activations,
 * ascending; the gate's activation is evaluated in fp64.  NaN never passes.
 * With relu and tau = 0 this is the exact mask {j : g_j > 0}.
 */
int orc_select_magnitude(const float *pre, int f, int act, float tau, int32_t *idx)
{
    int n = 0;
    for (int j = 0; j < f; j++) {
        double a = fabs(gate_act(act, (double)pre[j]));
        if (a > (double)tau)
            idx[n++] = j;
    }
    return n;
}

/* --------------------------------------------------------------- batches */

/*
 * Batch union, [P1] "When it breaks": the layer must read the union of the
 * tokens' active sets.  umask = OR of the B masks (bit j%32 of word j/32);
 * uidx = its set bits ascending.  Returns |U|.
 */
int orc_union(const uint32_t *masks, int B, int f, uint32_t *umask, int32_t *uidx)
{
    int words = (f + 31) / 32;
    int n = 0;
    for (int w = 0; w < words; w++) {
        uint32_t u = 0;
        for (int b = 0; b < B; b++)
            u |= masks[(size_t)b * words + w];
        if (w == words - 1 && (f & 31))
            u &= (1u << (f & 31)) - 1u;
        umask[w] = u;
        for (int bit = 0; bit < 32; bit++)
            if ((u >> bit) & 1u)
                uidx[n++] = w * 32 + bit;
    }
    return n;
}

/* --------------------------------------------------- recall and precision */

/*
 * [P1] "Precision, recall, and which error hurts": recall = |P & E| / |E|,
 * precision = |P & E| / |P|, with P the predicted set and E the exact one.
 * An empty denominator gives 1 (nothing to miss / nothing wrong).
 */
void orc_recall_precision(const int32_t *pred, int np, const int32_t *exact, int ne, int f,
                          double *recall, double *precision)
{
    unsigned char *inE = (unsigned char *)calloc((size_t)(f > 0 ? f : 1), 1);
    int hit = 0;
    for (int m = 0; m < ne; m++)
        inE[exact[m]] = 1;
    for (int m = 0; m < np; m++)
        hit += inE[pred[m]];
    free(inE);
    *recall = ne ? (double)hit / ne : 1.0;
    *precision = np ? (double)hit / np : 1.0;
}

/* ------------------------------------------------------------- attention */

typedef struct {
    int d, n_heads, d_head, dtype;
    const void *w_q;     /* [H * d_head, d]: rows h*d_head .. of head h          */
    const void *w_o_t;   /* [H * d_head, d]: W_o transposed, the same row blocks  */
} orc_attn;

/*
 * Head-sparse attention for one token ([P1] first section: a small,
 * input-dependent set of heads; [P2] "The Empirical Foundation": 20-30% of
 * heads contribute per token; [P2] "Implications for System Design": select
 * the heads to compute per token).  For each listed head h, over a cache of S
 * keys and values k_{h,i}, v_{h,i} ([H, S, d_head] each):
 *     q = W_q[h] x,  s_i = q . k_{h,i} / sqrt(d_head),  p = softmax(s),
 *     o = sum_i p_i v_{h,i},  y += W_o[:, h] o.
 * Heads in list order; ids outside [0, H) are a caller error (-1).
 */
int orc_attention(const orc_attn *A, const double *x, const int32_t *heads, int n, const void *kc,
                  const void *vc, int S, double *y)
{
    const int d = A->d, dh = A->d_head, H = A->n_heads;
    for (int t = 0; t < d; t++)
        y[t] = 0.0;
    if (n <= 0)
        return 0;
    if (S < 1)
        return -1;
    double *q = (double *)malloc(sizeof(double) * (size_t)dh);
    double *o = (double *)malloc(sizeof(double) * (size_t)dh);
    double *sc = (double *)malloc(sizeof(double) * (size_t)S);
    if (!q || !o || !sc)
        return -2;
    int rc = 0;
    const double scale = 1.0 / sqrt((double)dh);
    for (int m = 0; m < n && rc == 0; m++) {
        const int h = heads[m];
        if (h < 0 || h >= H) {
            rc = -1;
            break;
        }
        for (int c = 0; c < dh; c++) {
            double acc = 0.0;
            for (int t = 0; t < d; t++)
                acc += elem(A->w_q, A->dtype, ((size_t)h * dh + c) * d + t) * x[t];
            q[c] = acc;
        }
        double mx = -INFINITY;
        for (int i = 0; i < S; i++) {
            double acc = 0.0;
            for (int c = 0; c < dh; c++)
                acc += q[c] * elem(kc, A->dtype, ((size_t)h * S + i) * dh + c);
            sc[i] = acc * scale;
            if (sc[i] > mx) mx = sc[i];
        }
        double z = 0.0;
        for (int i = 0; i < S; i++) {
            sc[i] = exp(sc[i] - mx);
            z += sc[i];
        }
        for (int c = 0; c < dh; c++) {
            double acc = 0.0;
            for (int i = 0; i < S; i++)
                acc += sc[i] * elem(vc, A->dtype, ((size_t)h * S + i) * dh + c);
            o[c] = acc / z;
        }
        for (int t = 0; t < d; t++) {
            double acc = 0.0;
            for (int c = 0; c < dh; c++)
                acc += o[c] * elem(A->w_o_t, A->dtype, ((size_t)h * dh + c) * d + t);
            y[t] += acc;
        }
    }
    free(q); free(o); free(sc);
    return rc;
}

/* ------------------------------------------------------------------ stack */

typedef struct {
    int d, r, f, dtype;
    long ld_down, ld_up;
    const void *p_down;    /* [r, ld_down] */
    const void *p_up;      /* [f, ld_up]   */
} orc_pred;

enum { ORC_SEL_TOPK = 0, ORC_SEL_THRESHOLD = 1, ORC_SEL_EXACT = 2 };
enum { ORC_SEQUENTIAL = 0, ORC_LOOKAHEAD = 1 };

/*
 * A stack of L layers on the residual stream, [P1] "The predictor and its
 * budget": x_{l+1} = x_l + c * FFN_l(x_l).
 *   sequential: layer l's set is selected from P_l(x_l).
 *   look-ahead: layer l's set is selected from P_l(x_{l-1}) -- the predictor
 *               of the next layer reads the current layer's input -- and
 *               layer 0 from P_0(x_0).
 *   exact:      layer l's set is {j : |act(pre-activation)| > tau} at x_l
 *               (no predictor; mode is ignored): {j : pre-activation > 0}
 *               for relu at tau = 0.
 * Scores are rounded to fp32 before the selection decision.  x is updated in
 * place.  hot > 0: the layout is sorted hottest first, neurons 0 .. hot-1
 * are always taken and each predictor scores only the other f - hot neurons
 * (orc_select_hot).  Optional traces: per-layer counts [L], index lists
 * [L, f] and fp32 scores [L, f] (scores of the predictor that chose layer l's
 * set: its first f - hot entries when hot > 0).
 */
int orc_stack(int L, const orc_layer *layers, const orc_pred *preds, int mode, int sel_mode,
              int k, float tau, int hot, double resid_scale, double *x,
              int32_t *trace_count, int32_t *trace_idx, float *trace_scores)
{
    if (L <= 0)
        return 0;
    int d = layers[0].d;
    int fmax = 0, rmax = 1;
    for (int l = 0; l < L; l++) {
        if (layers[l].f > fmax) fmax = layers[l].f;
        if (preds && preds[l].r > rmax) rmax = preds[l].r;
    }
    double *xprev = (double *)malloc(sizeof(double) * d);
    double *y = (double *)malloc(sizeof(double) * d);
    double *h = (double *)malloc(sizeof(double) * rmax);
    double *s = (double *)malloc(sizeof(double) * fmax);
    float *s32 = (float *)malloc(sizeof(float) * fmax);
    int32_t *idx = (int32_t *)malloc(sizeof(int32_t) * fmax);
    if (!xprev || !y || !h || !s || !s32 || !idx)
        return -2;
    int rc = 0;
    memcpy(xprev, x, sizeof(double) * d);
    for (int l = 0; l < L && rc == 0; l++) {
        const orc_layer *Ly = &layers[l];
        int n;
        if (sel_mode == ORC_SEL_EXACT) {
            for (int j = 0; j < Ly->f; j++)
                s32[j] = (float)preact_j(Ly, x, j);
            n = orc_select_magnitude(s32, Ly->f, Ly->act, tau, idx);
        } else {
            const orc_pred *P = &preds[l];
            const double *xin = (mode == ORC_LOOKAHEAD && l > 0) ? xprev : x;
            /* the predictor scores the tail only: P->f == Ly->f - hot */
            if (hot < 0 || P->f != Ly->f - hot) {
                rc = -1;
                break;
            }
            orc_predict(P->d, P->r, P->f, P->dtype, P->p_down, P->ld_down, P->p_up, P->ld_up,
                        xin, h, s);
            for (int j = 0; j < P->f; j++)
                s32[j] = (float)s[j];
            n = orc_select_hot(s32, P->f, hot, sel_mode == ORC_SEL_TOPK ? 0 : 1, k, tau, idx);
        }
        if (trace_count) trace_count[l] = n;
        if (trace_idx) memcpy(trace_idx + (size_t)l * fmax, idx, sizeof(int32_t) * (size_t)n);
        if (trace_scores)
            memcpy(trace_scores + (size_t)l * fmax, s32,
                   sizeof(float) * (size_t)(sel_mode == ORC_SEL_EXACT ? Ly->f : preds[l].f));
        rc = orc_ffn(Ly, x, idx, n, y);
        memcpy(xprev, x, sizeof(double) * d);
        for (int i = 0; i < d; i++)
            x[i] = x[i] + resid_scale * y[i];
    }
    free(xprev); free(y); free(h); free(s); free(s32); free(idx);
    return rc;
}

/* Number of OpenMP threads the oracle runs with (1 without OpenMP). */
#ifdef _OPENMP
#include <omp.h>
int orc_threads(void) { return omp_get_max_threads(); }
void orc_set_threads(int n) { if (n > 0) omp_set_num_threads(n); }
#else
int orc_threads(void) { return 1; }
void orc_set_threads(int n) { (void)n; }
#endif
