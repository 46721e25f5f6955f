"""ctypes front end of the CPU oracle (``oracle/oracle.c``).

TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the CPU-baseline
leg of the benchmark use it.  The CUDA library never imports or calls it.

Functions take numpy arrays.  Weight arrays are in storage form: float32,
float16, or uint16 bit patterns for bf16, with a row stride ``ld`` in
elements.  Results are float64 (values) or int32 (index lists).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_OUT_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None

F32, F16, BF16 = 0, 1, 2
SEL_TOPK, SEL_THRESHOLD, SEL_EXACT = 0, 1, 2
SEQUENTIAL, LOOKAHEAD = 0, 1
ACT_RELU, ACT_SILU = 0, 1


def build(force: bool = False) -> str:
    """Compile liboracle.so with gcc (-O2, OpenMP).  Returns its path."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


class _Layer(C.Structure):
    _fields_ = [("d", C.c_int), ("f", C.c_int), ("dtype", C.c_int), ("ld", C.c_long),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_down_t", C.c_void_p),
                ("bias", C.c_void_p), ("act", C.c_int)]


class _Attn(C.Structure):
    _fields_ = [("d", C.c_int), ("n_heads", C.c_int), ("d_head", C.c_int), ("dtype", C.c_int),
                ("w_q", C.c_void_p), ("w_o_t", C.c_void_p)]


class _Pred(C.Structure):
    _fields_ = [("d", C.c_int), ("r", C.c_int), ("f", C.c_int), ("dtype", C.c_int),
                ("ld_down", C.c_long), ("ld_up", C.c_long),
                ("p_down", C.c_void_p), ("p_up", C.c_void_p)]


def lib():
    global _lib
    with _lock:
        if _lib is None:
            path = build()
            L = C.CDLL(path)
            P, I, D, F, LG = C.c_void_p, C.c_int, C.c_double, C.c_float, C.c_long
            L.orc_predict.argtypes = [I, I, I, I, P, LG, P, LG, P, P, P]
            L.orc_predict.restype = None
            L.orc_preact.argtypes = [C.POINTER(_Layer), P, P]
            L.orc_preact.restype = None
            L.orc_ffn.argtypes = [C.POINTER(_Layer), P, P, I, P]
            L.orc_ffn.restype = I
            L.orc_dense_ffn.argtypes = [C.POINTER(_Layer), P, P]
            L.orc_dense_ffn.restype = I
            L.orc_select_topk.argtypes = [P, I, I, P]
            L.orc_select_topk.restype = I
            L.orc_select_threshold.argtypes = [P, I, F, P]
            L.orc_select_threshold.restype = I
            L.orc_select_hot.argtypes = [P, I, I, I, I, F, P]
            L.orc_select_hot.restype = I
            L.orc_attention.argtypes = [C.POINTER(_Attn), P, P, I, P, P, I, P]
            L.orc_attention.restype = I
            L.orc_select_magnitude.argtypes = [P, I, I, F, P]
            L.orc_select_magnitude.restype = I
            L.orc_select_positive.argtypes = [P, I, P]
            L.orc_select_positive.restype = I
            L.orc_union.argtypes = [P, I, I, P, P]
            L.orc_union.restype = I
            L.orc_recall_precision.argtypes = [P, I, P, I, I, C.POINTER(D), C.POINTER(D)]
            L.orc_recall_precision.restype = None
            L.orc_stack.argtypes = [I, C.POINTER(_Layer), C.POINTER(_Pred), I, I, I, F, I, D, P,
                                    P, P, P]
            L.orc_stack.restype = I
            L.orc_decode.argtypes = [P, I, LG]
            L.orc_decode.restype = D
            L.orc_decode_array.argtypes = [P, I, LG, P]
            L.orc_decode_array.restype = None
            L.orc_threads.argtypes = []
            L.orc_threads.restype = I
            L.orc_set_threads.argtypes = [I]
            L.orc_set_threads.restype = None
            _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype=None):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=dtype) if dtype is not None else np.ascontiguousarray(a)


class Layer:
    """FFN layer in storage form.  Rows are neuron-major: w_gate, w_up and
    w_down_t are [f, ld]; row j of w_down_t is column j of W_down."""

    def __init__(self, d, f, dtype, w_gate, w_down_t, w_up=None, bias=None, ld=None, act=ACT_RELU):
        self.d, self.f, self.dtype = int(d), int(f), int(dtype)
        self.act = int(act)
        self.ld = int(ld if ld is not None else d)
        self.w_gate = _c(w_gate)
        self.w_down_t = _c(w_down_t)
        self.w_up = _c(w_up)
        self.bias = _c(bias, np.float32)
        for w in (self.w_gate, self.w_down_t, self.w_up):
            if w is not None and w.size < self.f * self.ld - (self.ld - self.d):
                raise ValueError("weight array too small for [f, ld]")

    def c(self):
        return _Layer(self.d, self.f, self.dtype, self.ld, _ptr(self.w_gate), _ptr(self.w_up),
                      _ptr(self.w_down_t), _ptr(self.bias), self.act)


class Predictor:
    def __init__(self, d, r, f, dtype, p_down, p_up, ld_down=None, ld_up=None):
        self.d, self.r, self.f, self.dtype = int(d), int(r), int(f), int(dtype)
        self.ld_down = int(ld_down if ld_down is not None else d)
        self.ld_up = int(ld_up if ld_up is not None else r)
        self.p_down = _c(p_down)
        self.p_up = _c(p_up)

    def c(self):
        return _Pred(self.d, self.r, self.f, self.dtype, self.ld_down, self.ld_up,
                     _ptr(self.p_down), _ptr(self.p_up))


def predict(P: Predictor, x):
    """(h [r], scores [f]) in fp64 for one token."""
    x = _c(x, np.float64)
    h = np.empty(P.r, np.float64)
    s = np.empty(P.f, np.float64)
    lib().orc_predict(P.d, P.r, P.f, P.dtype, _ptr(P.p_down), P.ld_down, _ptr(P.p_up), P.ld_up,
                      _ptr(x), _ptr(h), _ptr(s))
    return h, s


def preact(Ly: Layer, x):
    x = _c(x, np.float64)
    out = np.empty(Ly.f, np.float64)
    c = Ly.c()
    lib().orc_preact(C.byref(c), _ptr(x), _ptr(out))
    return out


def ffn(Ly: Layer, x, idx):
    x = _c(x, np.float64)
    idx = _c(idx, np.int32)
    y = np.empty(Ly.d, np.float64)
    c = Ly.c()
    rc = lib().orc_ffn(C.byref(c), _ptr(x), _ptr(idx), int(idx.size), _ptr(y))
    if rc != 0:
        raise ValueError(f"orc_ffn failed ({rc})")
    return y


def dense_ffn(Ly: Layer, x):
    x = _c(x, np.float64)
    y = np.empty(Ly.d, np.float64)
    c = Ly.c()
    rc = lib().orc_dense_ffn(C.byref(c), _ptr(x), _ptr(y))
    if rc != 0:
        raise ValueError(f"orc_dense_ffn failed ({rc})")
    return y


def select_topk(scores32, k):
    s = _c(scores32, np.float32)
    out = np.empty(max(s.size, 1), np.int32)
    n = lib().orc_select_topk(_ptr(s), int(s.size), int(k), _ptr(out))
    return out[:n].copy()


def select_threshold(scores32, tau):
    s = _c(scores32, np.float32)
    out = np.empty(max(s.size, 1), np.int32)
    n = lib().orc_select_threshold(_ptr(s), int(s.size), float(np.float32(tau)), _ptr(out))
    return out[:n].copy()


def select_positive(pre32):
    s = _c(pre32, np.float32)
    out = np.empty(max(s.size, 1), np.int32)
    n = lib().orc_select_positive(_ptr(s), int(s.size), _ptr(out))
    return out[:n].copy()


def select_hot(tail_scores32, hot, mode=SEL_TOPK, k=0, tau=0.0):
    """Hot-prefix selection: 0 .. hot-1, then hot + the tail's own top-k (or
    threshold) selection over the tail's fp32 scores."""
    s = _c(tail_scores32, np.float32)
    out = np.empty(max(int(hot) + s.size, 1), np.int32)
    n = lib().orc_select_hot(_ptr(s), int(s.size), int(hot), 0 if mode == SEL_TOPK else 1, int(k),
                             float(np.float32(tau)), _ptr(out))
    if n < 0:
        raise ValueError(f"orc_select_hot failed ({n})")
    return out[:n].copy()


def hot_order(freq):
    """The frequency-sorted layout's neuron order: most frequent first, equal
    frequencies by lower id (a stable sort on the negated frequencies)."""
    f = np.asarray(freq, np.float64)
    return np.argsort(-f, kind="stable").astype(np.int32)


def permute_rows(arr, perm):
    """Rows of a storage array in the order perm: out[i] = arr[perm[i]]."""
    return np.ascontiguousarray(np.asarray(arr)[np.asarray(perm, np.int64)])


def select_magnitude(pre32, act, tau):
    """Functional sparsity: {j : |act(g_j)| > tau} from fp32 pre-activations."""
    s = _c(pre32, np.float32)
    out = np.empty(max(s.size, 1), np.int32)
    n = lib().orc_select_magnitude(_ptr(s), int(s.size), int(act), float(np.float32(tau)), _ptr(out))
    return out[:n].copy()


def fit_predictor(Ly: Layer, P: Predictor, X, lam):
    """The up map fitted to a layer: with P_down fixed, the ridge regression of
    the gate pre-activations g(x) = W_gate x + b onto the bottleneck features
    h(x) = relu(P_down x) over the calibration inputs X [N, d],
        P_up = argmin_P  sum_n |P h(x_n) - g(x_n)|^2 + lam |P|_F^2
             = G^T H (H^T H + lam I)^-1        (fp64, [f, r]),
    with H = [h(x_n)]_n and G = [g(x_n)]_n.  Matrix products and the solve are
    numpy's; the weights come through the oracle's own bit decoders."""
    X = np.asarray(X, np.float64)
    pd = decode(P.p_down, P.dtype).reshape(P.r, P.ld_down)[:, :P.d]
    wg = decode(Ly.w_gate, Ly.dtype).reshape(Ly.f, Ly.ld)[:, :Ly.d]
    b = np.zeros(Ly.f) if Ly.bias is None else Ly.bias.astype(np.float64)
    H = np.maximum(X @ pd.T, 0.0)
    G = X @ wg.T + b
    A = H.T @ H + float(lam) * np.eye(P.r)
    return np.linalg.solve(A, H.T @ G).T


class AttnLayer:
    """Head-sparse attention weights in storage form: w_q and w_o_t are
    [H * d_head, d]; row block h holds head h (w_o_t is W_o transposed)."""

    def __init__(self, d, n_heads, d_head, dtype, w_q, w_o_t):
        self.d, self.n_heads, self.d_head, self.dtype = int(d), int(n_heads), int(d_head), int(dtype)
        self.w_q = _c(w_q)
        self.w_o_t = _c(w_o_t)

    def c(self):
        return _Attn(self.d, self.n_heads, self.d_head, self.dtype, _ptr(self.w_q), _ptr(self.w_o_t))


def attention(A: AttnLayer, x, heads, k_cache, v_cache):
    """y [d] (fp64) of head-sparse attention over the listed heads; caches are
    [H, S, d_head] storage arrays."""
    x = _c(x, np.float64)
    h = _c(heads, np.int32)
    kc, vc = _c(k_cache), _c(v_cache)
    S = kc.shape[1]
    y = np.empty(A.d, np.float64)
    c = A.c()
    rc = lib().orc_attention(C.byref(c), _ptr(x), _ptr(h), int(h.size), _ptr(kc), _ptr(vc), int(S), _ptr(y))
    if rc != 0:
        raise ValueError(f"orc_attention failed ({rc})")
    return y


def union(masks, f):
    m = _c(masks, np.uint32)
    B = m.shape[0]
    words = (f + 31) // 32
    umask = np.empty(words, np.uint32)
    uidx = np.empty(max(f, 1), np.int32)
    n = lib().orc_union(_ptr(m), int(B), int(f), _ptr(umask), _ptr(uidx))
    return umask, uidx[:n].copy()


def recall_precision(pred_idx, exact_idx, f):
    p = _c(pred_idx, np.int32)
    e = _c(exact_idx, np.int32)
    r, q = C.c_double(), C.c_double()
    lib().orc_recall_precision(_ptr(p), int(p.size), _ptr(e), int(e.size), int(f),
                               C.byref(r), C.byref(q))
    return r.value, q.value


def stack(layers, preds, x, *, mode=SEQUENTIAL, sel_mode=SEL_TOPK, k=0, tau=0.0,
          resid_scale=0.1, trace=False, hot=0):
    """Run an L-layer stack.  Returns x_L (fp64) and, with trace=True, a dict
    of per-layer counts, index lists and fp32 scores."""
    L = len(layers)
    x = np.array(x, dtype=np.float64, copy=True)
    larr = (_Layer * L)(*[l.c() for l in layers])
    parr = (_Pred * L)(*[p.c() for p in preds]) if preds is not None else None
    fmax = max(l.f for l in layers)
    cnt = np.zeros(L, np.int32) if trace else None
    tidx = np.zeros((L, fmax), np.int32) if trace else None
    tsc = np.zeros((L, fmax), np.float32) if trace else None
    rc = lib().orc_stack(L, larr, parr, int(mode), int(sel_mode), int(k), float(tau), int(hot),
                         float(resid_scale), _ptr(x), _ptr(cnt), _ptr(tidx), _ptr(tsc))
    if rc != 0:
        raise ValueError(f"orc_stack failed ({rc})")
    if not trace:
        return x
    return x, {"count": cnt, "idx": [tidx[l, :cnt[l]].copy() for l in range(L)], "scores": tsc}


def decode(arr, dtype):
    """Decode a storage array to fp64 with the oracle's own bit decoders."""
    a = np.ascontiguousarray(arr)
    out = np.empty(a.size, np.float64)
    if a.size:
        lib().orc_decode_array(_ptr(a.reshape(-1)), int(dtype), int(a.size), _ptr(out))
    return out.reshape(a.shape)


def threads() -> int:
    return lib().orc_threads()


def set_threads(n: int) -> None:
    lib().orc_set_threads(int(n))
