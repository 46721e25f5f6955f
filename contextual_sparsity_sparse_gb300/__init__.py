"""Python binding of the contextual-sparsity sparse FFN library (libcs.so).

Argument marshalling only: every step of the path runs in the library's CUDA
kernels.  PyTorch provides device memory and streams.  The functions carry the
C ABI's names (include/cs.h) and raise :class:`CsError` on a non-OK status.
There is no fallback: if libcs.so is missing, importing the binding's loader
raises.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

from . import build as _build

_lock = threading.Lock()
_lib = None

CS_F32, CS_F16, CS_BF16 = 0, 1, 2
CS_SEL_TOPK, CS_SEL_THRESHOLD, CS_SEL_EXACT = 0, 1, 2
CS_STACK_SEQUENTIAL, CS_STACK_LOOKAHEAD = 0, 1
CS_ACT_RELU, CS_ACT_SILU = 0, 1
CS_DEVERR_INDEX, CS_DEVERR_COUNT, CS_DEVERR_TIMEOUT = 0x1, 0x2, 0x4

_TORCH_DT = {torch.float32: CS_F32, torch.float16: CS_F16, torch.bfloat16: CS_BF16}

# every symbol include/cs.h declares
EXPORTS = ["cs_version", "cs_status_string", "cs_last_error", "cs_workspace_size",
           "cs_workspace_init", "cs_get_device_error", "cs_pack_transpose", "cs_predict",
           "cs_select", "cs_sparse_ffn", "cs_exact_ffn", "cs_union_mask", "cs_decode_stack",
           "cs_stack_release", "cs_sparse_ffn_noalloc", "cs_decode_layer", "cs_permute_rows",
           "cs_hot_order", "cs_fit_scratch_size", "cs_fit_predictor", "cs_sparse_attention",
           "cs_decode_attention"]


class CsError(RuntimeError):
    def __init__(self, status, msg):
        super().__init__(f"{msg} (status {status})")
        self.status = status


class _Pred(C.Structure):
    _fields_ = [("d", C.c_int), ("r", C.c_int), ("f", C.c_int), ("dtype", C.c_int),
                ("ld_down", C.c_int), ("ld_up", C.c_int), ("p_down", C.c_void_p),
                ("p_up", C.c_void_p)]


class _Layer(C.Structure):
    _fields_ = [("d", C.c_int), ("f", C.c_int), ("dtype", C.c_int), ("ld", C.c_int),
                ("w_gate", C.c_void_p), ("w_up", C.c_void_p), ("w_down_t", C.c_void_p),
                ("bias", C.c_void_p), ("act", C.c_int)]


class _Attn(C.Structure):
    _fields_ = [("d", C.c_int), ("n_heads", C.c_int), ("d_head", C.c_int), ("dtype", C.c_int),
                ("w_q", C.c_void_p), ("w_o_t", C.c_void_p)]


class _Sel(C.Structure):
    _fields_ = [("mode", C.c_int), ("k", C.c_int), ("tau", C.c_float), ("hot", C.c_int)]


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libcs.so (built by ``build()``); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            path = library_path()
            if not os.path.exists(path):
                raise ImportError(f"CUDA library {path} is missing; run "
                                  "contextual_sparsity_sparse_gb300.build.build() first")
            L = C.CDLL(path)
            P, I, S, U = C.c_void_p, C.c_int, C.c_size_t, C.c_uint32
            L.cs_version.restype = C.c_char_p
            L.cs_status_string.argtypes = [I]
            L.cs_status_string.restype = C.c_char_p
            L.cs_last_error.restype = C.c_char_p
            L.cs_workspace_size.argtypes = [I, I, I, I]
            L.cs_workspace_size.restype = S
            L.cs_workspace_init.argtypes = [P, S, P]
            L.cs_get_device_error.argtypes = [P, P, I, C.POINTER(U)]
            L.cs_pack_transpose.argtypes = [P, I, I, I, I, P, I, I, P]
            L.cs_predict.argtypes = [C.POINTER(_Pred), P, I, P, P, S, P]
            L.cs_select.argtypes = [P, I, I, C.POINTER(_Sel), P, P, P, P, S, P]
            L.cs_sparse_ffn.argtypes = [C.POINTER(_Layer), P, I, P, P, P, P, S, P]
            L.cs_exact_ffn.argtypes = [C.POINTER(_Layer), P, P, P, P, P, P, C.c_float, P, S, P]
            L.cs_union_mask.argtypes = [P, I, I, P, P, P, P, S, P]
            L.cs_decode_stack.argtypes = [C.POINTER(_Layer), C.POINTER(_Pred), I, P, C.c_float,
                                          C.POINTER(_Sel), I, P, P, P, S, P, P]
            L.cs_sparse_ffn_noalloc.argtypes = [C.POINTER(_Layer), P, I, P, P, P, P]
            L.cs_decode_layer.argtypes = [C.POINTER(_Layer), C.POINTER(_Pred), P, P, C.POINTER(_Sel),
                                          P, S, P, P, P]
            L.cs_permute_rows.argtypes = [P, I, I, P, I, I, I, P, I, P]
            L.cs_hot_order.argtypes = [P, I, P]
            L.cs_sparse_attention.argtypes = [C.POINTER(_Attn), P, P, P, P, P, I, P, P, S, P]
            L.cs_decode_attention.argtypes = [C.POINTER(_Attn), C.POINTER(_Pred), P, P, C.POINTER(_Sel),
                                              P, P, I, P, S, P, P, P]
            L.cs_fit_scratch_size.argtypes = [I, I, I, I]
            L.cs_fit_scratch_size.restype = S
            L.cs_fit_predictor.argtypes = [C.POINTER(_Layer), C.POINTER(_Pred), P, I, C.c_double, P, S, P]
            for name in ("cs_workspace_init", "cs_get_device_error", "cs_pack_transpose",
                         "cs_predict", "cs_select", "cs_sparse_ffn", "cs_exact_ffn",
                         "cs_union_mask", "cs_decode_stack", "cs_stack_release",
                         "cs_sparse_ffn_noalloc", "cs_decode_layer", "cs_permute_rows", "cs_hot_order",
                         "cs_fit_predictor", "cs_sparse_attention", "cs_decode_attention"):
                getattr(L, name).restype = I
            _lib = L
    return _lib


def _check(status):
    if status != 0:
        L = lib()
        raise CsError(status, f"{L.cs_status_string(status).decode()}: {L.cs_last_error().decode()}")


def _ptr(t):
    if t is None:
        return None
    if not t.is_cuda:
        raise ValueError("expected a CUDA tensor")
    return t.data_ptr()


def _stream(s):
    if s is None:
        return torch.cuda.current_stream().cuda_stream
    return s.cuda_stream if hasattr(s, "cuda_stream") else int(s)


def _dt(t):
    return _TORCH_DT[t.dtype]


class Predictor:
    """p_down [r, ld_down], p_up [f, ld_up]; d is the used width of p_down."""

    def __init__(self, p_down, p_up, d=None, r=None):
        self.p_down, self.p_up = p_down, p_up
        self.r, ldd = p_down.shape
        self.f, ldu = p_up.shape
        self.d = int(d if d is not None else ldd)
        if r is not None and r != self.r:
            raise ValueError("r does not match p_down")
        self.c = _Pred(self.d, self.r, self.f, _dt(p_down), ldd, ldu, _ptr(p_down), _ptr(p_up))


class FfnLayer:
    """Neuron-major layer: w_gate, w_up, w_down_t are [f, ld]; d is the used
    width (default ld).  w_up None gives the gate-only ReLU FFN."""

    def __init__(self, w_gate, w_down_t, w_up=None, bias=None, d=None, act=CS_ACT_RELU):
        self.w_gate, self.w_down_t, self.w_up, self.bias = w_gate, w_down_t, w_up, bias
        self.f, ld = w_gate.shape
        self.d = int(d if d is not None else ld)
        self.act = int(act)
        self.c = _Layer(self.d, self.f, _dt(w_gate), ld, _ptr(w_gate), _ptr(w_up), _ptr(w_down_t),
                        _ptr(bias), self.act)


def select_params(mode, k=0, tau=0.0, hot=0):
    """hot: an always-on prefix of neurons for a frequency-sorted layout (a
    multiple of 32); k and tau then apply to the tail (see include/cs.h)."""
    return _Sel(int(mode), int(k), float(tau), int(hot))


class Workspace:
    """Device workspace sized by cs_workspace_size and initialised once."""

    def __init__(self, d, f, r, B=1, device=None, stream=None):
        n = lib().cs_workspace_size(int(d), int(f), int(r), int(B))
        if n == 0:
            raise ValueError("bad workspace dimensions")
        self.nbytes = n
        self.buf = torch.empty(n + 256, dtype=torch.uint8, device=device or "cuda")
        base = self.buf.data_ptr()
        self.ptr = (base + 255) & ~255
        _check(lib().cs_workspace_init(self.ptr, self.nbytes, _stream(stream)))


def cs_version() -> str:
    return lib().cs_version().decode()


def cs_workspace_size(d, f, r, B=1) -> int:
    return int(lib().cs_workspace_size(int(d), int(f), int(r), int(B)))


def cs_get_device_error(ws: Workspace, stream=None, clear=False) -> int:
    v = C.c_uint32(0)
    _check(lib().cs_get_device_error(ws.ptr, _stream(stream), int(bool(clear)), C.byref(v)))
    return v.value


def cs_pack_transpose(src, dst, rows=None, cols=None, stream=None):
    """dst[c, r] = src[r, c] (with dtype conversion).  src [rows, ld_src],
    dst [cols, ld_dst]."""
    rows = src.shape[0] if rows is None else rows
    cols = src.shape[1] if cols is None else cols
    _check(lib().cs_pack_transpose(_ptr(src), _dt(src), int(rows), int(cols), src.shape[1],
                                   _ptr(dst), _dt(dst), dst.shape[1], _stream(stream)))


def cs_predict(pred: Predictor, x, scores, ws: Workspace, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    _check(lib().cs_predict(C.byref(pred.c), _ptr(x), B, _ptr(scores), ws.ptr, ws.nbytes,
                            _stream(stream)))


def cs_select(scores, params, idx, count, mask=None, ws: Workspace | None = None, stream=None):
    B, f = (scores.shape if scores.dim() == 2 else (1, scores.shape[0]))
    _check(lib().cs_select(_ptr(scores), B, f, C.byref(params), _ptr(idx), _ptr(count),
                           _ptr(mask), ws.ptr if ws else None, ws.nbytes if ws else 0,
                           _stream(stream)))


def cs_sparse_ffn(layer: FfnLayer, x, idx, count, y, ws: Workspace, stream=None):
    B = x.shape[0] if x.dim() == 2 else 1
    _check(lib().cs_sparse_ffn(C.byref(layer.c), _ptr(x), B, _ptr(idx), _ptr(count), _ptr(y),
                               ws.ptr, ws.nbytes, _stream(stream)))


def cs_sparse_ffn_noalloc(layer: FfnLayer, x, idx, count, y, stream=None):
    """cs_sparse_ffn without a workspace (see include/cs.h): scratch comes from
    a fixed array inside the library, so nothing is allocated."""
    B = x.shape[0] if x.dim() == 2 else 1
    _check(lib().cs_sparse_ffn_noalloc(C.byref(layer.c), _ptr(x), B, _ptr(idx), _ptr(count),
                                       _ptr(y), _stream(stream)))


def cs_exact_ffn(layer: FfnLayer, x, preact, idx, count, y, ws: Workspace, mask=None, stream=None,
                 tau=0.0):
    """tau: the magnitude cut |act(g_j)| > tau (0 with relu: the exact mask g_j > 0)."""
    _check(lib().cs_exact_ffn(C.byref(layer.c), _ptr(x), _ptr(preact), _ptr(idx), _ptr(count),
                              _ptr(mask), _ptr(y), float(tau), ws.ptr, ws.nbytes, _stream(stream)))


def cs_union_mask(masks, f, umask, uidx, ucount, ws: Workspace | None = None, stream=None):
    B = masks.shape[0]
    _check(lib().cs_union_mask(_ptr(masks), B, int(f), _ptr(umask), _ptr(uidx), _ptr(ucount),
                               ws.ptr if ws else None, ws.nbytes if ws else 0, _stream(stream)))


class StackArgs:
    """The layer and predictor arrays of a stack, marshalled once, for
    repeated cs_decode_stack calls."""

    def __init__(self, layers, preds):
        self.L = len(layers)
        self.layers = (_Layer * self.L)(*[l.c for l in layers])
        self.preds = (_Pred * self.L)(*[p.c for p in preds]) if preds is not None else None


def cs_decode_stack(layers, preds, x, resid_scale, params, mode, ws: Workspace, s_main=None,
                    s_pred=None, trace_count=None, trace_idx=None):
    """x_0 -> x_L in place (see include/cs.h).  x may be a CUDA tensor or a
    pinned CPU tensor.  layers may also be a StackArgs (preds then unused)."""
    sa = layers if isinstance(layers, StackArgs) else StackArgs(layers, preds)
    sp = None if s_pred is None else _stream(s_pred)
    d = sa.layers[0].d
    _check(lib().cs_decode_stack(sa.layers, sa.preds, sa.L, _io_ptr(x, d), float(resid_scale), C.byref(params),
                                 int(mode), _stream(s_main), sp, ws.ptr, ws.nbytes,
                                 _ptr(trace_count), _ptr(trace_idx)))


def _io_ptr(t, n):
    """x or y of cs_decode_layer / cs_decode_stack: a CUDA tensor or a pinned CPU tensor, fp32,
    contiguous, holding at least n values (the library itself refuses
    pageable host memory)."""
    if t.dtype != torch.float32 or not t.is_contiguous() or t.numel() < n:
        raise ValueError(f"expected a contiguous fp32 tensor of at least {n} values")
    return t.data_ptr()


def cs_decode_layer(layer: FfnLayer, pred, x, y, params, ws: Workspace, stream=None, idx=None,
                    count=None):
    """One token through one layer: y = FFN(x, select(P(x))) (see include/cs.h).
    x and y may live on the GPU or in pinned host memory."""
    d = layer.c.d
    _check(lib().cs_decode_layer(C.byref(layer.c), C.byref(pred.c) if pred is not None else None,
                                 _io_ptr(x, d), _io_ptr(y, d), C.byref(params), ws.ptr, ws.nbytes,
                                 _stream(stream), _ptr(idx), _ptr(count)))


def cs_permute_rows(src, perm, dst, rows=None, cols=None, stream=None):
    """dst[i, :cols] = src[perm[i], :cols] for i < rows (the frequency-sorted
    layout step; src and dst are 2-D CUDA tensors of one dtype, or 1-D fp32
    vectors such as the bias)."""
    if src.dtype != dst.dtype:
        raise ValueError("src and dst must have the same dtype")
    s2 = src if src.dim() == 2 else src.view(-1, 1)
    d2 = dst if dst.dim() == 2 else dst.view(-1, 1)
    rows = d2.shape[0] if rows is None else int(rows)
    cols = s2.shape[1] if cols is None else int(cols)
    if perm.dtype != torch.int32 or perm.numel() < rows or s2.stride(1) != 1 or d2.stride(1) != 1:
        raise ValueError("perm must be int32 with >= rows entries; rows must be contiguous")
    _check(lib().cs_permute_rows(_ptr(s2), s2.shape[0], s2.stride(0), _ptr(perm), rows, cols, _dt(s2),
                                 _ptr(d2), d2.stride(0), _stream(stream)))


def cs_hot_order(freq):
    """The frequency-sorted neuron order (host): most frequent first, ties by
    lower id.  freq: a sequence or CPU array of f frequencies; returns an
    int32 CPU tensor."""
    fr = torch.as_tensor(freq, dtype=torch.float32).contiguous()
    out = torch.empty(fr.numel(), dtype=torch.int32)
    _check(lib().cs_hot_order(fr.data_ptr(), fr.numel(), out.data_ptr()))
    return out


class AttnLayer:
    """Head-sparse attention weights: w_q and w_o_t are [n_heads * d_head, d]
    CUDA tensors of one dtype (w_o_t is W_o transposed)."""

    def __init__(self, w_q, w_o_t, n_heads):
        if w_q.shape != w_o_t.shape or w_q.dtype != w_o_t.dtype or w_q.shape[0] % int(n_heads):
            raise ValueError("w_q and w_o_t must both be [n_heads * d_head, d] of one dtype")
        self.w_q, self.w_o_t = w_q, w_o_t
        self.n_heads = int(n_heads)
        self.d_head = w_q.shape[0] // self.n_heads
        self.d = w_q.shape[1]
        self.c = _Attn(self.d, self.n_heads, self.d_head, _dt(w_q), _ptr(w_q), _ptr(w_o_t))


def cs_sparse_attention(layer: AttnLayer, x, heads, count, k_cache, v_cache, y, ws: Workspace, stream=None):
    """y = the selected heads' attention over the KV cache (see include/cs.h);
    k_cache / v_cache are [n_heads, seq_len, d_head] CUDA tensors."""
    _check(lib().cs_sparse_attention(C.byref(layer.c), _ptr(x), _ptr(heads), _ptr(count), _ptr(k_cache),
                                     _ptr(v_cache), int(k_cache.shape[1]), _ptr(y), ws.ptr, ws.nbytes,
                                     _stream(stream)))


def cs_decode_attention(layer: AttnLayer, pred, x, y, params, k_cache, v_cache, ws: Workspace, stream=None,
                        heads=None, count=None):
    """One token's head-sparse attention step: the predictor scores the heads,
    the selection picks them, y = their attention over the KV cache (see
    include/cs.h).  x and y may live on the GPU or in pinned host memory;
    k_cache / v_cache are [n_heads, seq_len, d_head] CUDA tensors."""
    d = layer.d
    _check(lib().cs_decode_attention(C.byref(layer.c), C.byref(pred.c), _io_ptr(x, d), _io_ptr(y, d),
                                     C.byref(params), _ptr(k_cache), _ptr(v_cache), int(k_cache.shape[1]),
                                     ws.ptr, ws.nbytes, _stream(stream), _ptr(heads), _ptr(count)))


def cs_fit_predictor(layer: FfnLayer, pred: Predictor, X, lam, stream=None):
    """Overwrite pred's up map with the ridge fit of the layer's gate
    pre-activations onto relu(P_down x) over the calibration inputs X [N, d]
    (see include/cs.h).  Waits for the stream."""
    if X.dtype != torch.float32 or not X.is_cuda or not X.is_contiguous():
        raise ValueError("X must be a contiguous fp32 CUDA tensor [N, d]")
    N = X.shape[0]
    n = lib().cs_fit_scratch_size(layer.d, layer.f, pred.r, N)
    if n == 0:
        raise ValueError("bad fit dimensions")
    buf = torch.empty(n + 256, dtype=torch.uint8, device=X.device)
    ptr = (buf.data_ptr() + 255) & ~255
    _check(lib().cs_fit_predictor(C.byref(layer.c), C.byref(pred.c), _ptr(X), N, float(lam), ptr, n,
                                  _stream(stream)))


def cs_stack_release():
    _check(lib().cs_stack_release())
