"""Shared helpers for the GPU parity tests: build the same synthetic layer on
the host (oracle inputs, from synth's C twin) and on the device (uploaded),
and compare results."""
from __future__ import annotations

import math

import numpy as np

import oracle
import synth

TOL = 2e-3  # max |gpu - oracle| / max |oracle| on scores and y


def rel_err(gpu, ref):
    gpu = np.asarray(gpu, np.float64)
    ref = np.asarray(ref, np.float64)
    den = np.abs(ref).max()
    if den == 0:
        return float(np.abs(gpu).max())
    return float(np.abs(gpu - ref).max() / den)


def torch_dtype(dt):
    import torch
    return {synth.F32: torch.float32, synth.F16: torch.float16, synth.BF16: torch.bfloat16}[dt]


def upload(arr, dt):
    """numpy storage array -> CUDA tensor of the storage dtype."""
    import torch
    if dt == synth.BF16:
        return torch.from_numpy(np.ascontiguousarray(arr).view(np.int16)).view(torch.bfloat16).cuda()
    return torch.from_numpy(np.ascontiguousarray(arr)).cuda()


def pad_ld(d, dt):
    """Smallest row stride >= d whose byte size is a multiple of 16."""
    per = 16 // synth.DTYPE_BYTES[dt]
    return (d + per - 1) // per * per


class HostLayer:
    """One synthetic layer + predictor, as host arrays (storage form)."""

    def __init__(self, d, f, r, dt, glu=False, seed=0, layer=0, rho=0.1, ld=None, bias=True, act=0):
        self.d, self.f, self.r, self.dt, self.glu = d, f, r, dt, glu
        self.act = act  # 0 relu, 1 silu
        self.ld = ld or pad_ld(d, dt)
        self.ldr = pad_ld(r, dt) if r else 0
        sd = 1 / math.sqrt(d)
        mk = lambda w, rows, cols, ld: synth.normal_matrix(seed, synth.tensor_id(layer, w), rows, cols, sd, dt, ld=ld)
        self.w_gate = mk(synth.W_GATE, f, d, self.ld)
        self.w_down_t = mk(synth.W_DOWN_T, f, d, self.ld)
        self.w_up = mk(synth.W_UP, f, d, self.ld) if glu else None
        self.bias = synth.zipf_bias(seed, layer, f, rho) if bias else None
        if r:
            self.p_down = mk(synth.P_DOWN, r, d, self.ld)
            self.p_up = mk(synth.P_UP, f, r, self.ldr)

    def oracle_layer(self):
        return oracle.Layer(self.d, self.f, self.dt, self.w_gate, self.w_down_t, w_up=self.w_up,
                            bias=self.bias, ld=self.ld, act=self.act)

    def oracle_pred(self):
        return oracle.Predictor(self.d, self.r, self.f, self.dt, self.p_down, self.p_up,
                                ld_down=self.ld, ld_up=self.ldr)

    def device(self):
        import torch
        import contextual_sparsity_sparse_gb300 as cs
        t = {k: upload(getattr(self, k), self.dt) for k in ("w_gate", "w_down_t")}
        t["w_up"] = upload(self.w_up, self.dt) if self.glu else None
        t["bias"] = torch.from_numpy(self.bias).cuda() if self.bias is not None else None
        layer = cs.FfnLayer(t["w_gate"], t["w_down_t"], w_up=t["w_up"], bias=t["bias"], d=self.d, act=self.act)
        pred = None
        if self.r:
            pd, pu = upload(self.p_down, self.dt), upload(self.p_up, self.dt)
            pred = cs.Predictor(pd, pu, d=self.d)
            pred.keep = (pd, pu)
        layer.keep = t
        return layer, pred


def score_bounds(P: HostLayer, x):
    """Oracle scores and a 10-sigma bound on |fp32 GPU score - exact score|.

    The kernels sum each dot product in fp32 along chains of at most ~64
    dependent roundings (per-thread runs, warp shuffles, a fixed cross-warp
    order).  Rounding errors are independent with |delta| <= u |partial|
    (u = 2^-24), so their sum has a spread of about u * sqrt(chain) *
    sqrt(sum terms^2); the bound takes 10 times that for both GEMVs (the
    bottleneck's error propagated through P_up), plus the final rounding of
    the score to fp32.  The kernels' measured error sits far inside it.
    """
    x = np.asarray(x, np.float64)
    pd = synth.storage_to_f64(P.p_down, P.dt)[:, :P.d]
    pu = synth.storage_to_f64(P.p_up, P.dt)[:, :P.r]
    h, s = oracle.predict(P.oracle_pred(), x)
    c = 10 * 2.0 ** -24 * 8.0
    dh = c * np.sqrt((pd * pd) @ (x * x))
    eps = c * np.sqrt((pu * pu) @ (h * h)) + np.sqrt((pu * pu) @ (dh * dh)) + 2.0 ** -24 * np.abs(s)
    return s, eps


def pick_k_with_gap(s, eps, k0, span=64):
    """A k near k0 whose boundary is decided beyond rounding: the k-th and
    (k+1)-th largest scores differ by more than both error bounds."""
    order = np.argsort(-s, kind="stable")
    for dk in range(span):
        for k in (k0 + dk, k0 - dk):
            if 0 < k < s.size:
                a, b = order[k - 1], order[k]
                if s[a] - s[b] > eps[a] + eps[b]:
                    return k
    raise AssertionError("no decidable k near k0")


def pick_tau_with_gap(s, eps, q):
    """A threshold near the q-quantile with no score within its error bound."""
    srt = np.sort(s)
    i0 = int(q * s.size)
    order = np.argsort(s, kind="stable")
    for di in range(s.size):
        for i in (i0 + di, i0 - di):
            if 0 < i < s.size:
                lo, hi = order[i - 1], order[i]
                if s[hi] - s[lo] > 2 * (eps[lo] + eps[hi]):
                    return np.float32((s[lo] + s[hi]) / 2)
    raise AssertionError("no decidable threshold")


def stack_inputs(L, d, f, r, dt, glu=False, seed=0, rho=0.1, act=0):
    Hs = [HostLayer(d, f, r, dt, glu=glu, seed=seed, layer=l, rho=rho, act=act) for l in range(L)]
    dev = [H.device() for H in Hs]
    return Hs, [a for a, _ in dev], [b for _, b in dev]


def oracle_stack_k(Hs, x0, mode, k0, scale):
    """A k at which every layer's top-k boundary is decided beyond rounding,
    with the oracle's output and trace at that k.  x_l comes from the oracle
    run on the first l layers; the bound is widened for the fp32 drift of the
    GPU's x_l."""
    layers = [H.oracle_layer() for H in Hs]
    preds = [H.oracle_pred() for H in Hs]
    for k in range(k0, k0 + 64):
        xs = [np.asarray(x0, np.float64)]
        for l in range(1, len(Hs)):
            xs.append(oracle.stack(layers[:l], preds[:l], x0, mode=mode, k=k, resid_scale=scale))
        ok = True
        for l, H in enumerate(Hs):
            xin = xs[l - 1] if (mode == oracle.LOOKAHEAD and l > 0) else xs[l]
            s, eps = score_bounds(H, xin)
            eps = 4 * eps + 1e-6 * np.abs(s).max()
            order = np.argsort(-s, kind="stable")
            a, b = order[k - 1], order[k]
            if s[a] - s[b] <= eps[a] + eps[b]:
                ok = False
                break
        if ok:
            xo, tr = oracle.stack(layers, preds, x0, mode=mode, k=k, resid_scale=scale, trace=True)
            return k, xo, tr
    raise AssertionError("no decidable k")
