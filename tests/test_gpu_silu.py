"""GPU parity of SiLU layers ("The SiLU/GELU Challenge: TurboSparse":
down(silu(gate x) * up x); "The Empirical Foundation": SiLU layers are only
functionally sparse) against the oracle: the CUDA-core gather, the tcgen05
batched path, the magnitude-cut exact mode and the layer stack."""
import math

import numpy as np
import pytest

import oracle
import synth
from _helpers import (TOL, HostLayer, pick_k_with_gap, rel_err, score_bounds, stack_inputs)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402

SILU = cs.CS_ACT_SILU


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


def run_ffn(H, X, sel):
    layer, _ = H.device()
    B, d = X.shape
    y = torch.empty((B, d), device="cuda")
    ws = cs.Workspace(d, H.f, 1, B)
    cs.cs_sparse_ffn(layer, torch.from_numpy(X).cuda(), torch.from_numpy(sel).cuda(),
                     torch.tensor([sel.size], dtype=torch.int32, device="cuda"), y, ws)
    torch.cuda.synchronize()
    assert cs.cs_get_device_error(ws) == 0
    return y.cpu().numpy()


@pytest.mark.parametrize("dt", [synth.F32, synth.F16, synth.BF16])
@pytest.mark.parametrize("glu", [False, True])
@pytest.mark.parametrize("B", [1, 2])
def test_silu_gather(dt, glu, B):
    d, f = 1000, 3001
    H = HostLayer(d, f, 0, dt, glu=glu, seed=21, act=SILU)
    X = synth.x_normal(22, B, d)
    sel = np.sort(np.random.default_rng(2).choice(f, size=700, replace=False)).astype(np.int32)
    Y = run_ffn(H, X, sel)
    O = H.oracle_layer()
    for b in range(B):
        assert rel_err(Y[b], oracle.ffn(O, X[b], sel)) < TOL, b


@pytest.mark.parametrize("dt", [synth.F16, synth.BF16])
@pytest.mark.parametrize("B", [4, 8, 32])
def test_silu_tensor_core_batch(dt, B):
    """B >= 4 with d a multiple of 64 takes the tcgen05 path: SwiGLU's gate
    activation is applied in the gate GEMM's epilogue."""
    d, f = 1024, 4096
    H = HostLayer(d, f, 0, dt, glu=True, seed=23, act=SILU)
    X = synth.x_normal(24, B, d)
    sel = np.sort(np.random.default_rng(3).choice(f, size=1500, replace=False)).astype(np.int32)
    Y = run_ffn(H, X, sel)
    O = H.oracle_layer()
    for b in (0, B // 2, B - 1):
        assert rel_err(Y[b], oracle.ffn(O, X[b], sel)) < TOL, b


def silu64(g):
    g = np.asarray(g, np.float64)
    with np.errstate(over="ignore"):
        return g / (1.0 + np.exp(-g))


@pytest.mark.parametrize("glu", [False, True])
@pytest.mark.parametrize("tau", [0.02, 0.1])
def test_silu_exact_magnitude_cut(glu, tau):
    """A = {j : |silu(g_j)| > tau}: every neuron decided beyond fp32 rounding
    agrees with the fp64 predicate on the GPU's own pre-activations; y matches
    the oracle on the GPU's set."""
    d, f = 2048, 6000
    H = HostLayer(d, f, 0, synth.BF16, glu=glu, seed=25, act=SILU)
    layer, _ = H.device()
    X = synth.x_normal(26, 1, d)
    pre = torch.empty(f, device="cuda")
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    mask = torch.empty((f + 31) // 32, dtype=torch.int32, device="cuda")
    y = torch.empty(d, device="cuda")
    ws = cs.Workspace(d, f, 1)
    cs.cs_exact_ffn(layer, torch.from_numpy(X).cuda(), pre, idx, cnt, y, ws, mask=mask, tau=tau)
    torch.cuda.synchronize()
    O = H.oracle_layer()
    opre = oracle.preact(O, X[0])
    gp = pre.cpu().numpy()
    assert rel_err(gp, opre) < 1e-5
    n = int(cnt.item())
    got = idx.cpu().numpy()[:n]
    assert np.all(np.diff(got) > 0)
    m = np.abs(silu64(gp))
    band = 1e-5 * max(tau, 1e-3)
    sure_in, sure_out = set(np.flatnonzero(m > tau + band)), set(np.flatnonzero(m < tau - band))
    gs = set(got.tolist())
    assert sure_in <= gs and not (gs & sure_out)
    assert 0 < n < f
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), synth.bits_from_bool(np.isin(np.arange(f), got)))
    assert rel_err(y.cpu().numpy(), oracle.ffn(O, X[0], got)) < TOL
    assert cs.cs_get_device_error(ws) == 0


def test_relu_exact_with_a_cut_is_bit_exact():
    """relu(g) > tau is g > tau: the same fp32 decision on both sides."""
    d, f = 1000, 3001
    H = HostLayer(d, f, 0, synth.F16, seed=27)
    layer, _ = H.device()
    X = synth.x_normal(28, 1, d)
    pre = torch.empty(f, device="cuda")
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    y = torch.empty(d, device="cuda")
    ws = cs.Workspace(d, f, 1)
    cs.cs_exact_ffn(layer, torch.from_numpy(X).cuda(), pre, idx, cnt, y, ws, tau=0.5)
    torch.cuda.synchronize()
    gp = pre.cpu().numpy()
    want = oracle.select_magnitude(gp, oracle.ACT_RELU, 0.5)
    n = int(cnt.item())
    assert np.array_equal(idx.cpu().numpy()[:n], want)
    assert rel_err(y.cpu().numpy(), oracle.ffn(H.oracle_layer(), X[0], want)) < TOL
    with pytest.raises(cs.CsError):   # a negative cut is refused
        cs.cs_exact_ffn(layer, torch.from_numpy(X).cuda(), pre, idx, cnt, y, ws, tau=-1.0)


def test_silu_step_topk():
    """Predictor, top-k and the SwiGLU gather: ids bit-exact, y within bound."""
    d, f, r = 2048, 8192, 128
    H = HostLayer(d, f, r, synth.BF16, glu=True, seed=29, act=SILU)
    layer, pred = H.device()
    X = synth.x_normal(30, 1, d)
    s_ref, eps = score_bounds(H, X[0])
    k = pick_k_with_gap(s_ref, eps, synth.ceil_k(f, 0.15))
    x = torch.from_numpy(X).cuda()
    y = torch.empty(d, device="cuda")
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    ws = cs.Workspace(d, f, r)
    s = torch.cuda.Stream()
    torch.cuda.synchronize()
    cs.cs_decode_layer(layer, pred, x[0], y, cs.select_params(cs.CS_SEL_TOPK, k), ws, stream=s,
                       idx=idx, count=cnt)
    s.synchronize()
    want = oracle.select_topk(s_ref.astype(np.float32), k)
    assert int(cnt.item()) == k and np.array_equal(idx.cpu().numpy()[:k], want)
    assert rel_err(y.cpu().numpy(), oracle.ffn(H.oracle_layer(), X[0], want)) < TOL


def test_silu_stack_exact_mode():
    """A 3-layer SiLU stack with the magnitude cut at tau = 0 (every neuron whose
    gate activation is not exactly zero): x_L against the oracle's stack."""
    L, d, f = 3, 512, 2048
    Hs, layers, _ = stack_inputs(L, d, f, 0, synth.F16, glu=True, act=SILU)
    X = synth.x_normal(31, 1, d)[0]
    x = torch.from_numpy(X.copy()).cuda()
    ws = cs.Workspace(d, f, 1)
    torch.cuda.synchronize()
    cs.cs_decode_stack(layers, None, x, 0.1, cs.select_params(cs.CS_SEL_EXACT, tau=0.0),
                       cs.CS_STACK_SEQUENTIAL, ws, s_main=torch.cuda.Stream())
    torch.cuda.synchronize()
    want = oracle.stack([H.oracle_layer() for H in Hs], None, X, sel_mode=oracle.SEL_EXACT, tau=0.0,
                        resid_scale=0.1)
    assert rel_err(x.cpu().numpy(), want) < TOL
    assert cs.cs_get_device_error(ws) == 0
