"""GPU parity of the whole decode step (predict -> select -> gathered FFN) and
of the layer stack, against the CPU oracle.

Selections are decided on fp32 scores on both sides.  The kernels' scores
carry fp32 rounding, so each test uses a k (or tau) whose boundary is decided
beyond the rounding bound computed by the oracle (``pick_k_with_gap``); there
the GPU must pick exactly the oracle's neurons."""
import numpy as np
import pytest

import oracle
import synth
from _helpers import (TOL, HostLayer, oracle_stack_k, pick_k_with_gap, pick_tau_with_gap, rel_err,
                      score_bounds, stack_inputs)

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


def run_step(layer, pred, x, params, f, d, ws):
    scores = torch.empty((1, f), device="cuda")
    idx = torch.empty((1, f), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    y = torch.empty((1, d), device="cuda")
    cs.cs_predict(pred, x, scores, ws)
    cs.cs_select(scores, params, idx, cnt, ws=ws)
    cs.cs_sparse_ffn(layer, x, idx, cnt, y, ws)
    n = int(cnt.item())
    return scores.cpu().numpy()[0], idx.cpu().numpy()[0, :n], y.cpu().numpy()[0]


# workloads: the tiny ReLU FFN (fp32, d512 f2048 r64, top-k 205) and the
# OPT-13B-shaped layer (fp16, d5120 f20480 r512, k = 5/10/20%)
STEP_CASES = [
    ("tiny-relu-f32", 512, 2048, 64, synth.F32, False, 0.10),
    ("opt13b-f16-5", 5120, 20480, 512, synth.F16, False, 0.05),
    ("opt13b-f16-10", 5120, 20480, 512, synth.F16, False, 0.10),
    ("opt13b-f16-20", 5120, 20480, 512, synth.F16, False, 0.20),
    ("glu-bf16", 2048, 6000, 128, synth.BF16, True, 0.15),
]


@pytest.mark.parametrize("case", STEP_CASES, ids=[c[0] for c in STEP_CASES])
def test_step_topk(case):
    name, d, f, r, dt, glu, rho = case
    H = HostLayer(d, f, r, dt, glu=glu, seed=0, rho=rho)
    layer, pred = H.device()
    ws = cs.Workspace(d, f, r)
    for t in range(2):
        X = synth.x_normal(100 + t, 1, d)
        s_ref, eps = score_bounds(H, X[0])
        k = pick_k_with_gap(s_ref, eps, synth.ceil_k(f, rho))
        s, idx, y = run_step(layer, pred, torch.from_numpy(X).cuda(),
                             cs.select_params(cs.CS_SEL_TOPK, k), f, d, ws)
        assert np.all(np.abs(s - s_ref) <= eps + 1e-30)
        want = oracle.select_topk(s_ref.astype(np.float32), k)
        assert np.array_equal(idx, want)
        # the GPU's own selection is exactly the top-k of its own scores
        assert np.array_equal(idx, oracle.select_topk(s, k))
        assert rel_err(y, oracle.ffn(H.oracle_layer(), X[0], want)) < TOL
    assert cs.cs_get_device_error(ws) == 0


@pytest.mark.parametrize("case", STEP_CASES[:4], ids=[c[0] for c in STEP_CASES[:4]])
def test_step_threshold(case):
    name, d, f, r, dt, glu, rho = case
    H = HostLayer(d, f, r, dt, glu=glu, seed=0, rho=rho)
    layer, pred = H.device()
    ws = cs.Workspace(d, f, r)
    X = synth.x_normal(7, 1, d)
    s_ref, eps = score_bounds(H, X[0])
    tau = pick_tau_with_gap(s_ref, eps, 1 - rho)
    s, idx, y = run_step(layer, pred, torch.from_numpy(X).cuda(),
                         cs.select_params(cs.CS_SEL_THRESHOLD, 0, float(tau)), f, d, ws)
    want = oracle.select_threshold(s_ref.astype(np.float32), tau)
    assert np.array_equal(idx, want)
    assert rel_err(y, oracle.ffn(H.oracle_layer(), X[0], want)) < TOL


def test_identity_predictor_recovers_exact_mask():
    """P_down = [I; -I], P_up = [W, -W]: scores = W x, so threshold 0 on the
    GPU scores gives the exact mask of a bias-free layer (recall = precision
    = 1 up to rounding at zero)."""
    d, f = 256, 1000
    W = synth.normal_matrix(4, 0, f, d, 1 / 16, synth.F32)
    eye = np.eye(d, dtype=np.float32)
    pd = torch.from_numpy(np.concatenate([eye, -eye])).cuda()
    pu = torch.from_numpy(np.concatenate([W, -W], axis=1)).cuda()
    pred = cs.Predictor(pd, pu)
    X = synth.x_normal(5, 1, d)
    scores = torch.empty((1, f), device="cuda")
    ws = cs.Workspace(d, f, 2 * d)
    cs.cs_predict(pred, torch.from_numpy(X).cuda(), scores, ws)
    idx = torch.empty((1, f), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    cs.cs_select(scores, cs.select_params(cs.CS_SEL_THRESHOLD, 0, 0.0), idx, cnt)
    pred_set = idx.cpu().numpy()[0, :int(cnt.item())]
    O = oracle.Layer(d, f, synth.F32, W, W)
    exact = oracle.select_positive(oracle.preact(O, X[0]).astype(np.float32))
    rec, prec = oracle.recall_precision(pred_set, exact, f)
    assert rec == 1.0 and prec == 1.0


# -------------------------------------------------------------------- stack

@pytest.mark.parametrize("mode", [cs.CS_STACK_SEQUENTIAL, cs.CS_STACK_LOOKAHEAD])
@pytest.mark.parametrize("dt,glu", [(synth.F16, False), (synth.BF16, True)])
def test_stack_topk(mode, dt, glu):
    L, d, f, r = 4, 512, 2048, 64
    Hs, layers, preds = stack_inputs(L, d, f, r, dt, glu=glu)
    X = synth.x_normal(11, 1, d)[0]
    omode = oracle.LOOKAHEAD if mode == cs.CS_STACK_LOOKAHEAD else oracle.SEQUENTIAL
    try:
        k, xo, tr = oracle_stack_k(Hs, X, omode, 205, 0.1)
    except AssertionError:
        pytest.skip("no decidable k")
    x = torch.from_numpy(X.copy()).cuda()
    ws = cs.Workspace(d, f, r)
    tc = torch.zeros(L, dtype=torch.int32, device="cuda")
    ti = torch.zeros((L, f), dtype=torch.int32, device="cuda")
    s_main, s_pred = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    cs.cs_decode_stack(layers, preds, x, 0.1, cs.select_params(cs.CS_SEL_TOPK, k), mode, ws,
                       s_main=s_main, s_pred=s_pred, trace_count=tc, trace_idx=ti)
    torch.cuda.synchronize()
    TC, TI = tc.cpu().numpy(), ti.cpu().numpy()
    for l in range(L):
        assert TC[l] == tr["count"][l]
        assert np.array_equal(TI[l, :TC[l]], tr["idx"][l]), l
    assert rel_err(x.cpu().numpy(), xo) < TOL
    first = x.cpu().numpy().copy()
    # replays of the cached graph, and the uncaptured path on the legacy stream,
    # give the same bits
    for sm in (s_main, s_main, None):
        x.copy_(torch.from_numpy(X.copy()))
        torch.cuda.synchronize()
        cs.cs_decode_stack(layers, preds, x, 0.1, cs.select_params(cs.CS_SEL_TOPK, k), mode, ws,
                           s_main=sm if sm is not None else torch.cuda.default_stream(),
                           s_pred=s_pred, trace_count=tc, trace_idx=ti)
        torch.cuda.synchronize()
        assert np.array_equal(first.view(np.uint32), x.cpu().numpy().view(np.uint32))
    assert cs.cs_get_device_error(ws) == 0


def test_stack_exact_equals_dense_composition():
    L, d, f = 3, 256, 1024
    Hs, layers, _ = stack_inputs(L, d, f, 0, synth.F16)
    X = synth.x_normal(12, 1, d)[0]
    x = torch.from_numpy(X.copy()).cuda()
    ws = cs.Workspace(d, f, 1)
    sm = torch.cuda.Stream()
    torch.cuda.synchronize()
    cs.cs_decode_stack(layers, None, x, 0.25, cs.select_params(cs.CS_SEL_EXACT), cs.CS_STACK_SEQUENTIAL,
                       ws, s_main=sm)
    torch.cuda.synchronize()
    want = oracle.stack([H.oracle_layer() for H in Hs], None, X, sel_mode=oracle.SEL_EXACT,
                        resid_scale=0.25)
    assert rel_err(x.cpu().numpy(), want) < TOL


def test_stack_lookahead_equals_sequential_at_zero_step():
    L, d, f, r = 3, 256, 1024, 32
    Hs, layers, preds = stack_inputs(L, d, f, r, synth.F16)
    X = synth.x_normal(13, 1, d)[0]
    outs = []
    for mode in (cs.CS_STACK_SEQUENTIAL, cs.CS_STACK_LOOKAHEAD):
        x = torch.from_numpy(X.copy()).cuda()
        tc = torch.zeros(L, dtype=torch.int32, device="cuda")
        ti = torch.zeros((L, f), dtype=torch.int32, device="cuda")
        ws = cs.Workspace(d, f, r)
        torch.cuda.synchronize()
        cs.cs_decode_stack(layers, preds, x, 0.0, cs.select_params(cs.CS_SEL_TOPK, 100), mode, ws,
                           s_main=torch.cuda.Stream(), s_pred=torch.cuda.Stream(),
                           trace_count=tc, trace_idx=ti)
        torch.cuda.synchronize()
        outs.append((x.cpu().numpy(), ti.cpu().numpy()))
    assert np.array_equal(outs[0][0], outs[1][0]) and np.array_equal(outs[0][1], outs[1][1])
    assert np.array_equal(outs[0][0], X)  # zero step leaves the stream unchanged


def test_stack_inside_caller_capture():
    L, d, f, r = 2, 256, 1024, 32
    Hs, layers, preds = stack_inputs(L, d, f, r, synth.F16)
    X = synth.x_normal(14, 1, d)[0]
    ws = cs.Workspace(d, f, r)
    ref = torch.from_numpy(X.copy()).cuda()
    cs.cs_decode_stack(layers, preds, ref, 0.1, cs.select_params(cs.CS_SEL_TOPK, 100),
                       cs.CS_STACK_LOOKAHEAD, ws, s_main=torch.cuda.current_stream(),
                       s_pred=torch.cuda.Stream())
    torch.cuda.synchronize()
    x = torch.from_numpy(X.copy()).cuda()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cs.cs_decode_stack(layers, preds, x, 0.1, cs.select_params(cs.CS_SEL_TOPK, 100),
                               cs.CS_STACK_LOOKAHEAD, ws, s_main=s, s_pred=torch.cuda.Stream())
    x.copy_(torch.from_numpy(X.copy()).cuda())
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(x.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("graph_io", ["1", "0"])
@pytest.mark.parametrize("L", [3, 4])
def test_stack_with_pinned_host_x(L, graph_io, monkeypatch):
    """x_0 in page-locked host memory: read and x_L written back by the
    call (by the graph's own copy kernels, or with CS_GRAPH_IO=0 by copies
    around the launch); the result is the device-x call's, bit for bit, and
    several host buffers replay one cached graph.  Pageable host memory is
    refused."""
    monkeypatch.setenv("CS_GRAPH_IO", graph_io)
    d, f, r = 512, 2048, 64
    Hs, layers, preds = stack_inputs(L, d, f, r, synth.BF16, glu=True)
    ws = cs.Workspace(d, f, r)
    sm, sp = torch.cuda.Stream(), torch.cuda.Stream()
    params = cs.select_params(cs.CS_SEL_TOPK, 205)
    for seed in (15, 16):
        X = synth.x_normal(seed, 1, d)[0]
        ref = torch.from_numpy(X.copy()).cuda()
        torch.cuda.synchronize()
        cs.cs_decode_stack(layers, preds, ref, 0.1, params, cs.CS_STACK_LOOKAHEAD, ws, s_main=sm, s_pred=sp)
        sm.synchronize()
        xh = torch.from_numpy(X.copy()).pin_memory()
        cs.cs_decode_stack(layers, preds, xh, 0.1, params, cs.CS_STACK_LOOKAHEAD, ws, s_main=sm, s_pred=sp)
        sm.synchronize()
        assert np.array_equal(xh.numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))
    with pytest.raises(cs.CsError):
        cs.cs_decode_stack(layers, preds, torch.from_numpy(X.copy()), 0.1, params, cs.CS_STACK_LOOKAHEAD, ws,
                           s_main=sm, s_pred=sp)
    assert cs.cs_get_device_error(ws) == 0
