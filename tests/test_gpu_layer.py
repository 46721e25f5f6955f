"""GPU parity of cs_decode_layer, the one-call decode step of one layer
(predictor -> selection -> gathered FFN, captured into a CUDA graph), against
the CPU oracle and against the same step issued as three separate calls.

The graph runs the very kernels of cs_predict, cs_select and cs_sparse_ffn,
so its ids and y must equal the three-call path's bit for bit, on the first
call (capture) and on every replay with a new x.  x and y are exercised both
in device memory and in pinned host memory (staged through the workspace)."""
import ctypes

import numpy as np
import pytest

import oracle
import synth
from _helpers import TOL, HostLayer, pick_k_with_gap, pick_tau_with_gap, rel_err, score_bounds

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402

CS_ERR_INVALID = 1


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


CASES = [
    ("tiny-relu-f32", 512, 2048, 64, synth.F32, False, 0.10),
    ("opt13b-f16-10", 5120, 20480, 512, synth.F16, False, 0.10),
    ("glu-bf16", 2048, 6000, 128, synth.BF16, True, 0.15),
]


def three_calls(layer, pred, X, params, f, d, s):
    """The same step as cs_predict + cs_select + cs_sparse_ffn on its own workspace."""
    ws = cs.Workspace(d, f, pred.c.r if pred is not None else 1, stream=s)
    x = torch.from_numpy(X).cuda()
    scores = torch.empty((1, f), device="cuda")
    idx = torch.empty((1, f), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    y = torch.empty((1, d), device="cuda")
    with torch.cuda.stream(s):
        cs.cs_predict(pred, x, scores, ws, stream=s)
        cs.cs_select(scores, params, idx, cnt, ws=ws, stream=s)
        cs.cs_sparse_ffn(layer, x, idx, cnt, y, ws, stream=s)
    s.synchronize()
    n = int(cnt.item())
    return idx.cpu().numpy()[0, :n], y.cpu().numpy()[0]


@pytest.mark.parametrize("io", ["device", "pinned", "pinned-copies"])
@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_layer_topk(case, io, monkeypatch):
    """pinned: the graph's own copy kernels read x and write y; pinned-copies
    (CS_GRAPH_IO=0): copies around the graph launch."""
    monkeypatch.setenv("CS_GRAPH_IO", "0" if io == "pinned-copies" else "1")
    name, d, f, r, dt, glu, rho = case
    H = HostLayer(d, f, r, dt, glu=glu, seed=0, rho=rho)
    layer, pred = H.device()
    O = H.oracle_layer()
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, f, r, stream=s)
    Xs = [synth.x_normal(300 + t, 1, d) for t in range(3)]
    s_ref, eps = score_bounds(H, Xs[0][0])
    k = pick_k_with_gap(s_ref, eps, synth.ceil_k(f, rho))
    params = cs.select_params(cs.CS_SEL_TOPK, k)
    idx = torch.full((f,), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    xd = torch.empty(d, device="cuda")
    yd = torch.empty(d, device="cuda")
    for t, X in enumerate(Xs):   # call 0 captures the graph, calls 1 and 2 replay it
        if io == "device":
            xd.copy_(torch.from_numpy(X[0]))
            x, y = xd, yd
        else:                    # a fresh pinned pair every call: host addresses change
            x = torch.from_numpy(X[0].copy()).pin_memory()
            y = torch.full((d,), float("nan")).pin_memory()
        torch.cuda.synchronize()
        cs.cs_decode_layer(layer, pred, x, y, params, ws, stream=s, idx=idx, count=cnt)
        s.synchronize()
        n = int(cnt.item())
        gi = idx.cpu().numpy()[:n]
        gy = y.cpu().numpy()
        ri, ry = three_calls(layer, pred, X, params, f, d, s)
        assert np.array_equal(gi, ri), t
        assert np.array_equal(gy.view(np.uint32), ry.view(np.uint32)), t
        assert rel_err(gy, oracle.ffn(O, X[0], gi)) < TOL, t
        if t == 0:
            assert np.array_equal(gi, oracle.select_topk(s_ref.astype(np.float32), k))
    assert cs.cs_get_device_error(ws) == 0


def test_layer_threshold_and_no_outputs():
    name, d, f, r, dt, glu, rho = CASES[0]
    H = HostLayer(d, f, r, dt, glu=glu, seed=1, rho=rho)
    layer, pred = H.device()
    X = synth.x_normal(21, 1, d)
    s_ref, eps = score_bounds(H, X[0])
    tau = pick_tau_with_gap(s_ref, eps, 1 - rho)
    params = cs.select_params(cs.CS_SEL_THRESHOLD, 0, float(tau))
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, f, r, stream=s)
    x = torch.from_numpy(X[0].copy()).cuda()
    y = torch.empty(d, device="cuda")
    y2 = torch.empty(d, device="cuda")
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    torch.cuda.synchronize()
    cs.cs_decode_layer(layer, pred, x, y, params, ws, stream=s, idx=idx, count=cnt)
    cs.cs_decode_layer(layer, pred, x, y2, params, ws, stream=s)   # ids kept in the workspace
    s.synchronize()
    want = oracle.select_threshold(s_ref.astype(np.float32), tau)
    assert np.array_equal(idx.cpu().numpy()[:int(cnt.item())], want)
    assert rel_err(y.cpu().numpy(), oracle.ffn(H.oracle_layer(), X[0], want)) < TOL
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))


@pytest.mark.parametrize("io", ["device", "pinned", "pinned_x", "pinned_y"])
def test_layer_exact_matches_exact_ffn(io):
    d, f = 1000, 3001
    H = HostLayer(d, f, 0, synth.BF16, glu=True, seed=8)
    layer, _ = H.device()
    X = synth.x_normal(22, 1, d)
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, f, 1, stream=s)
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    # pinned_x / pinned_y: one end in page-locked host memory, the other on
    # the device
    xp, yp = io in ("pinned", "pinned_x"), io in ("pinned", "pinned_y")
    x = torch.from_numpy(X[0].copy()).pin_memory() if xp else torch.from_numpy(X[0].copy()).cuda()
    y = torch.empty(d).pin_memory() if yp else torch.empty(d, device="cuda")
    torch.cuda.synchronize()
    cs.cs_decode_layer(layer, None, x, y, cs.select_params(cs.CS_SEL_EXACT), ws, stream=s,
                       idx=idx, count=cnt)
    s.synchronize()
    # the same three kernels through cs_exact_ffn
    ws2 = cs.Workspace(d, f, 1)
    pre = torch.empty(f, device="cuda")
    idx2 = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt2 = torch.empty(1, dtype=torch.int32, device="cuda")
    y2 = torch.empty(d, device="cuda")
    cs.cs_exact_ffn(layer, torch.from_numpy(X).cuda(), pre, idx2, cnt2, y2, ws2)
    torch.cuda.synchronize()
    n = int(cnt.item())
    assert n == int(cnt2.item())
    assert np.array_equal(idx.cpu().numpy()[:n], idx2.cpu().numpy()[:n])
    assert np.array_equal(y.cpu().numpy().view(np.uint32), y2.cpu().numpy().view(np.uint32))
    assert rel_err(y.cpu().numpy(), oracle.dense_ffn(H.oracle_layer(), X[0])) < TOL


def test_layer_inside_caller_capture():
    name, d, f, r, dt, glu, rho = CASES[0]
    H = HostLayer(d, f, r, dt, seed=2, rho=rho)
    layer, pred = H.device()
    params = cs.select_params(cs.CS_SEL_TOPK, 205)
    X = synth.x_normal(23, 2, d)
    ws = cs.Workspace(d, f, r)
    ref = torch.empty(d, device="cuda")
    x = torch.from_numpy(X[0].copy()).cuda()
    cs.cs_decode_layer(layer, pred, x, ref, params, ws, stream=torch.cuda.current_stream())
    torch.cuda.synchronize()
    y = torch.empty(d, device="cuda")
    x.copy_(torch.from_numpy(X[1]))
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            cs.cs_decode_layer(layer, pred, x, y, params, ws, stream=s)
    x.copy_(torch.from_numpy(X[0]))
    g.replay()
    torch.cuda.synchronize()
    assert np.array_equal(y.cpu().numpy().view(np.uint32), ref.cpu().numpy().view(np.uint32))


def test_layer_rejects_bad_arguments():
    name, d, f, r, dt, glu, rho = CASES[0]
    H = HostLayer(d, f, r, dt, seed=3, rho=rho)
    layer, pred = H.device()
    ws = cs.Workspace(d, f, r)
    params = cs.select_params(cs.CS_SEL_TOPK, 10)
    y = torch.empty(d, device="cuda")
    with pytest.raises(cs.CsError):          # pageable host memory
        cs.cs_decode_layer(layer, pred, torch.zeros(d), y, params, ws)
    with pytest.raises(ValueError):          # not fp32
        cs.cs_decode_layer(layer, pred, torch.zeros(d, dtype=torch.float16, device="cuda"), y, params, ws)
    pageable = np.zeros(d, np.float32)       # through the C ABI directly
    st = cs.lib().cs_decode_layer(ctypes.byref(layer.c), ctypes.byref(pred.c), pageable.ctypes.data,
                                  y.data_ptr(), ctypes.byref(params), ws.ptr, ws.nbytes,
                                  torch.cuda.current_stream().cuda_stream, None, None)
    assert st == CS_ERR_INVALID
    x = torch.zeros(d, device="cuda")
    with pytest.raises(cs.CsError):          # a predictor is needed for top-k
        cs.cs_decode_layer(layer, None, x, y, params, ws)
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    with pytest.raises(cs.CsError):          # idx without count
        cs.cs_decode_layer(layer, pred, x, y, params, ws, idx=idx)
    small = cs.Workspace(64, 64, 8)
    with pytest.raises(cs.CsError):          # workspace too small
        cs.cs_decode_layer(layer, pred, x, y, params, small)
