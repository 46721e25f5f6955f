"""GPU parity of the fitted predictor (cs_fit_predictor, the ridge fit of the
gate pre-activations onto relu(P_down x); "The Prediction Problem",
"Precision, recall, and which error hurts") against the oracle's fp64 fit,
its exact special case, and the recall it buys over a random up map."""
import math

import numpy as np
import pytest

import oracle
import synth
from _helpers import HostLayer, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


def device_bits_f64(t, dt):
    """A device storage tensor decoded to fp64 on the host."""
    if dt == synth.BF16:
        return synth.storage_to_f64(t.cpu().view(torch.int16).numpy().view(np.uint16), dt)
    return t.cpu().numpy().astype(np.float64)


@pytest.mark.parametrize("dt,tol", [(synth.F32, 1e-4), (synth.F16, 2e-3)])
def test_fit_matches_oracle(dt, tol):
    d, f, r, N, lam = 256, 1024, 64, 512, 2.0
    H = HostLayer(d, f, r, dt, seed=41, rho=0.1)
    layer, pred = H.device()
    X = synth.x_normal(42, N, d)
    cs.cs_fit_predictor(layer, pred, torch.from_numpy(X).cuda(), lam)
    got = device_bits_f64(pred.keep[1], dt)[:, :r]
    want = oracle.fit_predictor(H.oracle_layer(), H.oracle_pred(), X, lam)
    err = np.abs(got - want).max() / np.abs(want).max()
    assert err < tol, err


def test_fit_recovers_an_exactly_representable_layer():
    """P_down = [I; -I] and no bias: W x = [W, -W] relu-features exactly, so the
    fit returns [W, -W]."""
    d, f = 32, 200
    W = synth.normal_matrix(43, 0, f, d, 1 / math.sqrt(d), synth.F32)
    eye = np.concatenate([np.eye(d), -np.eye(d)]).astype(np.float32)
    wg, wd = torch.from_numpy(W).cuda(), torch.from_numpy(W).cuda()
    layer = cs.FfnLayer(wg, wd)
    pd = torch.from_numpy(eye).cuda()
    pu = torch.zeros((f, 2 * d), device="cuda")
    pred = cs.Predictor(pd, pu, d=d)
    X = synth.x_normal(44, 400, d)
    cs.cs_fit_predictor(layer, pred, torch.from_numpy(X).cuda(), 1e-6)
    np.testing.assert_allclose(pu.cpu().numpy(), np.concatenate([W, -W], axis=1), rtol=0, atol=1e-4)


def recall_precision(layer, pred, d, f, r, Xh, k):
    """Mean recall and precision of the predictor's top-k against the exact
    mask {g > 0}, both computed on the GPU, over held-out inputs."""
    ws = cs.Workspace(d, f, r)
    pre = torch.empty(f, device="cuda")
    ei = torch.empty(f, dtype=torch.int32, device="cuda")
    ec = torch.empty(1, dtype=torch.int32, device="cuda")
    y = torch.empty(d, device="cuda")
    sc = torch.empty((1, f), device="cuda")
    pi = torch.empty((1, f), dtype=torch.int32, device="cuda")
    pc = torch.empty(1, dtype=torch.int32, device="cuda")
    rec, prec = [], []
    for x in Xh:
        xt = torch.from_numpy(x[None]).cuda()
        cs.cs_exact_ffn(layer, xt, pre, ei, ec, y, ws)
        cs.cs_predict(pred, xt, sc, ws)
        cs.cs_select(sc, cs.select_params(cs.CS_SEL_TOPK, k), pi, pc, ws=ws)
        torch.cuda.synchronize()
        ex = ei.cpu().numpy()[:int(ec.item())]
        pr = pi.cpu().numpy()[0, :int(pc.item())]
        r_, p_ = oracle.recall_precision(pr, ex, f)
        rec.append(r_)
        prec.append(p_)
    return float(np.mean(rec)), float(np.mean(prec))


def test_fitted_predictor_beats_a_random_one():
    d, f, r, N = 1024, 4096, 256, 2048
    H = HostLayer(d, f, r, synth.F16, seed=45, rho=0.1)
    layer, pred = H.device()
    Xh = synth.x_normal(46, 16, d)
    k = 2 * synth.ceil_k(f, 0.1)
    rec0, _ = recall_precision(layer, pred, d, f, r, Xh, k)
    cs.cs_fit_predictor(layer, pred, torch.from_numpy(synth.x_normal(47, N, d)).cuda(), 1e-3 * N)
    rec1, prec1 = recall_precision(layer, pred, d, f, r, Xh, k)
    assert rec0 < 0.35                      # a random up map: recall near k / f = 0.2
    assert rec1 > 0.5 and rec1 > rec0 + 0.2, (rec0, rec1)
    assert prec1 > 0.2


def test_fit_rejects_bad_arguments():
    d, f, r = 64, 128, 8
    H = HostLayer(d, f, r, synth.F16, seed=48)
    layer, pred = H.device()
    X = torch.from_numpy(synth.x_normal(49, 16, d)).cuda()
    with pytest.raises(cs.CsError):
        cs.cs_fit_predictor(layer, pred, X, -1.0)          # negative ridge
    other = HostLayer(d, f + 32, r, synth.F16, seed=48)
    _, pred2 = other.device()
    with pytest.raises(cs.CsError):
        cs.cs_fit_predictor(layer, pred2, X, 1.0)          # predictor for another layer
    with pytest.raises(ValueError):
        cs.cs_fit_predictor(layer, pred, X.half(), 1.0)    # X must be fp32
