"""GPU parity of head-sparse attention (cs_sparse_attention: "Contextual
Sparsity and Activation Predictors", first section; "The Empirical
Foundation"; "Implications for System Design") against the oracle, alone and
behind the predictor and top-k that choose the heads."""
import math

import numpy as np
import pytest

import oracle
import synth
from _helpers import TOL, pick_k_with_gap, rel_err, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


def attn_case(d, H, dh, S, dt, seed):
    sd = 1 / math.sqrt(d)
    wq = synth.normal_matrix(seed, 0, H * dh, d, sd, dt)
    wo = synth.normal_matrix(seed, 1, H * dh, d, 1 / math.sqrt(dh), dt)
    kc = synth.normal_matrix(seed, 2, H * S, dh, 1.0, dt)
    vc = synth.normal_matrix(seed, 3, H * S, dh, 1.0, dt)
    A = oracle.AttnLayer(d, H, dh, dt, wq, wo)
    dev = dict(wq=upload(wq, dt), wo=upload(wo, dt), k=upload(kc, dt).view(H, S, dh), v=upload(vc, dt).view(H, S, dh))
    return A, dev, kc.reshape(H, S, dh), vc.reshape(H, S, dh)


def run_attn(dev, H, d, x, heads, ws=None):
    layer = cs.AttnLayer(dev["wq"], dev["wo"], H)
    ws = ws or cs.Workspace(d, 64, 8)
    hd = torch.tensor(list(heads) if len(heads) else [0], dtype=torch.int32, device="cuda")
    cnt = torch.tensor([len(heads)], dtype=torch.int32, device="cuda")
    y = torch.full((d,), float("nan"), device="cuda")
    cs.cs_sparse_attention(layer, torch.from_numpy(x).cuda(), hd, cnt, dev["k"], dev["v"], y, ws)
    torch.cuda.synchronize()
    return y.cpu().numpy(), ws


CASES = [(64, 4, 8, 1), (256, 8, 32, 7), (1024, 16, 64, 300), (5120, 40, 128, 2048), (2048, 16, 256, 33)]


@pytest.mark.parametrize("dt", [synth.F32, synth.F16, synth.BF16])
@pytest.mark.parametrize("case", CASES, ids=[f"d{c[0]}-H{c[1]}-dh{c[2]}-S{c[3]}" for c in CASES])
def test_attention_parity(dt, case):
    d, H, dh, S = case
    if dt == synth.F32 and dh < 4:
        pytest.skip("d_head below one 16-byte vector")
    A, dev, kc, vc = attn_case(d, H, dh, S, dt, seed=d + S)
    x = synth.x_normal(d, 1, d)[0]
    rng = np.random.default_rng(S)
    for heads in (sorted(rng.choice(H, size=max(1, H // 3), replace=False).tolist()), list(range(H)), []):
        y, ws = run_attn(dev, H, d, x, heads)
        want = oracle.attention(A, x, heads, kc, vc)
        if not heads:
            assert np.all(y == 0)
        else:
            assert rel_err(y, want) < TOL, (heads, rel_err(y, want))
        assert cs.cs_get_device_error(ws) == 0


def test_attention_flags_bad_ids_and_counts():
    d, H, dh, S = 256, 8, 32, 16
    A, dev, kc, vc = attn_case(d, H, dh, S, synth.F16, seed=3)
    x = synth.x_normal(4, 1, d)[0]
    y, ws = run_attn(dev, H, d, x, [1, 99])       # 99 is skipped and flagged
    assert rel_err(y, oracle.attention(A, x, [1], kc, vc)) < TOL
    assert cs.cs_get_device_error(ws, clear=True) & cs.CS_DEVERR_INDEX
    layer = cs.AttnLayer(dev["wq"], dev["wo"], H)
    hd = torch.arange(H, dtype=torch.int32, device="cuda")
    cnt = torch.tensor([H + 5], dtype=torch.int32, device="cuda")   # clamped to H and flagged
    yy = torch.empty(d, device="cuda")
    cs.cs_sparse_attention(layer, torch.from_numpy(x).cuda(), hd, cnt, dev["k"], dev["v"], yy, ws)
    torch.cuda.synchronize()
    assert rel_err(yy.cpu().numpy(), oracle.attention(A, x, list(range(H)), kc, vc)) < TOL
    assert cs.cs_get_device_error(ws) & cs.CS_DEVERR_COUNT


def test_attention_step_with_predicted_heads():
    """A predictor with one output per head, top-k heads (ids bit-exact when the
    boundary is decided beyond rounding), then the attention."""
    d, H, dh, S, r = 2048, 32, 64, 512, 64
    A, dev, kc, vc = attn_case(d, H, dh, S, synth.BF16, seed=11)
    sd = 1 / math.sqrt(d)
    pd = synth.normal_matrix(12, 0, r, d, sd, synth.BF16)
    pu = synth.normal_matrix(12, 1, H, r, 1 / math.sqrt(r), synth.BF16)
    P = oracle.Predictor(d, r, H, synth.BF16, pd, pu)
    pred = cs.Predictor(upload(pd, synth.BF16), upload(pu, synth.BF16))
    x = synth.x_normal(13, 1, d)
    _, s_ref = oracle.predict(P, x[0])
    s32 = s_ref.astype(np.float32)
    order = np.sort(s_ref)[::-1]
    gaps = order[:-1] - order[1:]
    k = int(np.argmax(gaps[4:12])) + 5        # a boundary between 5 and 12 heads with the widest gap
    ws = cs.Workspace(d, H, r)
    sc = torch.empty((1, H), device="cuda")
    hd = torch.empty((1, H), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    y = torch.empty(d, device="cuda")
    xt = torch.from_numpy(x).cuda()
    cs.cs_predict(pred, xt, sc, ws)
    cs.cs_select(sc, cs.select_params(cs.CS_SEL_TOPK, k), hd, cnt, ws=ws)
    cs.cs_sparse_attention(cs.AttnLayer(dev["wq"], dev["wo"], H), xt[0], hd[0], cnt, dev["k"], dev["v"], y, ws)
    torch.cuda.synchronize()
    got = hd.cpu().numpy()[0, :int(cnt.item())]
    assert np.array_equal(got, oracle.select_topk(s32, k))
    assert rel_err(y.cpu().numpy(), oracle.attention(A, x[0], got, kc, vc)) < TOL
    assert cs.cs_get_device_error(ws) == 0


def _predicted_heads_case():
    d, H, dh, S, r = 2048, 32, 64, 512, 64
    A, dev, kc, vc = attn_case(d, H, dh, S, synth.BF16, seed=11)
    sd = 1 / math.sqrt(d)
    pd = synth.normal_matrix(12, 0, r, d, sd, synth.BF16)
    pu = synth.normal_matrix(12, 1, H, r, 1 / math.sqrt(r), synth.BF16)
    P = oracle.Predictor(d, r, H, synth.BF16, pd, pu)
    pred = cs.Predictor(upload(pd, synth.BF16), upload(pu, synth.BF16))
    return d, H, r, A, dev, kc, vc, P, pred


def _widest_gap_k(s_ref, lo, hi):
    order = np.sort(s_ref)[::-1]
    gaps = order[:-1] - order[1:]
    return int(np.argmax(gaps[lo - 1:hi - 1])) + lo


@pytest.mark.parametrize("io", ["device", "pinned", "pinned_x", "pinned_y"])
@pytest.mark.parametrize("mode", ["topk", "threshold"])
def test_decode_attention_one_call(io, mode):
    """cs_decode_attention (predictor, head selection and attention as one
    cached graph, x and y on the device or in pinned host memory): the same
    heads and bit for bit the same y as the three calls, over tokens that
    re-point the graph's copy kernels; heads against the oracle's selection
    and y against the oracle's attention."""
    d, H, r, A, dev, kc, vc, P, pred = _predicted_heads_case()
    layer = cs.AttnLayer(dev["wq"], dev["wo"], H)
    ws = cs.Workspace(d, H, r)
    X = synth.x_normal(21, 3, d)
    xs_d = torch.from_numpy(X).cuda()
    xs_h = torch.from_numpy(X).pin_memory()
    ys_h = torch.full((3, d), float("nan")).pin_memory()
    ys_d = torch.full((3, d), float("nan"), device="cuda")
    sc = torch.empty((1, H), device="cuda")
    hd3 = torch.empty((1, H), dtype=torch.int32, device="cuda")
    cnt3 = torch.empty(1, dtype=torch.int32, device="cuda")
    y3 = torch.empty(d, device="cuda")
    hd = torch.full((H,), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    for t in range(3):
        _, s_ref = oracle.predict(P, X[t])
        s32 = s_ref.astype(np.float32)
        if mode == "topk":
            k = _widest_gap_k(s_ref, 5, 12)
            params = cs.select_params(cs.CS_SEL_TOPK, k)
            want = oracle.select_topk(s32, k)
        else:
            k = _widest_gap_k(s_ref, 4, 16)
            order = np.sort(s32)[::-1]
            tau = float((order[k - 1] + order[k]) / 2)
            params = cs.select_params(cs.CS_SEL_THRESHOLD, 0, tau)
            want = oracle.select_threshold(s32, np.float32(tau))
        cs.cs_predict(pred, xs_d[t:t + 1], sc, ws)
        cs.cs_select(sc, params, hd3, cnt3, ws=ws)
        cs.cs_sparse_attention(layer, xs_d[t], hd3[0], cnt3, dev["k"], dev["v"], y3, ws)
        x_in = xs_h[t] if io in ("pinned", "pinned_x") else xs_d[t]
        y_out = ys_h[t] if io in ("pinned", "pinned_y") else ys_d[t]
        cs.cs_decode_attention(layer, pred, x_in, y_out, params, dev["k"], dev["v"], ws, heads=hd, count=cnt)
        torch.cuda.synchronize()
        n = int(cnt.item())
        assert n == int(cnt3.item()) == want.size, (t, n, want.size)
        got = hd.cpu().numpy()[:n]
        assert np.array_equal(got, hd3.cpu().numpy()[0, :n])
        assert np.array_equal(got, want)
        y = y_out.cpu().numpy()
        assert np.array_equal(y, y3.cpu().numpy())
        assert rel_err(y, oracle.attention(A, X[t], got, kc, vc)) < TOL
    assert cs.cs_get_device_error(ws) == 0


def test_decode_attention_without_head_outputs():
    """Without heads / count the workspace holds them; y is unchanged."""
    d, H, r, A, dev, kc, vc, P, pred = _predicted_heads_case()
    layer = cs.AttnLayer(dev["wq"], dev["wo"], H)
    ws = cs.Workspace(d, H, r)
    x = synth.x_normal(22, 1, d)
    _, s_ref = oracle.predict(P, x[0])
    k = _widest_gap_k(s_ref, 5, 12)
    params = cs.select_params(cs.CS_SEL_TOPK, k)
    xt = torch.from_numpy(x[0]).cuda()
    y1 = torch.empty(d, device="cuda")
    y2 = torch.empty(d, device="cuda")
    hd = torch.empty(H, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    cs.cs_decode_attention(layer, pred, xt, y1, params, dev["k"], dev["v"], ws)
    cs.cs_decode_attention(layer, pred, xt, y2, params, dev["k"], dev["v"], ws, heads=hd, count=cnt)
    torch.cuda.synchronize()
    assert np.array_equal(y1.cpu().numpy(), y2.cpu().numpy())
    want = oracle.select_topk(s_ref.astype(np.float32), k)
    assert np.array_equal(hd.cpu().numpy()[:int(cnt.item())], want)
    assert rel_err(y1.cpu().numpy(), oracle.attention(A, x[0], want, kc, vc)) < TOL
    with pytest.raises(cs.CsError):
        cs.cs_decode_attention(layer, pred, xt, xt, params, dev["k"], dev["v"], ws)


@pytest.mark.parametrize("sel", ["k0", "tau_inf", "all"])
def test_decode_attention_edge_selections(sel):
    """No head chosen (k = 0, or a threshold above every score): y = 0 and
    count 0; every head chosen: the full attention, against the oracle."""
    d, H, r, A, dev, kc, vc, P, pred = _predicted_heads_case()
    layer = cs.AttnLayer(dev["wq"], dev["wo"], H)
    ws = cs.Workspace(d, H, r)
    x = synth.x_normal(23, 1, d)
    params = {"k0": cs.select_params(cs.CS_SEL_TOPK, 0),
              "tau_inf": cs.select_params(cs.CS_SEL_THRESHOLD, 0, float("inf")),
              "all": cs.select_params(cs.CS_SEL_TOPK, H + 3)}[sel]
    y = torch.full((d,), float("nan")).pin_memory()
    hd = torch.full((H,), -1, dtype=torch.int32, device="cuda")
    cnt = torch.full((1,), -1, dtype=torch.int32, device="cuda")
    cs.cs_decode_attention(layer, pred, torch.from_numpy(x[0]).pin_memory(), y, params, dev["k"], dev["v"], ws,
                           heads=hd, count=cnt)
    torch.cuda.synchronize()
    n = int(cnt.item())
    if sel == "all":
        assert n == H and np.array_equal(hd.cpu().numpy(), np.arange(H))
        assert rel_err(y.numpy(), oracle.attention(A, x[0], list(range(H)), kc, vc)) < TOL
    else:
        assert n == 0
        assert np.all(y.numpy() == 0)
    assert cs.cs_get_device_error(ws) == 0
