"""GPU parity of the frequency-sorted layout with a hot prefix ("Kernel-Level
Implementation": neurons pre-sorted by how often they fire; "Static
locality: hot and cold neurons").

The layout step (cs_permute_rows) must reproduce the oracle's row order bit
for bit; the selection with a hot prefix must give the oracle's ids, counts
and masks bit for bit; and the whole decode step on the permuted layout must
match the oracle there and, with the ids mapped back, the unpermuted layer."""
import numpy as np
import pytest

import oracle
import synth
from _helpers import TOL, HostLayer, pick_k_with_gap, rel_err, score_bounds, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


def storage_bits(t, dt):
    """A device tensor's storage bits as a numpy array (for bit comparisons)."""
    if dt == synth.BF16:
        return t.cpu().view(torch.int16).numpy().view(np.uint16)
    a = t.cpu().numpy()
    return a.view(np.uint16) if dt == synth.F16 else a.view(np.uint32)


def host_bits(a, dt):
    a = np.ascontiguousarray(a)
    return a.view(np.uint16) if dt in (synth.F16, synth.BF16) else a.view(np.uint32)


# ---------------------------------------------------------------- selection

@pytest.mark.parametrize("f_tail,hot", [(40, 64), (1000, 32), (2047, 1024), (19456, 1024), (27648, 1024)])
@pytest.mark.parametrize("B", [1, 3])
def test_select_hot_bit_exact(f_tail, hot, B):
    S = np.stack([synth.score_vector(50 + b, f_tail, ties=f_tail // 10, specials=bool(b % 2))
                  for b in range(B)])
    scores = torch.from_numpy(S).cuda()
    f = hot + f_tail
    W = (f + 31) // 32
    cases = [(cs.CS_SEL_TOPK, 0, 0.0), (cs.CS_SEL_TOPK, 1, 0.0), (cs.CS_SEL_TOPK, f_tail // 10, 0.0),
             (cs.CS_SEL_TOPK, f_tail, 0.0), (cs.CS_SEL_THRESHOLD, 0, 0.5)]
    for mode, k, tau in cases:
        idx = torch.full((B, f), -7, dtype=torch.int32, device="cuda")
        cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
        mask = torch.zeros((B, W), dtype=torch.int32, device="cuda")
        cs.cs_select(scores, cs.select_params(mode, k, tau, hot=hot), idx, cnt, mask=mask)
        torch.cuda.synchronize()
        I, N, M = idx.cpu().numpy(), cnt.cpu().numpy(), mask.cpu().numpy().view(np.uint32)
        omode = oracle.SEL_TOPK if mode == cs.CS_SEL_TOPK else oracle.SEL_THRESHOLD
        for b in range(B):
            want = oracle.select_hot(S[b], hot, omode, k=k, tau=tau)
            assert N[b] == want.size, (mode, k, b)
            assert np.array_equal(I[b, :N[b]], want), (mode, k, b)
            assert np.all(I[b, N[b]:] == -7)
            assert np.array_equal(M[b], synth.bits_from_bool(np.isin(np.arange(f), want))), (mode, k, b)


# ------------------------------------------------------------------- layout

@pytest.mark.parametrize("dt", [synth.F32, synth.F16, synth.BF16])
def test_permute_rows_bit_exact(dt):
    from _helpers import pad_ld
    f, d, hot = 3000, 200, 512
    A = synth.normal_matrix(1, 2, f, d, 0.1, dt, ld=pad_ld(d, dt))
    perm = oracle.hot_order(synth.firing_probs(1, 0, f, 0.1))
    perm_d = torch.from_numpy(perm).cuda()
    src = upload(A, dt)
    dst = torch.empty_like(src)
    cs.cs_permute_rows(src, perm_d, dst)
    tail = torch.empty((f - hot, src.shape[1]), dtype=src.dtype, device="cuda")
    cs.cs_permute_rows(src, perm_d[hot:], tail)
    b = torch.from_numpy(synth.zipf_bias(1, 0, f, 0.1)).cuda()
    bp = torch.empty_like(b)
    cs.cs_permute_rows(b, perm_d, bp)
    # an entry outside [0, f) gives a zero row
    bad = perm_d.clone()
    bad[5] = f
    z = torch.full_like(src, 7)
    cs.cs_permute_rows(src, bad, z)
    torch.cuda.synchronize()
    assert np.array_equal(storage_bits(dst, dt), host_bits(oracle.permute_rows(A, perm), dt))
    assert np.array_equal(storage_bits(tail, dt), host_bits(oracle.permute_rows(A, perm[hot:]), dt))
    assert np.array_equal(bp.cpu().numpy(), oracle.permute_rows(synth.zipf_bias(1, 0, f, 0.1), perm))
    zb = storage_bits(z, dt)
    assert np.all(zb[5] == 0) and np.array_equal(zb[6], host_bits(A, dt)[perm[6]])


# ---------------------------------------------------------- the whole step

class TailPredictor:
    """The predictor of a hot layout: P_down as is, P_up's rows for the tail
    neurons in layout order (host storage arrays, for the oracle)."""

    def __init__(self, H, perm, hot):
        self.d, self.r, self.dt, self.ld, self.ldr = H.d, H.r, H.dt, H.ld, H.ldr
        self.f = H.f - hot
        self.p_down = H.p_down
        self.p_up = oracle.permute_rows(H.p_up, perm[hot:])

    def oracle_pred(self):
        return oracle.Predictor(self.d, self.r, self.f, self.dt, self.p_down, self.p_up,
                                ld_down=self.ld, ld_up=self.ldr)


def hot_device_layout(H, perm, hot):
    """Upload the unpermuted layer, then build the hot layout on the GPU."""
    layer0, pred0 = H.device()
    perm_d = torch.from_numpy(perm).cuda()
    keep = {}
    for name in ("w_gate", "w_down_t", "w_up"):
        src = getattr(layer0, name)
        if src is None:
            keep[name] = None
            continue
        keep[name] = torch.empty_like(src)
        cs.cs_permute_rows(src, perm_d, keep[name])
    keep["bias"] = torch.empty_like(layer0.bias)
    cs.cs_permute_rows(layer0.bias, perm_d, keep["bias"])
    pd, pu = pred0.keep
    keep["p_up"] = torch.empty((H.f - hot, pu.shape[1]), dtype=pu.dtype, device="cuda")
    cs.cs_permute_rows(pu, perm_d[hot:], keep["p_up"])
    layer = cs.FfnLayer(keep["w_gate"], keep["w_down_t"], w_up=keep["w_up"], bias=keep["bias"], d=H.d)
    pred = cs.Predictor(pd, keep["p_up"], d=H.d)
    torch.cuda.synchronize()
    return layer, pred, keep


HOT_CASES = [
    ("opt13b-f16-hot1024", 5120, 20480, 512, synth.F16, False, 1024, 0.05),
    ("glu-bf16-hot256", 2048, 6000, 128, synth.BF16, True, 256, 0.10),
]


@pytest.mark.parametrize("case", HOT_CASES, ids=[c[0] for c in HOT_CASES])
def test_hot_step(case):
    name, d, f, r, dt, glu, hot, share = case
    H = HostLayer(d, f, r, dt, glu=glu, seed=0, rho=0.10)
    perm = oracle.hot_order(synth.firing_probs(0, 0, f, 0.10))
    layer, pred, keep = hot_device_layout(H, perm, hot)
    assert np.array_equal(storage_bits(keep["w_gate"], dt), host_bits(oracle.permute_rows(H.w_gate, perm), dt))
    Lp = oracle.Layer(d, f, dt, oracle.permute_rows(H.w_gate, perm), oracle.permute_rows(H.w_down_t, perm),
                      w_up=oracle.permute_rows(H.w_up, perm) if glu else None,
                      bias=oracle.permute_rows(H.bias, perm), ld=H.ld)
    T = TailPredictor(H, perm, hot)
    X = synth.x_normal(61, 1, d)
    s_ref, eps = score_bounds(T, X[0])
    k = pick_k_with_gap(s_ref, eps, synth.ceil_k(f, share))
    params = cs.select_params(cs.CS_SEL_TOPK, k, hot=hot)
    ws = cs.Workspace(d, f, r)
    x = torch.from_numpy(X).cuda()
    scores = torch.empty((1, f - hot), device="cuda")
    idx = torch.full((1, f), -1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    y = torch.empty((1, d), device="cuda")
    cs.cs_predict(pred, x, scores, ws)
    cs.cs_select(scores, params, idx, cnt, ws=ws)
    cs.cs_sparse_ffn(layer, x, idx[0], cnt, y, ws)
    torch.cuda.synchronize()
    s = scores.cpu().numpy()[0]
    assert np.all(np.abs(s - s_ref) <= eps + 1e-30)
    n = int(cnt.item())
    want = oracle.select_hot(s_ref.astype(np.float32), hot, oracle.SEL_TOPK, k=k)
    assert n == hot + k and np.array_equal(idx.cpu().numpy()[0, :n], want)
    gy = y.cpu().numpy()[0]
    assert rel_err(gy, oracle.ffn(Lp, X[0], want)) < TOL
    # the same neurons in the original numbering, on the unpermuted layer
    assert rel_err(gy, oracle.ffn(H.oracle_layer(), X[0], np.sort(perm[want]))) < TOL
    # one call per token does the same, bit for bit
    y2 = torch.empty(d, device="cuda")
    s2 = torch.cuda.Stream()
    torch.cuda.synchronize()
    cs.cs_decode_layer(layer, pred, x[0], y2, params, ws, stream=s2)
    s2.synchronize()
    assert np.array_equal(y2.cpu().numpy().view(np.uint32), gy.view(np.uint32))
    assert cs.cs_get_device_error(ws) == 0


@pytest.mark.parametrize("mode", [cs.CS_STACK_SEQUENTIAL, cs.CS_STACK_LOOKAHEAD])
def test_hot_stack_extremes(mode):
    """No tail budget: every layer takes exactly the prefix; the whole tail:
    every neuron.  Traces and x_L against the oracle's stack."""
    Ls, d, f, r, hot, dt = 3, 512, 2048, 64, 256, synth.F16
    Hs = [HostLayer(d, f, r, dt, seed=0, layer=l, rho=0.1) for l in range(Ls)]
    layers, preds, keep = [], [], []
    opreds = []
    for Hh in Hs:
        lay, _ = Hh.device()
        pd, pu = upload(Hh.p_down, dt), upload(np.ascontiguousarray(Hh.p_up[hot:]), dt)
        keep.append((lay, pd, pu))
        layers.append(lay)
        preds.append(cs.Predictor(pd, pu, d=d))
        opreds.append(oracle.Predictor(d, r, f - hot, dt, Hh.p_down, np.ascontiguousarray(Hh.p_up[hot:]),
                                       ld_down=Hh.ld, ld_up=Hh.ldr))
    olayers = [Hh.oracle_layer() for Hh in Hs]
    omode = oracle.LOOKAHEAD if mode == cs.CS_STACK_LOOKAHEAD else oracle.SEQUENTIAL
    X = synth.x_normal(12, 1, d)[0]
    for k, ids in ((0, np.arange(hot)), (f - hot, np.arange(f))):
        x = torch.from_numpy(X.copy()).cuda()
        ws = cs.Workspace(d, f, r)
        tc = torch.zeros(Ls, dtype=torch.int32, device="cuda")
        ti = torch.zeros((Ls, f), dtype=torch.int32, device="cuda")
        torch.cuda.synchronize()
        cs.cs_decode_stack(layers, preds, x, 0.1, cs.select_params(cs.CS_SEL_TOPK, k, hot=hot), mode, ws,
                           s_main=torch.cuda.Stream(), s_pred=torch.cuda.Stream(), trace_count=tc, trace_idx=ti)
        torch.cuda.synchronize()
        TC, TI = tc.cpu().numpy(), ti.cpu().numpy()
        for l in range(Ls):
            assert TC[l] == ids.size and np.array_equal(TI[l, :TC[l]], ids), (k, l)
        want = oracle.stack(olayers, opreds, X, mode=omode, k=k, hot=hot, resid_scale=0.1)
        assert rel_err(x.cpu().numpy(), want) < TOL
        assert cs.cs_get_device_error(ws) == 0
