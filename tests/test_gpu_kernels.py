"""GPU parity: each entry point against the CPU oracle on the same seeded
inputs.  Indices and masks must match bit for bit; scores and y within
TOL = 2e-3 (infinity-norm relative)."""
import math

import numpy as np
import pytest

import oracle
import synth
from _helpers import TOL, HostLayer, rel_err, upload

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402

DTYPES = [synth.F32, synth.F16, synth.BF16]


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()
    yield
    torch.cuda.synchronize()


def ws_for(d, f, r, B=1):
    return cs.Workspace(d, f, r, B)


def dev_err(ws):
    return cs.cs_get_device_error(ws, clear=True)


# ------------------------------------------------------------------- synth

@pytest.mark.parametrize("dt", DTYPES)
def test_device_generator_matches_host(dt):
    import synth.device as sd
    sd.build()
    rows, cols, ld = 129, 77, 80
    t = torch.empty((rows, ld), dtype={0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[dt],
                    device="cuda")
    sd.fill_normal(t, 5, 17, 0.25, cols=cols)
    host = synth.normal_matrix(5, 17, rows, cols, 0.25, dt, ld=ld)
    got = t.cpu()
    got = got.view(torch.int16).numpy().view(np.uint16) if dt == synth.BF16 else got.numpy()
    assert np.array_equal(got.view(np.uint8), host.view(np.uint8))


# --------------------------------------------------------------- predictor

@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("shape", [(3, 3, 4), (100, 17, 333), (512, 64, 2048), (1000, 40, 777)])
@pytest.mark.parametrize("B", [1, 3, 6])
def test_predict(dt, shape, B):
    d, r, f = shape
    H = HostLayer(d, f, r, dt, seed=1)
    _, pred = H.device()
    X = synth.x_normal(2, B, d)
    x = torch.from_numpy(X).cuda()
    scores = torch.empty((B, f), device="cuda")
    ws = ws_for(d, f, r, B)
    cs.cs_predict(pred, x, scores, ws)
    got = scores.cpu().numpy()
    for b in range(B):
        _, s = oracle.predict(H.oracle_pred(), X[b])
        assert rel_err(got[b], s) < TOL
        assert rel_err(got[b], s) < 1e-5  # fp32 accumulation is far inside the bar
    assert dev_err(ws) == 0


# --------------------------------------------------------------- selection

SEL_F = [1, 7, 33, 40, 64, 65, 1000, 2048, 20480, 32768, 49152]


@pytest.mark.parametrize("f", SEL_F)
def test_topk_bit_exact(f):
    B = 3
    S = np.stack([synth.score_vector(10 * f + b, f, ties=f // 4, specials=(b == 1),
                                     quantize=0.05 if b == 2 else None) for b in range(B)])
    s = torch.from_numpy(S).cuda()
    idx = torch.full((B, f), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
    words = (f + 31) // 32
    mask = torch.zeros((B, words), dtype=torch.int32, device="cuda")
    for k in sorted({0, 1, f // 3, f // 2, f - 1, f, f + 5}):
        cs.cs_select(s, cs.select_params(cs.CS_SEL_TOPK, k), idx, cnt, mask)
        I, N, M = idx.cpu().numpy(), cnt.cpu().numpy(), mask.cpu().numpy().view(np.uint32)
        for b in range(B):
            want = oracle.select_topk(S[b], k)
            assert N[b] == want.size, (f, k, b)
            assert np.array_equal(I[b, :N[b]], want), (f, k, b)
            assert np.array_equal(M[b], synth.bits_from_bool(np.isin(np.arange(f), want)))


def _tail_rows(f, seed):
    """Rows that stress the bounds of the selection's bucket map: heavy tails,
    a few huge outliers, a mostly-zero row, and a row whose every fourth score
    is one constant (a sample of ids on any grid of multiples of 4 sees no
    spread there)."""
    rng = np.random.default_rng(seed)
    cauchy = rng.standard_cauchy(f).astype(np.float32)
    outl = rng.standard_normal(f).astype(np.float32)
    outl[rng.choice(f, 5, replace=False)] = np.array([1e30, -1e30, 3e29, 1e20, -7e25], np.float32)
    sparse = np.zeros(f, np.float32)
    sparse[rng.choice(f, 100, replace=False)] = rng.random(100).astype(np.float32) + 0.25
    grid = rng.standard_normal(f).astype(np.float32)
    grid[::4] = 0.5
    return np.stack([cauchy, outl, sparse, grid])


@pytest.mark.parametrize("f", [2048, 28672, 49152])
def test_topk_heavy_tails_bit_exact(f):
    S = _tail_rows(f, 31 + f)
    B = S.shape[0]
    s = torch.from_numpy(S).cuda()
    idx = torch.full((B, f), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
    mask = torch.zeros((B, (f + 31) // 32), dtype=torch.int32, device="cuda")
    for k in sorted({1, 3, 5, 6, 50, 100, 101, f // 100, f // 7, f // 4, f // 2, f - 2}):
        cs.cs_select(s, cs.select_params(cs.CS_SEL_TOPK, k), idx, cnt, mask)
        I, N, M = idx.cpu().numpy(), cnt.cpu().numpy(), mask.cpu().numpy().view(np.uint32)
        for b in range(B):
            want = oracle.select_topk(S[b], k)
            assert N[b] == want.size, (f, k, b)
            assert np.array_equal(I[b, :N[b]], want), (f, k, b)
            assert np.array_equal(M[b], synth.bits_from_bool(np.isin(np.arange(f), want))), (f, k, b)


@pytest.mark.parametrize("f", SEL_F)
def test_threshold_bit_exact(f):
    B = 2
    S = np.stack([synth.score_vector(f + b, f, ties=f // 8, specials=True, quantize=0.1)
                  for b in range(B)])
    s = torch.from_numpy(S).cuda()
    idx = torch.zeros((B, f), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(B, dtype=torch.int32, device="cuda")
    for tau in (-np.inf, -0.3, 0.0, 0.1, 1.2816, np.inf, np.nan):
        cs.cs_select(s, cs.select_params(cs.CS_SEL_THRESHOLD, 0, tau), idx, cnt)
        I, N = idx.cpu().numpy(), cnt.cpu().numpy()
        for b in range(B):
            want = oracle.select_threshold(S[b], tau)
            assert N[b] == want.size and np.array_equal(I[b, :N[b]], want), (f, tau)


COOP_F = [1024, 1057, 2048, 4900, 20480, 32768, 49152]


@pytest.mark.parametrize("f", COOP_F)
def test_topk_single_row_bit_exact(f):
    """Single rows at large f, every k from 0 to past f, with ties, specials
    and a coarse quantisation (masses of equal scores), repeated on one
    workspace."""
    ws = ws_for(64, f, 8)
    idx = torch.full((1, f), -7, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    mask = torch.zeros((1, (f + 31) // 32), dtype=torch.int32, device="cuda")
    for variant in range(4):
        S = synth.score_vector(7 * f + variant, f, ties=f // 3 if variant else 0,
                               specials=variant == 2, quantize=0.02 if variant == 3 else None)[None]
        s = torch.from_numpy(S).cuda()
        for k in sorted({0, 1, 2, f // 10, f // 3, f // 2, f - 1, f, f + 5}):
            cs.cs_select(s, cs.select_params(cs.CS_SEL_TOPK, k), idx, cnt, mask, ws=ws)
            want = oracle.select_topk(S[0], k)
            n = int(cnt.item())
            assert n == want.size, (f, k, variant)
            assert np.array_equal(idx.cpu().numpy()[0, :n], want), (f, k, variant)
            assert np.array_equal(mask.cpu().numpy()[0].view(np.uint32),
                                  synth.bits_from_bool(np.isin(np.arange(f), want)))
        for tau in (-np.inf, 0.0, 0.7, np.nan):
            cs.cs_select(s, cs.select_params(cs.CS_SEL_THRESHOLD, 0, tau), idx, cnt, mask, ws=ws)
            want = oracle.select_threshold(S[0], tau)
            n = int(cnt.item())
            assert n == want.size and np.array_equal(idx.cpu().numpy()[0, :n], want), (f, tau)
    # a mass of equal scores: the pivot bucket overflows the exact ranking and
    # the radix fallback resolves it
    S = np.zeros((1, f), np.float32)
    S[0, ::7] = 1.0
    s = torch.from_numpy(S).cuda()
    for k in (1, f // 7, f // 7 + 1, f // 2, f - 3):
        cs.cs_select(s, cs.select_params(cs.CS_SEL_TOPK, k), idx, cnt, mask, ws=ws)
        want = oracle.select_topk(S[0], k)
        n = int(cnt.item())
        assert n == want.size and np.array_equal(idx.cpu().numpy()[0, :n], want), (f, k)
    assert dev_err(ws) == 0


def test_select_rejects_bad_args():
    s = torch.zeros((1, 8), device="cuda")
    idx = torch.zeros((1, 8), dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(cs.CsError):
        cs.cs_select(s, cs.select_params(cs.CS_SEL_EXACT), idx, cnt)
    big = torch.zeros((1, 49153), device="cuda")
    with pytest.raises(cs.CsError):
        cs.cs_select(big, cs.select_params(cs.CS_SEL_TOPK, 3), torch.zeros((1, 49153), dtype=torch.int32, device="cuda"), cnt)


# ------------------------------------------------------------- sparse FFN

FFN_SHAPES = [(3, 4), (100, 333), (512, 2048), (1000, 1500), (5120, 1200), (8192, 700)]


@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("glu", [False, True])
@pytest.mark.parametrize("shape", FFN_SHAPES)
def test_sparse_ffn(dt, glu, shape):
    d, f = shape
    H = HostLayer(d, f, 0, dt, glu=glu, seed=3)
    layer, _ = H.device()
    O = H.oracle_layer()
    X = synth.x_normal(4, 1, d)
    x = torch.from_numpy(X).cuda()
    y = torch.empty((1, d), device="cuda")
    ws = ws_for(d, f, 1)
    rng = np.random.default_rng(d + f)
    for n in sorted({0, 1, min(f, 7), f // 10, f // 2, f}):
        sel = np.sort(rng.choice(f, size=n, replace=False)).astype(np.int32)
        idx = torch.from_numpy(np.concatenate([sel, np.zeros(1, np.int32)])).cuda()
        cnt = torch.tensor([n], dtype=torch.int32, device="cuda")
        cs.cs_sparse_ffn(layer, x, idx, cnt, y, ws)
        want = oracle.ffn(O, X[0], sel)
        got = y.cpu().numpy()[0]
        if n == 0:
            assert not got.any()
        else:
            assert rel_err(got, want) < TOL, (n, rel_err(got, want))
    assert dev_err(ws) == 0


@pytest.mark.parametrize("dt", [synth.F16, synth.BF16])
@pytest.mark.parametrize("B", [2, 3, 5])
@pytest.mark.parametrize("glu", [False, True])
def test_sparse_ffn_batched(dt, B, glu):
    d, f = 1024, 3000
    H = HostLayer(d, f, 0, dt, glu=glu, seed=5)
    layer, _ = H.device()
    O = H.oracle_layer()
    X = synth.x_normal(6, B, d)
    x = torch.from_numpy(X).cuda()
    y = torch.empty((B, d), device="cuda")
    ws = ws_for(d, f, 1, B)
    sel = np.sort(np.random.default_rng(1).choice(f, size=900, replace=False)).astype(np.int32)
    cs.cs_sparse_ffn(layer, x, torch.from_numpy(sel).cuda(),
                     torch.tensor([sel.size], dtype=torch.int32, device="cuda"), y, ws)
    Y = y.cpu().numpy()
    for b in range(B):
        assert rel_err(Y[b], oracle.ffn(O, X[b], sel)) < TOL


def test_sparse_ffn_is_deterministic():
    d, f = 5120, 4000
    H = HostLayer(d, f, 0, synth.F16, seed=6)
    layer, _ = H.device()
    x = torch.from_numpy(synth.x_normal(1, 1, d)).cuda()
    sel = torch.arange(0, f, 2, dtype=torch.int32, device="cuda")
    cnt = torch.tensor([sel.numel()], dtype=torch.int32, device="cuda")
    ws = ws_for(d, f, 1)
    outs = []
    for _ in range(3):
        y = torch.empty((1, d), device="cuda")
        cs.cs_sparse_ffn(layer, x, sel, cnt, y, ws)
        outs.append(y.cpu().numpy())
    assert all(np.array_equal(outs[0].view(np.uint32), o.view(np.uint32)) for o in outs[1:])


def test_sparse_ffn_flags_bad_index_and_count():
    d, f = 256, 100
    H = HostLayer(d, f, 0, synth.F16, seed=7)
    layer, _ = H.device()
    O = H.oracle_layer()
    X = synth.x_normal(1, 1, d)
    x = torch.from_numpy(X).cuda()
    y = torch.empty((1, d), device="cuda")
    ws = ws_for(d, f, 1)
    idx = torch.tensor([3, 500, 7, -2, 9], dtype=torch.int32, device="cuda")
    cs.cs_sparse_ffn(layer, x, idx, torch.tensor([5], dtype=torch.int32, device="cuda"), y, ws)
    assert dev_err(ws) & cs.CS_DEVERR_INDEX
    # the bad ids are skipped, the good ones summed
    assert rel_err(y.cpu().numpy()[0], oracle.ffn(O, X[0], np.array([3, 7, 9], np.int32))) < TOL
    big = torch.arange(0, f, dtype=torch.int32, device="cuda")
    cs.cs_sparse_ffn(layer, x, big, torch.tensor([f + 50], dtype=torch.int32, device="cuda"), y, ws)
    assert dev_err(ws) & cs.CS_DEVERR_COUNT
    assert rel_err(y.cpu().numpy()[0], oracle.dense_ffn(O, X[0])) < TOL


def test_sparse_ffn_rejects_bad_layout():
    d, f = 100, 10
    w = torch.zeros((f, 100), dtype=torch.float16, device="cuda")  # 200-byte rows: not 16-aligned
    layer = cs.FfnLayer(w, w, d=d)
    x = torch.zeros((1, d), device="cuda")
    y = torch.zeros((1, d), device="cuda")
    ws = ws_for(d, f, 1)
    with pytest.raises(cs.CsError):
        cs.cs_sparse_ffn(layer, x, torch.zeros(1, dtype=torch.int32, device="cuda"),
                         torch.zeros(1, dtype=torch.int32, device="cuda"), y, ws)
    small = cs.Workspace(d, f, 1)
    small.nbytes = 256
    ok = cs.FfnLayer(torch.zeros((f, 104), dtype=torch.float16, device="cuda"),
                     torch.zeros((f, 104), dtype=torch.float16, device="cuda"), d=d)
    with pytest.raises(cs.CsError):
        cs.cs_sparse_ffn(ok, x, torch.zeros(1, dtype=torch.int32, device="cuda"),
                         torch.zeros(1, dtype=torch.int32, device="cuda"), y, small)


# --------------------------------------------------------------- exact mask

@pytest.mark.parametrize("dt", DTYPES)
@pytest.mark.parametrize("glu", [False, True])
@pytest.mark.parametrize("shape", [(64, 100), (1000, 3001), (5120, 20480)])
def test_exact_ffn(dt, glu, shape):
    d, f = shape
    H = HostLayer(d, f, 0, dt, glu=glu, seed=8)
    layer, _ = H.device()
    O = H.oracle_layer()
    X = synth.x_normal(9, 1, d)
    x = torch.from_numpy(X).cuda()
    pre = torch.empty(f, device="cuda")
    idx = torch.empty(f, dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    mask = torch.empty((f + 31) // 32, dtype=torch.int32, device="cuda")
    y = torch.empty(d, device="cuda")
    ws = ws_for(d, f, 1)
    cs.cs_exact_ffn(layer, x, pre, idx, cnt, y, ws, mask=mask)
    opre = oracle.preact(O, X[0])
    assert rel_err(pre.cpu().numpy(), opre) < 1e-5
    # neurons whose pre-activation is decided beyond fp32 rounding must agree
    wg = synth.storage_to_f64(H.w_gate, dt)[:, :d]
    eps = 64 * 2.0 ** -24 * (np.abs(wg) @ np.abs(X[0].astype(np.float64)) + np.abs(H.bias))
    n = int(cnt.item())
    gpre = pre.cpu().numpy()
    gidx = idx.cpu().numpy()[:n]
    # bit-exact: the oracle's exact mask {g > 0} taken on the GPU's own fp32
    # pre-activations is the GPU's index list and mask
    assert np.array_equal(gidx, oracle.select_positive(gpre))
    assert np.array_equal(mask.cpu().numpy().view(np.uint32), synth.bits_from_bool(gpre > 0))
    # and every neuron decided beyond fp32 rounding agrees with the fp64 oracle
    got = set(gidx.tolist())
    sure_in = set(np.flatnonzero(opre > eps).tolist())
    sure_out = set(np.flatnonzero(opre < -eps).tolist())
    assert sure_in <= got and not (got & sure_out)
    assert rel_err(y.cpu().numpy(), oracle.ffn(O, X[0], gidx)) < TOL
    assert rel_err(y.cpu().numpy(), oracle.dense_ffn(O, X[0])) < TOL


# -------------------------------------------------------------------- union

@pytest.mark.parametrize("f", [1, 31, 33, 2048, 32768, 40000, 262145])
@pytest.mark.parametrize("B", [1, 2, 7, 32])
def test_union_bit_exact(f, B):
    M = synth.union_masks(3, B, f, 0.1)
    if f % 32:  # bits beyond f must be ignored
        M[:, -1] |= np.uint32(~np.uint32((1 << (f % 32)) - 1))
    m = torch.from_numpy(M.view(np.int32)).cuda()
    words = (f + 31) // 32
    umask = torch.zeros(words, dtype=torch.int32, device="cuda")
    uidx = torch.zeros(f, dtype=torch.int32, device="cuda")
    ucnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs.cs_union_mask(m, f, umask, uidx, ucnt)
    wm, wi = oracle.union(M, f)
    n = int(ucnt.item())
    assert n == wi.size and np.array_equal(uidx.cpu().numpy()[:n], wi)
    assert np.array_equal(umask.cpu().numpy().view(np.uint32), wm)


@pytest.mark.parametrize("f", [4096, 40001])
def test_union_all_set(f):
    """Every bit set: each warp's 32 words hold 1,024 ids, the most its
    staging buffer takes; the ids run 0 .. f-1 across every block."""
    words = (f + 31) // 32
    M = np.full((3, words), 0xffffffff, dtype=np.uint32)
    m = torch.from_numpy(M.view(np.int32)).cuda()
    umask = torch.zeros(words, dtype=torch.int32, device="cuda")
    uidx = torch.full((f,), -1, dtype=torch.int32, device="cuda")
    ucnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs.cs_union_mask(m, f, umask, uidx, ucnt)
    assert int(ucnt.item()) == f
    assert np.array_equal(uidx.cpu().numpy(), np.arange(f, dtype=np.int32))


# -------------------------------------------------------------------- layout

@pytest.mark.parametrize("src_dt,dst_dt", [(synth.F32, synth.F16), (synth.F32, synth.BF16),
                                           (synth.F16, synth.F16), (synth.BF16, synth.F32)])
def test_pack_transpose(src_dt, dst_dt):
    rows, cols = 77, 130  # W_down [d, f]
    A = synth.normal_matrix(1, 1, rows, cols, 1.0, src_dt)
    src = upload(A, src_dt)
    ld_dst = 80 if dst_dt != synth.F32 else 80
    from _helpers import torch_dtype
    dst = torch.zeros((cols, ld_dst), dtype=torch_dtype(dst_dt), device="cuda")
    cs.cs_pack_transpose(src, dst)
    got = dst.float().cpu().numpy()[:, :rows].astype(np.float64)
    want = synth.storage_to_f64(A, src_dt).T
    want = synth.storage_to_f64(synth.to_storage(want.astype(np.float32), dst_dt), dst_dt)
    assert np.array_equal(got, want)
