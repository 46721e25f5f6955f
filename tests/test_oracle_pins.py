"""Pins the CPU oracle to closed forms, brute force and exact invariants.

Nothing here re-derives the oracle's own loops: each check is a property
fixed by the mathematics of the method (which neurons a permutation routes
where, the identity predictor, ReLU zeros), a brute-force enumeration on tiny
inputs, or a library routine on a special case.
"""
import math

import numpy as np
import pytest
import torch

import synth

DTYPES = [synth.F32, synth.F16, synth.BF16]


# ------------------------------------------------------------------ decoders

def test_f16_decoder_all_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = orc.decode(bits.view(np.float16), synth.F16)
    want = bits.view(np.float16).astype(np.float64)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


def test_bf16_decoder_all_patterns(orc):
    bits = np.arange(1 << 16, dtype=np.uint16)
    got = orc.decode(bits, synth.BF16)
    want = torch.from_numpy(bits.astype(np.int16)).view(torch.bfloat16).to(torch.float64).numpy()
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all()


# ------------------------------------------------------- permutation closed form

def perm_rows(n_rows, n_cols, cols):
    m = np.zeros((n_rows, n_cols), np.float32)
    m[np.arange(n_rows), cols] = 1.0
    return m


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("glu", [False, True])
def test_ffn_permutation_closed_form(orc, dtype, glu):
    """Gate row j picks x[pi(j)], up row j picks x[rho(j)], down row j (column
    j of W_down) writes to output sigma(j): y[sigma(j)] = relu(x[pi(j)] + b_j)
    * x[rho(j)] for each selected j, and 0 elsewhere.  A transposed operand, a
    wrong row or a dropped bias moves or changes a value."""
    rng = np.random.default_rng(3)
    d = f = 97
    pi, rho, sigma = rng.permutation(d), rng.permutation(d), rng.permutation(d)
    x = np.round(rng.standard_normal(d) * 8) / 8          # exact in every dtype
    b = (np.round(rng.standard_normal(f) * 4) / 4).astype(np.float32)
    L = orc.Layer(d, f, dtype, synth.to_storage(perm_rows(f, d, pi), dtype),
                  synth.to_storage(perm_rows(f, d, sigma), dtype),
                  w_up=synth.to_storage(perm_rows(f, d, rho), dtype) if glu else None, bias=b)
    sel = np.sort(rng.choice(f, size=40, replace=False)).astype(np.int32)
    y = orc.ffn(L, x, sel)
    want = np.zeros(d)
    for j in sel:
        a = max(0.0, x[pi[j]] + float(b[j]))
        want[sigma[j]] = a * (x[rho[j]] if glu else 1.0)
    assert np.array_equal(y, want)


# ------------------------------------------------------------ ReLU invariants

def random_layer(orc, d, f, dtype, glu, seed=0, rho=0.2, ld=None):
    ld = ld or d
    def mat(which):
        m = synth.normal_matrix(seed, synth.tensor_id(0, which), f, d, 1 / math.sqrt(d), dtype)
        if ld != d:
            pad = np.zeros((f, ld), m.dtype)
            pad[:, :d] = m
            m = pad
        return m
    return orc.Layer(d, f, dtype, mat(synth.W_GATE), mat(synth.W_DOWN_T),
                     w_up=mat(synth.W_UP) if glu else None,
                     bias=synth.zipf_bias(seed, 0, f, rho), ld=ld)


@pytest.mark.parametrize("dtype", DTYPES)
@pytest.mark.parametrize("glu", [False, True])
def test_exact_mask_and_all_true_reproduce_dense(orc, dtype, glu):
    """With ReLU, neurons whose pre-activation is <= 0 contribute exact zeros,
    so the exact-mask sparse FFN equals the dense FFN bit for bit, and so does
    the all-neuron list (k = f)."""
    d, f = 200, 333
    L = random_layer(orc, d, f, dtype, glu, ld=208)
    x = synth.x_normal(1, 1, d)[0].astype(np.float64)
    dense = orc.dense_ffn(L, x)
    exact = orc.select_positive(orc.preact(L, x).astype(np.float32))
    assert 0 < exact.size < f
    assert np.array_equal(orc.ffn(L, x, exact), dense)
    assert np.array_equal(orc.ffn(L, x, np.arange(f, dtype=np.int32)), dense)
    topf = orc.select_topk(orc.preact(L, x).astype(np.float32), f)
    assert np.array_equal(orc.ffn(L, x, topf), dense)
    # dropping one active neuron changes the result
    assert not np.array_equal(orc.ffn(L, x, exact[1:]), dense)


def test_dense_matches_numpy_matmul(orc):
    """Special case that reduces to a library routine: the dense gate-only FFN
    is W_down @ relu(W_gate @ x + b)."""
    d, f = 64, 150
    L = random_layer(orc, d, f, synth.F32, glu=False)
    x = synth.x_normal(2, 1, d)[0].astype(np.float64)
    wg = L.w_gate.astype(np.float64)
    wd = L.w_down_t.astype(np.float64)
    want = wd.T @ np.maximum(wg @ x + L.bias, 0.0)
    np.testing.assert_allclose(orc.dense_ffn(L, x), want, rtol=1e-12, atol=1e-12)


# ---------------------------------------------------------------- predictor

@pytest.mark.parametrize("dtype", DTYPES)
def test_identity_predictor_scores_are_gate_products(orc, dtype):
    """r = 2d, P_down = [I; -I], P_up = [W, -W]: relu(t) - relu(-t) = t, so the
    scores are W x exactly (up to summation order), and thresholding them at 0
    reproduces the exact mask of a bias-free layer: recall = precision = 1."""
    d, f = 48, 120
    W = synth.normal_matrix(5, 0, f, d, 1 / math.sqrt(d), dtype)
    Wf = synth.storage_to_f64(W, dtype)
    eye = np.eye(d, dtype=np.float32)
    p_down = synth.to_storage(np.concatenate([eye, -eye]), dtype)
    p_up = np.concatenate([W, (W ^ np.uint16(0x8000)) if dtype == synth.BF16 else -W], axis=1)
    P = orc.Predictor(d, 2 * d, f, dtype, p_down, p_up)
    x = synth.x_normal(6, 1, d)[0].astype(np.float64)
    h, s = orc.predict(P, x)
    assert np.array_equal(h, np.concatenate([np.maximum(x, 0), np.maximum(-x, 0)]))
    np.testing.assert_allclose(s, Wf @ x, rtol=0, atol=1e-12)
    L = orc.Layer(d, f, dtype, W, W)
    exact = orc.select_positive(orc.preact(L, x).astype(np.float32))
    pred = orc.select_threshold(s.astype(np.float32), 0.0)
    assert orc.recall_precision(pred, exact, f) == (1.0, 1.0)


def test_predictor_matches_numpy(orc):
    d, r, f = 80, 24, 300
    pd = synth.normal_matrix(0, synth.P_DOWN, r, d, 1 / math.sqrt(d), synth.F16)
    pu = synth.normal_matrix(0, synth.P_UP, f, r, 1 / math.sqrt(d), synth.F16)
    P = orc.Predictor(d, r, f, synth.F16, pd, pu)
    x = synth.x_normal(0, 1, d)[0].astype(np.float64)
    h, s = orc.predict(P, x)
    hw = np.maximum(pd.astype(np.float64) @ x, 0)
    np.testing.assert_allclose(h, hw, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(s, pu.astype(np.float64) @ hw, rtol=1e-12, atol=1e-13)


def test_random_predictor_recall_is_k_over_f(orc):
    """A predictor unrelated to the layer picks neurons at random, so its
    expected recall against the exact mask is k/f (binomial spread)."""
    d, r, f = 128, 32, 2048
    L = random_layer(orc, d, f, synth.F32, glu=False, rho=0.1)
    pd = synth.normal_matrix(9, synth.P_DOWN, r, d, 1 / math.sqrt(d), synth.F32)
    pu = synth.normal_matrix(9, synth.P_UP, f, r, 1 / math.sqrt(d), synth.F32)
    P = orc.Predictor(d, r, f, synth.F32, pd, pu)
    k = 512
    hits = exact_total = 0
    for t in range(24):
        x = synth.x_normal(100 + t, 1, d)[0].astype(np.float64)
        _, s = orc.predict(P, x)
        pred = orc.select_topk(s.astype(np.float32), k)
        exact = orc.select_positive(orc.preact(L, x).astype(np.float32))
        hits += np.intersect1d(pred, exact).size
        exact_total += exact.size
    rec = hits / exact_total
    sd = math.sqrt((k / f) * (1 - k / f) / exact_total)
    assert abs(rec - k / f) < 6 * sd + 0.03


# ---------------------------------------------------------------- selection

def brute_topk(s, k):
    def key(j):
        v = s[j]
        return (0 if math.isnan(v) else 1, 0.0 if math.isnan(v) else float(v) + 0.0, -j)
    order = sorted(range(len(s)), key=key, reverse=True)
    return sorted(order[:max(0, min(k, len(s)))])


@pytest.mark.parametrize("seed", range(40))
def test_topk_brute_force(orc, seed):
    rng = np.random.default_rng(seed)
    f = int(rng.integers(1, 65))
    s = synth.score_vector(seed, f, ties=int(rng.integers(0, f + 1)), specials=bool(seed % 2),
                           quantize=0.5 if seed % 3 == 0 else None)
    for k in sorted({0, 1, f // 3, f // 2, f - 1, f, f + 3}):
        assert orc.select_topk(s, k).tolist() == brute_topk(s, k), (f, k)


@pytest.mark.parametrize("seed", range(20))
def test_threshold_brute_force(orc, seed):
    rng = np.random.default_rng(seed)
    f = int(rng.integers(1, 200))
    s = synth.score_vector(seed, f, ties=5, specials=True, quantize=0.25)
    for tau in (-np.inf, -1.0, 0.0, -0.0, 0.25, 1.5, np.inf, np.nan):
        want = [j for j in range(f) if s[j] >= np.float32(tau)]
        assert orc.select_threshold(s, tau).tolist() == want
    assert orc.select_positive(s).tolist() == [j for j in range(f) if s[j] > 0]


def test_topk_dominance_large(orc):
    """Every chosen neuron outranks every unchosen one, |A| = min(k, f)."""
    f = 5000
    s = synth.score_vector(11, f, ties=800, specials=True, quantize=0.01)
    for k in (1, 77, 2500, 4999):
        A = orc.select_topk(s, k)
        assert A.size == k and np.all(np.diff(A) > 0)
        inA = np.zeros(f, bool)
        inA[A] = True
        key = np.where(np.isnan(s), -np.inf, s).astype(np.float64)
        nan = np.isnan(s)
        # lowest chosen vs highest unchosen under the ranking rule
        ch = [(not nan[j], key[j], -j) for j in A]
        un = [(not nan[j], key[j], -j) for j in np.flatnonzero(~inA)]
        assert min(ch) > max(un)


# ------------------------------------------------------------------- union

def test_union_matches_set_union(orc):
    rng = np.random.default_rng(4)
    for f in (1, 31, 32, 33, 1000):
        B = int(rng.integers(1, 9))
        sets = [set(rng.choice(f, size=int(rng.integers(0, f + 1)), replace=False).tolist())
                for _ in range(B)]
        masks = np.stack([synth.bits_from_bool(np.isin(np.arange(f), sorted(s))) for s in sets])
        umask, uidx = orc.union(masks, f)
        want = sorted(set().union(*sets))
        assert uidx.tolist() == want
        assert np.array_equal(synth.bool_from_bits(umask, f), np.isin(np.arange(f), want))


def test_union_density_closed_form(orc):
    """Expected union density of B tokens drawn Bernoulli(p_j) plus a uniform
    3% tail: mean_j 1 - ((1 - p_j) * 0.97)^B."""
    f = 32768
    p = synth.firing_probs(2, 0, f, 0.10)
    for B in (1, 4, 16):
        masks = synth.union_masks(2, B, f, 0.10)
        _, uidx = orc.union(masks, f)
        expect = float(np.mean(1 - ((1 - p) * 0.97) ** B))
        assert abs(uidx.size / f - expect) < 0.01, (B, uidx.size / f, expect)


# --------------------------------------------------------- generator profile

def test_zipf_layer_fires_at_target_rate(orc):
    """Bias b_j = PhiInv(p_j) with rows ~ N(0, 1/d) makes neuron j fire with
    probability ~p_j; the mean over neurons is the target share rho."""
    d, f, rho = 256, 2048, 0.10
    L = random_layer(orc, d, f, synth.F16, glu=False, rho=rho, seed=7)
    p = synth.firing_probs(7, 0, f, rho)
    T = 48
    fired = np.zeros(f)
    for t in range(T):
        x = synth.x_normal(500 + t, 1, d)[0].astype(np.float64)
        fired += orc.preact(L, x) > 0
    rate = fired.sum() / (T * f)
    assert abs(rate - rho) < 0.01
    hot, cold = p >= 0.5, p <= np.quantile(p, 0.2)
    assert abs(fired[hot].mean() / T - p[hot].mean()) < 0.05
    assert abs(fired[cold].mean() / T - p[cold].mean()) < 0.02


# -------------------------------------------------------------------- stack

def small_stack(orc, L_, d, f, r, dtype, glu=False, seed=0):
    layers, preds = [], []
    for l in range(L_):
        mk = lambda w, rows, cols: synth.normal_matrix(seed, synth.tensor_id(l, w), rows, cols,
                                                       1 / math.sqrt(d), dtype)
        layers.append(orc.Layer(d, f, dtype, mk(synth.W_GATE, f, d), mk(synth.W_DOWN_T, f, d),
                                w_up=mk(synth.W_UP, f, d) if glu else None,
                                bias=synth.zipf_bias(seed, l, f, 0.1)))
        preds.append(orc.Predictor(d, r, f, dtype, mk(synth.P_DOWN, r, d), mk(synth.P_UP, f, r)))
    return layers, preds


def test_lookahead_equals_sequential_without_residual_update(orc):
    """With c = 0 the stream does not move, x_l = x_{l-1}, so predicting layer
    l from layer l-1's input is the same prediction: identical output."""
    layers, preds = small_stack(orc, 4, 64, 256, 16, synth.F16)
    x = synth.x_normal(3, 1, 64)[0]
    a, ta = orc.stack(layers, preds, x, mode=orc.SEQUENTIAL, k=40, resid_scale=0.0, trace=True)
    b, tb = orc.stack(layers, preds, x, mode=orc.LOOKAHEAD, k=40, resid_scale=0.0, trace=True)
    assert np.array_equal(a, b)
    assert all(np.array_equal(i, j) for i, j in zip(ta["idx"], tb["idx"]))
    # a large residual step moves the stream enough to change some prediction
    s_, ts = orc.stack(layers, preds, x, mode=orc.SEQUENTIAL, k=40, resid_scale=4.0, trace=True)
    c, tc = orc.stack(layers, preds, x, mode=orc.LOOKAHEAD, k=40, resid_scale=4.0, trace=True)
    assert np.array_equal(ts["idx"][0], tc["idx"][0])
    assert not all(np.array_equal(i, j) for i, j in zip(ts["idx"], tc["idx"]))


def test_exact_stack_equals_dense_composition(orc):
    """With exact masks every layer equals its dense FFN, so the stack is the
    composition x <- x + c * W_down relu(W_gate x + b), here via numpy."""
    layers, preds = small_stack(orc, 3, 40, 100, 8, synth.F32)
    x = synth.x_normal(4, 1, 40)[0].astype(np.float64)
    got = orc.stack(layers, preds, x, sel_mode=orc.SEL_EXACT, resid_scale=0.25)
    want = x.copy()
    for L in layers:
        want = want + 0.25 * (L.w_down_t.astype(np.float64).T
                              @ np.maximum(L.w_gate.astype(np.float64) @ want + L.bias, 0))
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12)


# -------------------------------------------------------- hot-prefix layout

@pytest.mark.parametrize("seed", range(16))
def test_hot_select_brute_force(orc, seed):
    """Hot prefix: ids 0 .. H-1 always, then H + the tail's own selection,
    checked against the brute-force ranking above."""
    rng = np.random.default_rng(100 + seed)
    ft = int(rng.integers(0, 50))
    hot = [0, 1, 5, 32][seed % 4]
    s = synth.score_vector(seed, max(ft, 1), ties=int(rng.integers(0, ft + 1)), specials=bool(seed % 2),
                           quantize=0.5 if seed % 3 == 0 else None)[:ft]
    for k in sorted({0, 1, ft // 2, ft, ft + 2}):
        want = list(range(hot)) + [hot + j for j in brute_topk(s, k)]
        assert orc.select_hot(s, hot, orc.SEL_TOPK, k=k).tolist() == want, (ft, hot, k)
    for tau in (-np.inf, 0.0, 0.5, np.nan):
        want = list(range(hot)) + [hot + j for j in range(ft) if s[j] >= np.float32(tau)]
        assert orc.select_hot(s, hot, orc.SEL_THRESHOLD, tau=tau).tolist() == want


def test_hot_order_sorts_by_frequency_then_id(orc):
    rng = np.random.default_rng(7)
    freq = rng.integers(0, 6, size=300).astype(np.float64) / 5   # many equal frequencies
    o = orc.hot_order(freq)
    assert sorted(o.tolist()) == list(range(300))
    for a, b in zip(o[:-1], o[1:]):   # adjacent pairs: strictly hotter, or equal and lower id
        assert freq[a] > freq[b] or (freq[a] == freq[b] and a < b)
    # the synthetic Zipf profile: its hottest neurons are the low ranks
    p = synth.firing_probs(0, 0, 2048, 0.10)
    o = orc.hot_order(p)
    assert np.all(np.diff(p[o]) <= 0) and p[o[0]] == p.max()


@pytest.mark.parametrize("dtype", [synth.F32, synth.F16])
def test_hot_layout_leaves_the_ffn_unchanged(orc, dtype):
    """Reordering neurons (rows of W_gate, W_down^T and the bias together) and
    renaming the chosen set with them changes nothing but the summation
    order: dense and sparse FFN agree to fp64 rounding."""
    d, f = 24, 96
    sd = 1 / math.sqrt(d)
    wg = synth.normal_matrix_np(3, 1, f, d, sd, dtype)
    wd = synth.normal_matrix_np(3, 2, f, d, sd, dtype)
    b = synth.zipf_bias(3, 0, f, 0.1)
    x = synth.x_normal(5, 1, d)[0]
    perm = orc.hot_order(synth.firing_probs(3, 0, f, 0.1))
    L0 = orc.Layer(d, f, dtype, wg, wd, bias=b)
    L1 = orc.Layer(d, f, dtype, orc.permute_rows(wg, perm), orc.permute_rows(wd, perm),
                   bias=orc.permute_rows(b, perm))
    np.testing.assert_allclose(orc.dense_ffn(L1, x), orc.dense_ffn(L0, x), rtol=1e-12, atol=1e-13)
    inv = np.empty(f, np.int32)
    inv[perm] = np.arange(f, dtype=np.int32)
    A = np.array([3, 17, 40, 41, 77, 95], np.int32)
    np.testing.assert_allclose(orc.ffn(L1, x, np.sort(inv[A])), orc.ffn(L0, x, A), rtol=1e-12, atol=1e-13)


def small_hot_stack(orc, L, d, f, r, hot, dtype):
    sd = 1 / math.sqrt(d)
    layers, preds = [], []
    for l in range(L):
        mk = lambda w, rows, cols: synth.normal_matrix_np(0, synth.tensor_id(l, w), rows, cols, sd, dtype)
        layers.append(orc.Layer(d, f, dtype, mk(synth.W_GATE, f, d), mk(synth.W_DOWN_T, f, d),
                                bias=synth.zipf_bias(0, l, f, 0.1)))
        preds.append(orc.Predictor(d, r, f - hot, dtype, mk(synth.P_DOWN, r, d), mk(synth.P_UP, f - hot, r)))
    return layers, preds


def numpy_stack(layers, x, c, sets):
    x = x.astype(np.float64).copy()
    for L, A in zip(layers, sets):
        A = np.asarray(A, np.int64)
        wg, wd = L.w_gate.astype(np.float64)[A], L.w_down_t.astype(np.float64)[A]
        x = x + c * (wd.T @ np.maximum(wg @ x + L.bias[A], 0))
    return x


@pytest.mark.parametrize("mode", ["seq", "look"])
def test_hot_stack_extremes(orc, mode):
    """With no tail budget every layer takes exactly the prefix; with the whole
    tail it takes every neuron.  Both are plain numpy compositions."""
    Ls, d, f, r, hot = 3, 32, 128, 8, 32
    layers, preds = small_hot_stack(orc, Ls, d, f, r, hot, synth.F32)
    m = orc.SEQUENTIAL if mode == "seq" else orc.LOOKAHEAD
    x = synth.x_normal(9, 1, d)[0]
    got, tr = orc.stack(layers, preds, x, mode=m, k=0, hot=hot, resid_scale=0.3, trace=True)
    assert all(i.tolist() == list(range(hot)) for i in tr["idx"])
    np.testing.assert_allclose(got, numpy_stack(layers, x, 0.3, [range(hot)] * Ls), rtol=1e-12, atol=1e-12)
    got, tr = orc.stack(layers, preds, x, mode=m, k=f - hot, hot=hot, resid_scale=0.3, trace=True)
    assert all(i.tolist() == list(range(f)) for i in tr["idx"])
    np.testing.assert_allclose(got, numpy_stack(layers, x, 0.3, [range(f)] * Ls), rtol=1e-12, atol=1e-12)
    with pytest.raises(ValueError):   # a predictor must cover exactly the tail
        orc.stack(layers, preds, x, mode=m, k=4, hot=hot + 32)


# ------------------------------------------------------------- SiLU (next row 2)

def silu_pair_layer(orc, d, npairs, glu, dtype, seed=0):
    """Neurons in pairs whose contributions differ by the sign of silu(-g):
    gated (w, u, v) and (-w, -u, v), gate-only (w, v) and (-w, -v).  Since
    silu(g) - silu(-g) = g for every g, each pair adds exactly
    g * (u . x or 1) * v."""
    rng = np.random.default_rng(seed)
    W = (rng.standard_normal((npairs, d)) / math.sqrt(d)).astype(np.float32)
    U = (rng.standard_normal((npairs, d)) / math.sqrt(d)).astype(np.float32)
    V = rng.standard_normal((npairs, d)).astype(np.float32)
    wg = np.concatenate([W, -W]).astype(np.float32)
    wu = np.concatenate([U, -U]).astype(np.float32)
    wd = np.concatenate([V, V if glu else -V]).astype(np.float32)
    L = orc.Layer(d, 2 * npairs, synth.F32, wg, wd, w_up=wu if glu else None, act=orc.ACT_SILU)
    return L, W.astype(np.float64), U.astype(np.float64), V.astype(np.float64)


@pytest.mark.parametrize("glu", [False, True])
def test_silu_odd_part_closed_form(orc, glu):
    d, npairs = 48, 40
    L, W, U, V = silu_pair_layer(orc, d, npairs, glu, synth.F32)
    x = synth.x_normal(8, 1, d)[0].astype(np.float64) * 3.0   # g spans the curved region and beyond
    g = W @ x
    coef = g * (U @ x) if glu else g
    want = V.T @ coef
    got = orc.dense_ffn(L, x)
    np.testing.assert_allclose(got, want, rtol=1e-12, atol=1e-12 * np.abs(want).max())


def test_silu_limits_and_a_known_value(orc):
    """silu(g) -> g far above 0 and -> 0 far below it; silu(0) = 0; and
    silu(1) = e / (1 + e), the logistic function at 1 times 1."""
    d, f = 16, 3
    eye = np.zeros((f, d), np.float32)
    for j in range(f):
        eye[j, j] = 1.0
    down = np.eye(f, d, dtype=np.float32)
    x = np.zeros(d)
    for bias, want in ((np.array([40.0, 60.0, 35.5], np.float32), [40.0, 60.0, 35.5]),
                       (np.array([-40.0, -60.0, 0.0], np.float32), [0.0, 0.0, 0.0]),
                       (np.array([1.0, 0.0, -1.0], np.float32),
                        [math.e / (1 + math.e), 0.0, -1.0 / (1 + math.e)])):
        L = orc.Layer(d, f, synth.F32, eye, down, bias=bias, act=orc.ACT_SILU)
        y = orc.dense_ffn(L, x)[:f]
        np.testing.assert_allclose(y, want, rtol=1e-14, atol=1e-15)
        # ReLU is the SiLU limit on the positive side
        if bias[0] > 0 and bias[2] > 0:
            Lr = orc.Layer(d, f, synth.F32, eye, down, bias=bias)
            np.testing.assert_allclose(orc.dense_ffn(Lr, x)[:f], y, rtol=1e-14)


@pytest.mark.parametrize("seed", range(8))
def test_magnitude_selection_brute_force(orc, seed):
    s = synth.score_vector(seed, 300, ties=20, specials=True, quantize=0.25 if seed % 2 else None) * 2
    sig = lambda v: 1.0 / (1.0 + np.exp(-v))
    with np.errstate(over="ignore", invalid="ignore"):
        silu = np.where(np.isnan(s), np.nan, s.astype(np.float64) * sig(s.astype(np.float64)))
    silu = np.where(np.isinf(s) & (s < 0), 0.0, silu)
    relu = np.maximum(s.astype(np.float64), 0)
    for tau in (0.0, 0.05, 0.2, 0.27, 1.0):
        assert orc.select_magnitude(s, orc.ACT_SILU, tau).tolist() == \
            [j for j in range(s.size) if abs(silu[j]) > tau], tau
        assert orc.select_magnitude(s, orc.ACT_RELU, tau).tolist() == \
            [j for j in range(s.size) if relu[j] > tau], tau
    # relu at tau = 0 is the exact mask
    assert orc.select_magnitude(s, orc.ACT_RELU, 0.0).tolist() == orc.select_positive(s).tolist()


# ------------------------------------------------ fitted predictor (next row 3)

def identity_predictor(orc, d, f, dtype):
    """r = 2d, P_down = [I; -I]: h(x) = [relu(x); relu(-x)], and x = h_top - h_bottom."""
    eye = np.concatenate([np.eye(d), -np.eye(d)]).astype(np.float32)
    pd = synth.to_storage(eye, dtype)
    return orc.Predictor(d, 2 * d, f, dtype, pd, np.zeros((f, 2 * d), pd.dtype))


@pytest.mark.parametrize("dtype", [synth.F32, synth.F16])
def test_fit_recovers_an_exactly_representable_layer(orc, dtype):
    """With P_down = [I; -I] and no bias, W x = [W, -W] h(x) exactly, so the
    least-squares fit (lam -> 0) must return [W, -W]."""
    d, f = 16, 40
    W = synth.normal_matrix(6, 0, f, d, 1 / math.sqrt(d), dtype)
    L = orc.Layer(d, f, dtype, W, W)
    P = identity_predictor(orc, d, f, dtype)
    X = synth.x_normal(7, 300, d)
    got = orc.fit_predictor(L, P, X, 1e-10)
    w = synth.storage_to_f64(W, dtype)
    np.testing.assert_allclose(got, np.concatenate([w, -w], axis=1), rtol=0, atol=1e-7)


def test_fit_heavy_ridge_limit_and_linearity(orc):
    """(H^T H + lam I)^-1 -> I / lam as lam grows, so lam * P_up -> G^T H; and
    doubling the layer (weights and bias) doubles the fit."""
    d, f, r = 24, 60, 10
    sd = 1 / math.sqrt(d)
    W = synth.normal_matrix(8, 0, f, d, sd, synth.F32)
    b = synth.zipf_bias(8, 0, f, 0.1)
    pd = synth.normal_matrix(8, 1, r, d, sd, synth.F32)
    L = orc.Layer(d, f, synth.F32, W, W, bias=b)
    P = orc.Predictor(d, r, f, synth.F32, pd, np.zeros((f, r), np.float32))
    X = synth.x_normal(9, 50, d).astype(np.float64)
    H = np.maximum(X @ pd.astype(np.float64).T, 0)
    G = X @ W.astype(np.float64).T + b
    lam = 1e12
    np.testing.assert_allclose(lam * orc.fit_predictor(L, P, X, lam), G.T @ H, rtol=1e-6)
    L2 = orc.Layer(d, f, synth.F32, 2 * W, W, bias=2 * b)
    np.testing.assert_allclose(orc.fit_predictor(L2, P, X, 0.5), 2 * orc.fit_predictor(L, P, X, 0.5),
                               rtol=1e-12, atol=1e-12)


# ------------------------------------------------ head-sparse attention (next row 4)

def attn_inputs(orc, d, H, dh, S, dtype, seed):
    sd = 1 / math.sqrt(d)
    wq = synth.normal_matrix(seed, 0, H * dh, d, sd, dtype)
    wo = synth.normal_matrix(seed, 1, H * dh, d, 1 / math.sqrt(dh), dtype)
    kc = synth.normal_matrix(seed, 2, H * S, dh, 1.0, dtype).reshape(H, S, dh)
    vc = synth.normal_matrix(seed, 3, H * S, dh, 1.0, dtype).reshape(H, S, dh)
    return orc.AttnLayer(d, H, dh, dtype, wq, wo), wq, wo, kc, vc


def test_attention_one_key_returns_its_value(orc):
    """With one cached position the softmax weight is 1 whatever q is:
    y = sum_h W_o[:, h] v_h0, the same for any W_q."""
    d, H, dh = 32, 4, 8
    A, wq, wo, kc, vc = attn_inputs(orc, d, H, dh, 1, synth.F32, 1)
    A0 = orc.AttnLayer(d, H, dh, synth.F32, np.zeros_like(wq), wo)
    x = synth.x_normal(2, 1, d)[0]
    heads = [0, 2, 3]
    want = sum(wo[h * dh:(h + 1) * dh].astype(np.float64).T @ vc[h, 0].astype(np.float64) for h in heads)
    np.testing.assert_allclose(orc.attention(A, x, heads, kc, vc), want, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(orc.attention(A0, x, heads, kc, vc), want, rtol=1e-12, atol=1e-12)


def test_attention_equal_keys_average_the_values(orc):
    d, H, dh, S = 32, 3, 8, 9
    A, wq, wo, kc, vc = attn_inputs(orc, d, H, dh, S, synth.F32, 3)
    kc[:] = kc[:, :1, :]   # every position of a head has the same key
    x = synth.x_normal(4, 1, d)[0]
    want = sum(wo[h * dh:(h + 1) * dh].astype(np.float64).T @ vc[h].astype(np.float64).mean(axis=0)
               for h in range(H))
    np.testing.assert_allclose(orc.attention(A, x, range(H), kc, vc), want, rtol=1e-12, atol=1e-12)


def test_attention_two_keys_logistic_weight(orc):
    """q = (c, 0, ..) and keys (a, 0, ..), 0: the weights are the logistic
    function of c a / sqrt(d_head) and its complement."""
    d, H, dh = 16, 2, 8
    wq = np.zeros((H * dh, d), np.float32)
    wq[1 * dh + 0, 5] = 1.0                 # head 1: q_0 = x_5
    wo = np.zeros((H * dh, d), np.float32)
    wo[1 * dh:2 * dh, :dh] = np.eye(dh)     # head 1: y[:dh] = o
    kc = np.zeros((H, 2, dh), np.float32)
    kc[1, 0, 0] = 1.5
    vc = np.zeros((H, 2, dh), np.float32)
    vc[1, 0, :] = 1.0
    vc[1, 1, :] = -3.0
    A = orc.AttnLayer(d, H, dh, synth.F32, wq, wo)
    x = np.zeros(d)
    x[5] = 2.0
    p = 1.0 / (1.0 + math.exp(-2.0 * 1.5 / math.sqrt(dh)))
    y = orc.attention(A, x, [1], kc, vc)
    np.testing.assert_allclose(y[:dh], p * 1.0 + (1 - p) * -3.0, rtol=1e-14)
    assert np.all(y[dh:] == 0)


def test_attention_is_additive_over_heads_and_blind_to_cache_order(orc):
    d, H, dh, S = 40, 6, 8, 13
    A, wq, wo, kc, vc = attn_inputs(orc, d, H, dh, S, synth.F16, 5)
    x = synth.x_normal(6, 1, d)[0]
    heads = [1, 2, 4, 5]
    both = orc.attention(A, x, heads, kc, vc)
    np.testing.assert_allclose(both, sum(orc.attention(A, x, [h], kc, vc) for h in heads), rtol=1e-12,
                               atol=1e-12)
    perm = np.random.default_rng(7).permutation(S)
    np.testing.assert_allclose(orc.attention(A, x, heads, kc[:, perm], vc[:, perm]), both, rtol=1e-12,
                               atol=1e-12)
    assert np.all(orc.attention(A, x, [], kc, vc) == 0)
