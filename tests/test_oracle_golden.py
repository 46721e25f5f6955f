"""Pins the CPU oracle to hand-worked examples (tests/golden/*.json).

Each fixture states its source passage.  All numbers are small binary
fractions, so the oracle must reproduce them exactly, in every storage dtype
that represents them exactly (fp32, fp16, bf16).
"""
import json
import os

import numpy as np
import pytest

import synth

GOLD = os.path.join(os.path.dirname(__file__), "golden")


def load(name):
    with open(os.path.join(GOLD, name)) as fh:
        return json.load(fh)


def store(a, dtype):
    return synth.to_storage(np.asarray(a, dtype=np.float32), dtype)


DTYPES = [synth.F32, synth.F16, synth.BF16]


def tiny_layer(orc, g, dtype, glu):
    return orc.Layer(g["d"], g["f"], dtype, store(g["w_gate"], dtype), store(g["w_down_t"], dtype),
                     w_up=store(g["w_up"], dtype) if glu else None, bias=g["bias"])


@pytest.mark.parametrize("dtype", DTYPES)
def test_ffn_relu_tiny(orc, dtype):
    g = load("ffn_tiny.json")
    L = tiny_layer(orc, g, dtype, glu=False)
    x = np.array(g["x"], np.float64)
    assert np.array_equal(orc.preact(L, x), np.array(g["preact"], np.float64))
    assert np.array_equal(orc.dense_ffn(L, x), np.array(g["relu"]["dense"], np.float64))
    for case in g["relu"]["subsets"]:
        y = orc.ffn(L, x, np.array(case["idx"], np.int32))
        assert np.array_equal(y, np.array(case["y"], np.float64)), case
    exact = orc.select_positive(orc.preact(L, x).astype(np.float32))
    assert exact.tolist() == g["relu"]["exact_idx"]
    assert np.array_equal(orc.ffn(L, x, exact), orc.dense_ffn(L, x))


@pytest.mark.parametrize("dtype", DTYPES)
def test_ffn_glu_tiny(orc, dtype):
    g = load("ffn_tiny.json")
    L = tiny_layer(orc, g, dtype, glu=True)
    x = np.array(g["x"], np.float64)
    assert np.array_equal(orc.dense_ffn(L, x), np.array(g["glu"]["dense"], np.float64))
    for case in g["glu"]["subsets"]:
        y = orc.ffn(L, x, np.array(case["idx"], np.int32))
        assert np.array_equal(y, np.array(case["y"], np.float64)), case


def test_ffn_rejects_bad_index(orc):
    g = load("ffn_tiny.json")
    L = tiny_layer(orc, g, synth.F32, glu=False)
    with pytest.raises(ValueError):
        orc.ffn(L, np.array(g["x"], np.float64), np.array([0, 4], np.int32))


@pytest.mark.parametrize("dtype", DTYPES)
def test_predictor_tiny(orc, dtype):
    g = load("predictor_tiny.json")
    P = orc.Predictor(g["d"], g["r"], g["f"], dtype, store(g["p_down"], dtype), store(g["p_up"], dtype))
    h, s = orc.predict(P, np.array(g["x"], np.float64))
    assert np.array_equal(h, np.array(g["h"], np.float64))
    assert np.array_equal(s, np.array(g["scores"], np.float64))
    s32 = s.astype(np.float32)
    for k, want in g["topk"].items():
        assert orc.select_topk(s32, int(k)).tolist() == want, k
    for tau, want in g["threshold"].items():
        assert orc.select_threshold(s32, float(tau)).tolist() == want, tau


def test_select_specials(orc):
    g = load("select_specials.json")
    s = np.array([float(v) for v in g["scores"]], np.float32)
    for k, want in g["topk"].items():
        assert orc.select_topk(s, int(k)).tolist() == want, k
    for tau, want in g["threshold"].items():
        assert orc.select_threshold(s, float(tau)).tolist() == want, tau
    assert orc.select_positive(s).tolist() == g["positive"]
    # the rank order itself: top-(m+1) minus top-m is the (m+1)-th ranked id
    prev = set()
    for m, j in enumerate(g["rank_order"]):
        cur = set(orc.select_topk(s, m + 1).tolist())
        assert cur - prev == {j}
        prev = cur


def test_recall_precision_tiny(orc):
    g = load("sets_tiny.json")["recall_precision"]
    r, p = orc.recall_precision(np.array(g["pred"]), np.array(g["exact"]), g["f"])
    assert r == g["recall"]
    assert p == g["precision_num"] / g["precision_den"]


def test_union_tiny(orc):
    g = load("sets_tiny.json")["union"]
    f = g["f"]
    masks = np.stack([synth.bits_from_bool(np.isin(np.arange(f), s)) for s in g["sets"]])
    umask, uidx = orc.union(masks, f)
    assert uidx.tolist() == g["union"]
    assert umask.tolist() == g["words"]


@pytest.mark.parametrize("dtype", DTYPES)
def test_stack_tiny(orc, dtype):
    g = load("stack_tiny.json")
    f = load("ffn_tiny.json")
    layers = [tiny_layer(orc, f, dtype, glu=False) for _ in range(2)]
    preds = [orc.Predictor(3, 3, 4, dtype, store(g[p]["p_down"], dtype), store(g[p]["p_up"], dtype))
             for p in ("pred0", "pred1")]
    x0 = np.array(g["x0"], np.float64)
    c = g["resid_scale"]
    for name, mode, sel in (("exact", orc.SEQUENTIAL, orc.SEL_EXACT),
                            ("sequential", orc.SEQUENTIAL, orc.SEL_TOPK),
                            ("lookahead", orc.LOOKAHEAD, orc.SEL_TOPK)):
        want = g[name]
        x1, tr1 = orc.stack(layers[:1], preds[:1], x0, mode=mode, sel_mode=sel, k=g["k"],
                            resid_scale=c, trace=True)
        x2, tr2 = orc.stack(layers, preds, x0, mode=mode, sel_mode=sel, k=g["k"],
                            resid_scale=c, trace=True)
        assert np.array_equal(x1, np.array(want["x1"], np.float64)), name
        assert np.array_equal(x2, np.array(want["x2"], np.float64)), name
        assert [i.tolist() for i in tr2["idx"]] == want["idx"], name
