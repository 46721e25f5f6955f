"""The C ABI library loads and exports every symbol include/cs.h declares;
host-side argument validation rejects bad calls without touching a GPU."""
import ctypes as C
import os
import re
import subprocess

import pytest

import contextual_sparsity_sparse_gb300 as cs
from contextual_sparsity_sparse_gb300 import build as cb

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include", "cs.h")


@pytest.fixture(scope="module")
def lib():
    cb.build()
    return cs.lib()


def declared():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(cs_[a-z_]+)\s*\(", text)))


def test_header_declares_the_binding_exports():
    assert declared() == sorted(cs.EXPORTS)


def test_library_exports_every_declared_symbol(lib):
    out = subprocess.run(["nm", "-D", "--defined-only", cb.LIB], capture_output=True, text=True,
                         check=True).stdout
    syms = {line.split()[-1] for line in out.splitlines() if line.strip()}
    for name in declared():
        assert name in syms, name
        assert hasattr(lib, name)


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.cs_version()
    assert lib.cs_status_string(0) == b"ok"
    assert lib.cs_status_string(5).startswith(b"workspace")


def test_validation_without_gpu(lib):
    # null layer / predictor / params: rejected on the host before any CUDA call
    assert lib.cs_sparse_ffn(None, None, 1, None, None, None, None, 0, None) == 1
    assert lib.cs_predict(None, None, 1, None, None, 0, None) == 1
    assert lib.cs_select(None, 1, 1, None, None, None, None, None, 0, None) == 1
    assert b"params" in lib.cs_last_error()
    L = cs._Layer(100, 10, cs.CS_F16, 100, 16, 0, 16, 0)  # 200-byte rows
    assert lib.cs_sparse_ffn(C.byref(L), None, 1, None, None, None, None, 0, None) == 1
    assert b"16 bytes" in lib.cs_last_error()
    P = cs._Pred(64, 8, 100, 7, 0, 0, 16, 16)  # bad dtype
    assert lib.cs_predict(C.byref(P), None, 1, None, None, 0, None) == 1
    assert lib.cs_union_mask(None, 1, 1, None, None, None, None, 0, None) == 1
    sel = cs.select_params(cs.CS_SEL_TOPK, 1)
    assert lib.cs_decode_stack(None, None, 0, None, 0.1, C.byref(sel), 0, None, None, None, 0, None, None) == 1
    assert lib.cs_pack_transpose(None, 0, 1, 1, 1, None, 0, 1, None) == 1


def test_decode_layer_validation_without_gpu(lib):
    # every case below is refused on the host before the first CUDA call
    sel = cs.select_params(cs.CS_SEL_TOPK, 1)
    good = cs._Layer(128, 64, cs.CS_F16, 128, 256, 0, 256, 0)
    pred = cs._Pred(128, 8, 64, cs.CS_F16, 0, 0, 256, 256)
    x = y = 1024  # never dereferenced on these paths

    def call(layer, p, params, idx=None, count=None, xx=x):
        ref = lambda v: C.byref(v) if v is not None else None
        return lib.cs_decode_layer(ref(layer), ref(p), xx, y, ref(params), 4096, 1 << 20, None, idx, count)

    assert call(None, pred, sel) == 1
    assert call(good, pred, sel, idx=4096, count=None) == 1
    assert b"together" in lib.cs_last_error()
    assert call(good, pred, sel, xx=1026) == 1          # x not 4-byte aligned
    assert call(good, None, sel) == 1
    assert b"predictor is required" in lib.cs_last_error()
    bad_mode = cs._Sel(7, 1, 0.0)
    assert call(good, pred, bad_mode) == 1
    assert b"selection mode" in lib.cs_last_error()
    bad_ld = cs._Layer(100, 64, cs.CS_F16, 100, 256, 0, 256, 0)   # 200-byte rows
    assert call(bad_ld, pred, sel) == 1
    assert b"layout" in lib.cs_last_error()
    short_pred = cs._Pred(128, 8, 32, cs.CS_F16, 0, 0, 256, 256)  # f differs from the layer's
    assert call(good, short_pred, sel) == 1
    assert b"predictor 0" in lib.cs_last_error()


def test_hot_order_matches_the_oracle(lib):
    """cs_hot_order runs on the host: most frequent first, ties by lower id,
    NaN last, exactly as the oracle's stable sort."""
    import numpy as np
    import oracle
    import synth
    rng = np.random.default_rng(3)
    for f in (0, 1, 37, 2048):
        freq = (rng.integers(0, 9, size=f) / 8).astype(np.float32)
        if f > 10:
            freq[::7] = np.nan
        got = cs.cs_hot_order(freq).numpy()
        assert np.array_equal(got, oracle.hot_order(freq)), f
    p = synth.firing_probs(0, 0, 20480, 0.10).astype(np.float32)
    assert np.array_equal(cs.cs_hot_order(p).numpy(), oracle.hot_order(p))


def test_select_hot_validation_without_gpu(lib):
    fake = 4096  # never dereferenced: the call is refused first
    for hot in (-32, 16, 33):
        sel = cs.select_params(cs.CS_SEL_TOPK, 5, hot=hot)
        assert lib.cs_select(fake, 1, 64, C.byref(sel), fake, fake, None, None, 0, None) == 1
        assert b"hot" in lib.cs_last_error()
    L = cs._Layer(128, 64, cs.CS_F16, 128, 256, 0, 256, 0)
    P = cs._Pred(128, 8, 64, cs.CS_F16, 0, 0, 256, 256)   # scores all 64 neurons
    sel = cs.select_params(cs.CS_SEL_TOPK, 5, hot=32)       # ... but only 32 are a tail
    assert lib.cs_decode_layer(C.byref(L), C.byref(P), 1024, 1024, C.byref(sel), 4096, 1 << 20, None,
                               None, None) == 1
    assert b"tail" in lib.cs_last_error()
    allhot = cs.select_params(cs.CS_SEL_TOPK, 5, hot=64)    # no tail left to predict
    P0 = cs._Pred(128, 8, 0, cs.CS_F16, 0, 0, 256, 256)
    assert lib.cs_decode_layer(C.byref(L), C.byref(P0), 1024, 1024, C.byref(allhot), 4096, 1 << 20, None,
                               None, None) == 1
    assert b"tail" in lib.cs_last_error()
    ex = cs.select_params(cs.CS_SEL_EXACT, hot=32)
    assert lib.cs_decode_layer(C.byref(L), None, 1024, 1024, C.byref(ex), 4096, 1 << 20, None,
                               None, None) == 1


def test_attention_and_fit_validation_without_gpu(lib):
    """Bad layouts are refused on the host, before any CUDA call."""
    fake = 4096
    A = cs._Attn(512, 8, 64, cs.CS_F16, fake, fake)
    # d_head not a power of two
    bad = cs._Attn(512, 8, 48, cs.CS_F16, fake, fake)
    assert lib.cs_sparse_attention(C.byref(bad), fake, fake, fake, fake, fake, 16, fake, fake, 1 << 20, None) == 1
    assert b"d_head" in lib.cs_last_error()
    # misaligned weights
    mis = cs._Attn(512, 8, 64, cs.CS_F16, fake + 2, fake)
    assert lib.cs_sparse_attention(C.byref(mis), fake, fake, fake, fake, fake, 16, fake, fake, 1 << 20, None) == 1
    # seq_len outside [1, 16384] (x and y distinct here)
    y = 2 * fake
    assert lib.cs_sparse_attention(C.byref(A), fake, fake, fake, fake, fake, 0, y, fake, 1 << 20, None) == 1
    assert lib.cs_sparse_attention(C.byref(A), fake, fake, fake, fake, fake, 20000, y, fake, 1 << 20, None) == 3
    # x aliasing y
    assert lib.cs_sparse_attention(C.byref(A), fake, fake, fake, fake, fake, 16, fake, fake, 1 << 20, None) == 1
    # the one-call attention step: heads without a count, an exact or hot
    # selection, a predictor that does not score one output per head
    P8 = cs._Pred(512, 16, 8, cs.CS_F16, 512, 16, fake, fake)
    top = cs.select_params(cs.CS_SEL_TOPK, 2)
    args = (fake, fake, 16, fake, 1 << 20, None)
    assert lib.cs_decode_attention(None, C.byref(P8), fake, y, C.byref(top), *args, None, None) == 1
    assert lib.cs_decode_attention(C.byref(A), C.byref(P8), fake, fake, C.byref(top), *args, None, None) == 1
    assert lib.cs_decode_attention(C.byref(A), C.byref(P8), fake, y, C.byref(top), *args, fake, None) == 1
    for bad_sel in (cs.select_params(cs.CS_SEL_EXACT), cs.select_params(cs.CS_SEL_TOPK, 2, hot=32)):
        assert lib.cs_decode_attention(C.byref(A), C.byref(P8), fake, y, C.byref(bad_sel), *args,
                                       None, None) == 1
    assert b"top-k or a threshold" in lib.cs_last_error()
    P9 = cs._Pred(512, 16, 9, cs.CS_F16, 512, 16, fake, fake)
    assert lib.cs_decode_attention(C.byref(A), C.byref(P9), fake, y, C.byref(top), *args, None, None) == 1
    assert b"heads" in lib.cs_last_error()
    assert lib.cs_decode_attention(C.byref(bad), C.byref(P8), fake, y, C.byref(top), *args, None, None) == 1
    assert b"d_head" in lib.cs_last_error()
    # the fit: negative ridge, a predictor for another layer
    L = cs._Layer(128, 64, cs.CS_F16, 128, 256, 0, 256, 0)
    P = cs._Pred(128, 8, 64, cs.CS_F16, 0, 0, 256, 256)
    assert lib.cs_fit_predictor(C.byref(L), C.byref(P), fake, 16, -1.0, fake, 1 << 30, None) == 1
    P2 = cs._Pred(128, 8, 32, cs.CS_F16, 0, 0, 256, 256)
    assert lib.cs_fit_predictor(C.byref(L), C.byref(P2), fake, 16, 1.0, fake, 1 << 30, None) == 1
    assert b"match the layer" in lib.cs_last_error()
    assert lib.cs_fit_scratch_size(128, 64, 8, 0) == 0
    assert lib.cs_fit_scratch_size(128, 64, 8, 16) > 16 * 64 * 4
