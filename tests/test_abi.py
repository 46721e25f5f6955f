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
