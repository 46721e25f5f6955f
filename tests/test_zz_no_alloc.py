"""The workspace-free FFN entry point (cs_sparse_ffn_noalloc).

It serves callers that cannot allocate device memory (a plugin inside a host
framework that owns every allocation, or a path where cudaMalloc may not be
issued).  It must compute what cs_sparse_ffn computes: checked here through
the C ABI against the workspace entry point and against the CPU oracle, on
two calls in a row (the shared scratch keeps the previous call's contents).
This file is collected last so a failure here does not hide the other tests.
"""
import ctypes as C

import numpy as np
import pytest

import oracle
import synth
from _helpers import TOL, HostLayer, rel_err

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402


def _noalloc(layer, x, B, idx, cnt, y):
    L = cs.lib()
    st = L.cs_sparse_ffn_noalloc(C.byref(layer.c), x.data_ptr(), B, idx.data_ptr(), cnt.data_ptr(),
                                 y.data_ptr(), None)
    assert st == 0, L.cs_last_error()


# (d, f, dtype, B, bitwise): below 4 tokens cs_sparse_ffn runs the same gather
# kernel, so the two agree bit for bit; at B = 4 with d a multiple of 64 it
# takes the tensor-core path and the two agree within the tolerance
CASES = [(5120, 4096, synth.F16, 1, True), (5120, 4096, synth.BF16, 2, True),
         (512, 2048, synth.F16, 4, False)]


@pytest.mark.parametrize("case", CASES, ids=[f"d{c[0]}-B{c[3]}" for c in CASES])
def test_noalloc_matches_workspace_entry_point_and_oracle(case):
    d, f, dt, B, bitwise = case
    cs.build.build()
    oracle.build()
    H = HostLayer(d, f, 0, dt, seed=21)
    layer, _ = H.device()
    O = H.oracle_layer()
    ws = cs.Workspace(d, f, 1, B)
    rng = np.random.default_rng(5)
    for call in range(2):
        X = synth.x_normal(40 + call, B, d)
        x = torch.from_numpy(X).cuda()
        sel = np.sort(rng.choice(f, size=f // 7 + 100 * call, replace=False)).astype(np.int32)
        idx = torch.from_numpy(sel).cuda()
        cnt = torch.tensor([sel.size], dtype=torch.int32, device="cuda")
        y_ws = torch.empty((B, d), device="cuda")
        y_na = torch.full((B, d), float("nan"), device="cuda")
        cs.cs_sparse_ffn(layer, x, idx, cnt, y_ws, ws)
        _noalloc(layer, x, B, idx, cnt, y_na)
        torch.cuda.synchronize()
        a, b = y_ws.cpu().numpy(), y_na.cpu().numpy()
        assert np.isfinite(b).all()
        for t in range(B):
            assert rel_err(b[t], a[t]) < TOL
            assert rel_err(b[t], oracle.ffn(O, X[t], sel)) < TOL, (call, t)
        if bitwise:
            # same kernel, same fixed-order reduction: the results agree bit for bit
            assert np.array_equal(a.view(np.uint32), b.view(np.uint32)), call


def test_noalloc_rejects_oversize_call():
    d, f = 8192, 64
    w = torch.zeros((f, d), dtype=torch.float16, device="cuda")
    layer = cs.FfnLayer(w, w)
    B = 8  # SMs * 8 * 8192 partial sums exceed the fixed scratch
    x = torch.zeros((B, d), device="cuda")
    y = torch.zeros((B, d), device="cuda")
    idx = torch.zeros(1, dtype=torch.int32, device="cuda")
    cnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    with pytest.raises(cs.CsError) as ei:
        cs.cs_sparse_ffn_noalloc(layer, x, idx, cnt, y)
    assert ei.value.status == 3
