"""GPU parity of the tensor-core (tcgen05) batched path against the oracle.

cs_sparse_ffn takes this path for B >= 4 tokens sharing one union list when
the weights are fp16 / bf16 and d is a multiple of 64 (below that, or for fp32
weights, the CUDA-core gather kernel serves the batch).  Every token's y must
match the oracle's fp64 sparse FFN over the union within the 2e-3 bound.
"""
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


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


def run_union(H, B, seed, rho=0.10, idx=None):
    """Union of B synthetic masks (or a given list), then the batched FFN."""
    d, f = H.d, H.f
    layer, _ = H.device()
    if idx is None:
        M = synth.union_masks(seed, B, f, rho)
        m = torch.from_numpy(M.view(np.int32)).cuda()
        umask = torch.zeros((f + 31) // 32, dtype=torch.int32, device="cuda")
        uidx = torch.zeros(f, dtype=torch.int32, device="cuda")
        ucnt = torch.zeros(1, dtype=torch.int32, device="cuda")
        cs.cs_union_mask(m, f, umask, uidx, ucnt)
        _, wi = oracle.union(M, f)
    else:
        wi = np.asarray(idx, np.int32)
        uidx = torch.zeros(max(f, 1), dtype=torch.int32, device="cuda")
        if wi.size:
            uidx[:wi.size] = torch.from_numpy(wi).cuda()
        ucnt = torch.tensor([wi.size], dtype=torch.int32, device="cuda")
    X = synth.x_normal(seed + 100, B, d)
    x = torch.from_numpy(X).cuda()
    y = torch.full((B, d), float("nan"), device="cuda")
    ws = cs.Workspace(d, f, 1, B)
    cs.cs_sparse_ffn(layer, x, uidx, ucnt, y, ws)
    torch.cuda.synchronize()
    assert cs.cs_get_device_error(ws) == 0
    n = int(ucnt.item())
    assert n == wi.size and np.array_equal(uidx.cpu().numpy()[:n], wi)
    return X, y.cpu().numpy(), wi


@pytest.mark.parametrize("dt", [synth.F16, synth.BF16], ids=["f16", "bf16"])
@pytest.mark.parametrize("glu", [False, True], ids=["relu", "glu"])
@pytest.mark.parametrize("B", [4, 5, 8, 16, 32])
def test_tc_batch_parity(dt, glu, B):
    H = HostLayer(1024, 4096, 0, dt, glu=glu, seed=5, rho=0.10)
    X, Y, wi = run_union(H, B, seed=40 + B)
    O = H.oracle_layer()
    assert wi.size % 128 != 0  # a ragged last tile
    for b in range(B):
        assert rel_err(Y[b], oracle.ffn(O, X[b], wi)) < TOL, b


@pytest.mark.parametrize("case", ["empty", "one", "dense", "d960"])
def test_tc_edges(case):
    if case == "d960":
        # d a multiple of 64 but not of 128: the last output tile is half empty
        H = HostLayer(960, 2048, 0, synth.BF16, glu=True, seed=6)
        X, Y, wi = run_union(H, 6, seed=7)
    else:
        H = HostLayer(512, 2048, 0, synth.F16, seed=6)
        idx = {"empty": [], "one": [1234], "dense": list(range(2048))}[case]
        X, Y, wi = run_union(H, 4, seed=8, idx=idx)
    O = H.oracle_layer()
    for b in range(Y.shape[0]):
        want = oracle.ffn(O, X[b], wi)
        if wi.size == 0:
            assert np.all(Y[b] == 0.0)
        else:
            assert rel_err(Y[b], want) < TOL, (case, b)


@pytest.mark.parametrize("B", [8, 32])
def test_tc_full_shape(B):
    """Falcon-40B-shaped union (d=8192, f=32768, bf16); tokens 0 and B-1 checked."""
    H = HostLayer(8192, 32768, 0, synth.BF16, seed=2, rho=0.10)
    X, Y, wi = run_union(H, B, seed=2)
    O = H.oracle_layer()
    for b in (0, B - 1):
        assert rel_err(Y[b], oracle.ffn(O, X[b], wi)) < TOL, b
