"""GPU parity at the full shapes of the stack and batch workloads.

The stacks are checked on their first two layers (the oracle runs them in
seconds) through cs_decode_stack, in the configuration the benchmark times:
OPT-30B-shaped layers (d=7168, f=28672, r=512, fp16, ReLU) and
LLaMA-70B-shaped ReLUfied gated layers (d=8192, f=28672, r=1024, bf16).  The
batch union runs at the Falcon-40B shape (d=8192, f=32768, bf16)."""
import numpy as np
import pytest

import oracle
import synth
from _helpers import TOL, HostLayer, oracle_stack_k, rel_err, stack_inputs

pytestmark = pytest.mark.gpu

torch = pytest.importorskip("torch")
if not torch.cuda.is_available():
    pytest.skip("no CUDA device", allow_module_level=True)

import contextual_sparsity_sparse_gb300 as cs  # noqa: E402

STACKS = [
    ("opt30b", 7168, 28672, 512, synth.F16, False, 0.10),
    ("llama70b", 8192, 28672, 1024, synth.BF16, True, 0.15),
]


@pytest.fixture(scope="module", autouse=True)
def _built():
    cs.build.build()
    oracle.build()


@pytest.mark.parametrize("case", STACKS, ids=[c[0] for c in STACKS])
@pytest.mark.parametrize("mode", [cs.CS_STACK_SEQUENTIAL, cs.CS_STACK_LOOKAHEAD], ids=["seq", "lookahead"])
def test_stack_prefix_full_shape(case, mode):
    name, d, f, r, dt, glu, rho = case
    L = 2
    Hs, layers, preds = stack_inputs(L, d, f, r, dt, glu=glu, rho=rho)
    X = synth.x_normal(31, 1, d)[0]
    omode = oracle.LOOKAHEAD if mode == cs.CS_STACK_LOOKAHEAD else oracle.SEQUENTIAL
    k, xo, tr = oracle_stack_k(Hs, X, omode, synth.ceil_k(f, rho), 0.1)
    x = torch.from_numpy(X.copy()).cuda()
    ws = cs.Workspace(d, f, r)
    tc = torch.zeros(L, dtype=torch.int32, device="cuda")
    ti = torch.zeros((L, f), dtype=torch.int32, device="cuda")
    sm, sp = torch.cuda.Stream(), torch.cuda.Stream()
    torch.cuda.synchronize()
    cs.cs_decode_stack(layers, preds, x, 0.1, cs.select_params(cs.CS_SEL_TOPK, k), mode, ws,
                       s_main=sm, s_pred=sp, trace_count=tc, trace_idx=ti)
    torch.cuda.synchronize()
    TC, TI = tc.cpu().numpy(), ti.cpu().numpy()
    for l in range(L):
        assert TC[l] == tr["count"][l] == k
        assert np.array_equal(TI[l, :k], tr["idx"][l]), l
    assert rel_err(x.cpu().numpy(), xo) < TOL
    assert cs.cs_get_device_error(ws) == 0


@pytest.mark.parametrize("B", [1, 2, 4])
def test_union_batch_full_shape(B):
    d, f = 8192, 32768
    H = HostLayer(d, f, 0, synth.BF16, seed=2, rho=0.10)
    layer, _ = H.device()
    O = H.oracle_layer()
    M = synth.union_masks(2, B, f, 0.10)
    m = torch.from_numpy(M.view(np.int32)).cuda()
    umask = torch.zeros((f + 31) // 32, dtype=torch.int32, device="cuda")
    uidx = torch.zeros(f, dtype=torch.int32, device="cuda")
    ucnt = torch.zeros(1, dtype=torch.int32, device="cuda")
    cs.cs_union_mask(m, f, umask, uidx, ucnt)
    X = synth.x_normal(3, B, d)
    x = torch.from_numpy(X).cuda()
    y = torch.empty((B, d), device="cuda")
    ws = cs.Workspace(d, f, 1, B)
    cs.cs_sparse_ffn(layer, x, uidx, ucnt, y, ws)
    _, wi = oracle.union(M, f)
    n = int(ucnt.item())
    assert n == wi.size and np.array_equal(uidx.cpu().numpy()[:n], wi)
    Y = y.cpu().numpy()
    for b in range(B):
        assert rel_err(Y[b], oracle.ffn(O, X[b], wi)) < TOL, b
    assert cs.cs_get_device_error(ws) == 0
