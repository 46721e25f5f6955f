"""End-to-end drift of the full-size layer stacks against the CPU oracle.

"Contextual Sparsity and Activation Predictors", section "The predictor and
its budget" (the residual stream x_{l+1} = x_l + c FFN_l(x_l, A_l), with A_l
predicted from x_l, or from x_{l-1} with look-ahead) and section "When it
breaks" (look-ahead is weakest in the early layers).

The GPU runs cs_decode_stack over all L layers of the OPT-30B-shaped (48) or
LLaMA-70B-shaped (80) stack; the oracle runs its own fp64 stack from the same
x_0: per layer its own predictor scores (rounded to fp32, as the oracle always
decides), its own top-k, and the sparse FFN over the chosen rows.  Nothing is
teacher-forced, so a near-tie that falls the other way in one layer changes
that layer's set and everything after it: the report shows how far the two
stacks drift apart, it is not a pass / fail test.  The oracle needs only the
predictor and the chosen rows of each layer, which the seeded generator
produces on demand, so the 112 GB stack never has to sit in host memory.

    python tests/drift_report.py --workload llama70b --mode lookahead --tokens 2

prints one JSON line: per token the relative error max|x_L - o_L| / max|o_L|,
the layers whose selections match exactly, and the mean Jaccard overlap of the
selections.
"""
from __future__ import annotations

import argparse
import json
import math
import os
import sys
import time

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import oracle  # noqa: E402
import synth  # noqa: E402

SHAPES = {
    # d, f, r, dtype, gated, rho (profile and top-k share), layers
    "opt30b": (7168, 28672, 512, synth.F16, False, 0.10, 48),
    "llama70b": (8192, 28672, 1024, synth.BF16, True, 0.15, 80),
}


def oracle_layer_rows(l, d, f, dt, glu, rho, rows):
    """Layer l restricted to the given rows (ascending ids): an oracle Layer of
    len(rows) neurons whose row m is neuron rows[m]."""
    sd = 1 / math.sqrt(d)
    mk = lambda which: synth.normal_matrix(0, synth.tensor_id(l, which), f, d, sd, dt, row_ids=rows)
    bias = synth.zipf_bias(0, l, f, rho)[rows]
    return oracle.Layer(d, len(rows), dt, mk(synth.W_GATE), mk(synth.W_DOWN_T),
                        w_up=mk(synth.W_UP) if glu else None, bias=bias)


def oracle_predictor(l, d, f, r, dt):
    sd = 1 / math.sqrt(d)
    return oracle.Predictor(d, r, f, dt, synth.normal_matrix(0, synth.tensor_id(l, synth.P_DOWN), r, d, sd, dt),
                            synth.normal_matrix(0, synth.tensor_id(l, synth.P_UP), f, r, sd, dt))


def oracle_stack(x0, L, d, f, r, dt, glu, rho, k, lookahead, scale=0.1):
    """The oracle's own stack, layer by layer.  Returns x_L and the sets."""
    x = np.asarray(x0, np.float64).copy()
    sets = []
    xprev = x.copy()
    for l in range(L):
        src = xprev if (lookahead and l > 0) else x
        _, s = oracle.predict(oracle_predictor(l, d, f, r, dt), src)
        sel = oracle.select_topk(s.astype(np.float32), k)
        sets.append(sel)
        Ly = oracle_layer_rows(l, d, f, dt, glu, rho, sel)
        y = oracle.ffn(Ly, x, np.arange(sel.size, dtype=np.int32))
        xprev = x
        x = x + scale * y
    return x, sets


def gpu_stack(xs, L, d, f, r, dt, glu, rho, k, lookahead, scale=0.1):
    import torch

    import contextual_sparsity_sparse_gb300 as cs
    import synth.device as synthdev
    cs.build.build()
    synthdev.build()
    tdt = {synth.F16: torch.float16, synth.BF16: torch.bfloat16}[dt]
    sd = 1 / math.sqrt(d)
    layers, preds, keep = [], [], []
    for l in range(L):
        t = {}
        for name, which, rows, cols in (("w_gate", synth.W_GATE, f, d), ("w_down_t", synth.W_DOWN_T, f, d),
                                        ("p_down", synth.P_DOWN, r, d), ("p_up", synth.P_UP, f, r)):
            t[name] = torch.empty((rows, cols), dtype=tdt, device="cuda")
            synthdev.fill_normal(t[name], 0, synth.tensor_id(l, which), sd)
        if glu:
            t["w_up"] = torch.empty((f, d), dtype=tdt, device="cuda")
            synthdev.fill_normal(t["w_up"], 0, synth.tensor_id(l, synth.W_UP), sd)
        t["bias"] = torch.from_numpy(synth.zipf_bias(0, l, f, rho)).cuda()
        layers.append(cs.FfnLayer(t["w_gate"], t["w_down_t"], w_up=t.get("w_up"), bias=t["bias"]))
        preds.append(cs.Predictor(t["p_down"], t["p_up"]))
        keep.append(t)
    SA = cs.StackArgs(layers, preds)
    ws = cs.Workspace(d, f, r)
    tc = torch.zeros(L, dtype=torch.int32, device="cuda")
    ti = torch.zeros((L, f), dtype=torch.int32, device="cuda")
    sm, sp = torch.cuda.Stream(), torch.cuda.Stream()
    mode = cs.CS_STACK_LOOKAHEAD if lookahead else cs.CS_STACK_SEQUENTIAL
    out = []
    for x0 in xs:
        x = torch.from_numpy(np.asarray(x0, np.float32).copy()).cuda()
        torch.cuda.synchronize()
        cs.cs_decode_stack(SA, None, x, scale, cs.select_params(cs.CS_SEL_TOPK, k), mode, ws, s_main=sm, s_pred=sp,
                           trace_count=tc, trace_idx=ti)
        torch.cuda.synchronize()
        TC, TI = tc.cpu().numpy(), ti.cpu().numpy()
        out.append((x.cpu().numpy().astype(np.float64), [TI[l, :TC[l]].copy() for l in range(L)]))
    assert cs.cs_get_device_error(ws) == 0
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--workload", default="llama70b", choices=sorted(SHAPES))
    ap.add_argument("--mode", default="lookahead", choices=["lookahead", "seq"])
    ap.add_argument("--tokens", type=int, default=2)
    ap.add_argument("--layers", type=int, default=None)
    a = ap.parse_args()
    d, f, r, dt, glu, rho, L = SHAPES[a.workload]
    L = a.layers or L
    k = synth.ceil_k(f, rho)
    lookahead = a.mode == "lookahead"
    oracle.build()
    xs = synth.x_normal(4242, a.tokens, d)
    t0 = time.time()
    gpu = gpu_stack(xs, L, d, f, r, dt, glu, rho, k, lookahead)
    t1 = time.time()
    rows = []
    for t, x0 in enumerate(xs):
        oxL, osets = oracle_stack(x0, L, d, f, r, dt, glu, rho, k, lookahead)
        gxL, gsets = gpu[t]
        jac = [np.intersect1d(g, o).size / max(np.union1d(g, o).size, 1) for g, o in zip(gsets, osets)]
        same = [bool(np.array_equal(g, o)) for g, o in zip(gsets, osets)]
        first_diff = next((l for l, s in enumerate(same) if not s), None)
        rows.append({"token": t, "rel_err_xL": float(np.abs(gxL - oxL).max() / np.abs(oxL).max()),
                     "layers_identical": int(sum(same)), "first_layer_differing": first_diff,
                     "mean_jaccard": float(np.mean(jac)), "min_jaccard": float(np.min(jac))})
    print(json.dumps({"workload": a.workload, "mode": a.mode, "layers": L, "k": k, "tokens": a.tokens,
                      "gpu_s": round(t1 - t0, 1), "oracle_s": round(time.time() - t1, 1), "per_token": rows}))


if __name__ == "__main__":
    main()
