"""Recall and precision of three predictor constructions for one OPT-13B-shaped
layer, against the exact mask {g > 0}, on the CPU (oracle side).

"Contextual Sparsity: Activation-Aware LLM Inference and the Deja Vu
Paradigm", section "The Prediction Problem" (a small low-rank predictor
trained to reproduce the layer's active set) and "Contextual Sparsity and
Activation Predictors", section "Precision, recall, and which error hurts".

The predictor scores s = P_up relu(P_down x), rank r (no bias term).  With
g = W_gate x + b the layer's gate pre-activations:

  random+ridge   P_down random (the seeded synthetic predictor), P_up the ridge
                 regression of g onto relu(P_down x) over calibration tokens
                 (oracle.fit_predictor, the same fit cs_fit_predictor runs);
  svd            the closed form of the best rank-q approximation of W_gate:
                 V_q = the top q = r/2 right singular vectors (eigenvectors of
                 W_gate^T W_gate), P_down = [V_q; -V_q], P_up = [W V_q^T, -W V_q^T],
                 so relu(P_down x) differences give s = W V_q^T V_q x exactly
                 (the bias b cannot enter: the predictor has no constant term);
  svd+ridge      the same P_down, P_up fitted by the ridge regression.

Scores and masks are fp64 (the predictor weights are not rounded); top-k
takes the k largest scores.  Not a test: prints one JSON line.

    python tests/predictor_report.py [--tokens 32] [--calib 2048]
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

D, F, R, RHO = 5120, 20480, 512, 0.10
SHARES = (0.05, 0.10, 0.15, 0.20, 0.30)


def curve(S, G):
    """Mean recall / precision of top-k of each row of S against {G > 0}."""
    out = []
    for q in SHARES:
        k = synth.ceil_k(F, q)
        rec, prec = [], []
        for s, g in zip(S, G):
            top = np.argpartition(-s, k - 1)[:k]
            act = g > 0
            hit = int(act[top].sum())
            rec.append(hit / max(int(act.sum()), 1))
            prec.append(hit / k)
        out.append({"share": q, "k": k, "recall": round(float(np.mean(rec)), 4),
                    "precision": round(float(np.mean(prec)), 4)})
    return out


def ridge(Pd, W, b, Xc, lam):
    H = np.maximum(Xc @ Pd.T, 0.0)
    G = Xc @ W.T + b
    return np.linalg.solve(H.T @ H + lam * np.eye(Pd.shape[0]), H.T @ G).T


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--tokens", type=int, default=32)
    ap.add_argument("--calib", type=int, default=2048)
    ap.add_argument("--lam-per-token", type=float, default=1e-3)
    a = ap.parse_args()
    t0 = time.time()
    sd = 1 / math.sqrt(D)
    W = oracle.decode(synth.normal_matrix(0, synth.tensor_id(0, synth.W_GATE), F, D, sd, synth.F16), synth.F16)
    W = W.reshape(F, D)
    b = synth.zipf_bias(0, 0, F, RHO).astype(np.float64)
    Pd = oracle.decode(synth.normal_matrix(0, synth.tensor_id(0, synth.P_DOWN), R, D, sd, synth.F16), synth.F16)
    Pd = Pd.reshape(R, D)
    Xc = synth.x_normal(5000, a.calib, D).astype(np.float64)
    Xt = synth.x_normal(7000, a.tokens, D).astype(np.float64)
    G = Xt @ W.T + b
    lam = a.lam_per_token * a.calib

    res = {}
    Pu = ridge(Pd, W, b, Xc, lam)
    res["random+ridge"] = curve(np.maximum(Xt @ Pd.T, 0) @ Pu.T, G)

    # top q eigenvectors of W^T W = the top right singular vectors of W
    q = R // 2
    evals, evecs = np.linalg.eigh(W.T @ W)
    order = np.argsort(evals)[::-1]
    Vq = evecs[:, order[:q]].T                       # [q, D]
    captured = float(evals[order[:q]].sum() / evals.sum())
    Pd2 = np.vstack([Vq, -Vq])
    WV = W @ Vq.T
    Pu2 = np.hstack([WV, -WV])
    H2 = np.maximum(Xt @ Pd2.T, 0)
    res["svd"] = curve(H2 @ Pu2.T, G)
    res["svd+ridge"] = curve(H2 @ ridge(Pd2, W, b, Xc, lam).T, G)
    print(json.dumps({"layer": "opt13b (d=5120, f=20480), layer 0, fp16 weights decoded to fp64",
                      "r": R, "svd_rank": q, "variance_captured_by_svd_rank": round(captured, 4),
                      "calibration_tokens": a.calib, "lambda": lam, "held_out_tokens": a.tokens,
                      "mean_exact_mask_size": float((G > 0).sum(1).mean()), "curves": res,
                      "seconds": round(time.time() - t0, 1)}))


if __name__ == "__main__":
    main()
