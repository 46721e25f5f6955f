"""Benchmark: sparse-FFN decode tokens/s at batch 1 on one GB300, with the HBM
roofline fraction of the dominant kernel and the CPU oracle as baseline.

Default workload: the OPT-13B-shaped layer (d=5120, f=20480, predictor r=512,
fp16 weights, fp32 accumulation), top-k selection at 10% (k=2048), batch 1.
A step is one token through the whole hot path: predictor (two GEMVs), top-k
selection, gathered FFN (gate GEMV + ReLU + down AXPY + reduction).  Steps
rotate over NCOPY independent layer copies and 512 distinct inputs, so each
copy's touched bytes are evicted from L2 by the other copies before reuse.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas: the path has no exchange step); value = all ranks' steps / max time.
--impl reference times the CPU oracle (the only reference this method has) on
rank 0.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "sparse-FFN decode tokens/s at batch 1 and effective HBM GB/s vs GB300 peak"

WORKLOADS = {
    # name: d, f, r, dtype, glu, rho (profile), mode, share (k or threshold quantile)
    "opt13b-topk10": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.10),
    "opt13b-topk5": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.05),
    "opt13b-topk20": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.20),
    "opt13b-thr10": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="threshold", share=0.10),
    "tiny-relu-topk10": dict(d=512, f=2048, r=64, dt=0, glu=False, rho=0.10, mode="topk", share=0.10),
    # frequency-sorted layout: the 1024 hottest neurons always on, top-k 5% of
    # the other 19,456 predicted (10% active in all, as opt13b-topk10)
    "opt13b-hot5-topk5": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.05,
                              hot=1024),
    # opt13b-topk10 with every up map fitted to its layer (ridge regression over
    # 2,048 synthetic calibration tokens); the line adds recall and precision
    "opt13b-fitted-topk10": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.10,
                                 fit=dict(N=2048, lam_per_token=1e-3)),
    # head-sparse attention of an OPT-13B-shaped layer: 40 heads of 128, a
    # 2,048-position KV cache, the top 25% of heads by a predictor (r = 128)
    "opt13b-attn-heads25": dict(d=5120, H=40, dh=128, S=2048, r=128, dt=1, share=0.25, attn=True),
    # one LLaMA-70B-shaped SwiGLU layer with SiLU kept (functional sparsity), top-k 15%
    "llama70b-silu-topk15": dict(d=8192, f=28672, r=1024, dt=2, glu=True, rho=0.15, mode="topk", share=0.15,
                                 act=1),
    # layer stacks: one step = one token through every layer (cs_decode_stack)
    "opt30b-stack-seq": dict(d=7168, f=28672, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.10,
                             L=48, stack="seq"),
    "opt30b-stack-lookahead": dict(d=7168, f=28672, r=512, dt=1, glu=False, rho=0.10, mode="topk", share=0.10,
                                   L=48, stack="lookahead"),
    "llama70b-stack-seq": dict(d=8192, f=28672, r=1024, dt=2, glu=True, rho=0.15, mode="topk", share=0.15,
                               L=80, stack="seq"),
    "llama70b-stack-lookahead": dict(d=8192, f=28672, r=1024, dt=2, glu=True, rho=0.15, mode="topk",
                                     share=0.15, L=80, stack="lookahead"),
}
# batched union (Falcon-40B-shaped layer): a step = union of B token masks +
# the batched FFN over the union, for B tokens
for _B in (1, 2, 4, 8, 16, 32):
    WORKLOADS[f"falcon40b-union-b{_B}"] = dict(d=8192, f=32768, r=1, dt=2, glu=False, rho=0.10, mode="union",
                                              share=0.10, union=_B)
NCOPY = 8
NX = 200


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=20000)
    p.add_argument("--warmup", type=int, default=2000)
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default="opt13b-topk10", choices=sorted(WORKLOADS))
    p.add_argument("--cpu-sample-s", type=float, default=12.0)
    p.add_argument("--no-cpu-baseline", action="store_true")
    return p.parse_args()


def peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as fh:
            m = json.load(fh)
        return float(m["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


class Clocks:
    """nvidia-smi sampling during the timed region."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, dev_index):
        self.dev = dev_index
        self.proc = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except Exception:
            self.proc = None

    def stop(self):
        if not self.proc:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        out, _ = self.proc.communicate(timeout=10)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in out.splitlines():
            parts = [x.strip() for x in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for n, v in zip(names, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(sm), "reasons": sorted(reasons)}


def src_sha(path):
    with open(path, "rb") as fh:
        return hashlib.sha256(fh.read()).hexdigest()[:16]


def profile_traffic(kernel, workload):
    """DRAM bytes per launch from a committed ncu summary, if the kernel source
    is unchanged since the capture; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            t = json.load(fh)
        e = t[kernel][workload]
        if e["source_sha"] != src_sha(os.path.join(ROOT, e["source"])):
            return None
        return e["traffic_bytes"]
    except Exception:
        return None


# ----------------------------------------------------------------------------
# replicas across ranks (one process per GPU, no data-path collective)
# ----------------------------------------------------------------------------

def init_dist(world):
    """Join the process group (NCCL on GPUs, gloo on CPU-only hosts)."""
    if world <= 1:
        return
    import torch
    import torch.distributed as dist
    dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")


def max_over_ranks(ms, world):
    """The largest per-rank elapsed time, returned on every rank."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([ms], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def replica_value(units_per_rank, world, ms):
    """Whole-job throughput: the units all ranks processed / the slowest rank's time."""
    return world * units_per_rank / (ms / 1e3)


# ----------------------------------------------------------------------------
# our arm
# ----------------------------------------------------------------------------

def build_copies(W, torch, cs, synthdev):
    import synth
    d, f, r, dt = W["d"], W["f"], W["r"], W["dt"]
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[dt]
    sd = 1 / math.sqrt(d)
    copies = []
    for l in range(NCOPY):
        t = {}
        for name, which, rows, cols in (("w_gate", synth.W_GATE, f, d), ("w_down_t", synth.W_DOWN_T, f, d),
                                        ("p_down", synth.P_DOWN, r, d), ("p_up", synth.P_UP, f, r)):
            t[name] = torch.empty((rows, cols), dtype=tdt, device="cuda")
            synthdev.fill_normal(t[name], 0, synth.tensor_id(l, which), sd)
        if W["glu"]:
            t["w_up"] = torch.empty((f, d), dtype=tdt, device="cuda")
            synthdev.fill_normal(t["w_up"], 0, synth.tensor_id(l, synth.W_UP), sd)
        t["bias"] = torch.from_numpy(synth.zipf_bias(0, l, f, W["rho"])).cuda()
        hot = W.get("hot", 0)
        if hot:
            # the frequency-sorted layout: rows hottest first (layer l's own
            # firing profile), the predictor's up map for the tail only
            perm = cs.cs_hot_order(synth.firing_probs(0, l, f, W["rho"])).cuda()
            for name in ("w_gate", "w_down_t", "w_up", "bias"):
                if name in t:
                    dst = torch.empty_like(t[name])
                    cs.cs_permute_rows(t[name], perm, dst)
                    t[name] = dst
            pu = torch.empty((f - hot, r), dtype=tdt, device="cuda")
            cs.cs_permute_rows(t["p_up"], perm[hot:], pu)
            t["p_up"] = pu
        layer = cs.FfnLayer(t["w_gate"], t["w_down_t"], w_up=t.get("w_up"), bias=t["bias"], act=W.get("act", 0))
        pred = cs.Predictor(t["p_down"], t["p_up"])
        copies.append((layer, pred, t))
    torch.cuda.synchronize()
    return copies


def fitted_quality(cs, torch, copy, d, f, r, k, n_tokens=32):
    """Mean recall and precision of a layer copy's predictor (top-k) against
    the exact mask {g > 0}, both computed on the GPU, over held-out tokens."""
    import numpy as np
    import synth
    layer, pred, _ = copy
    ws = cs.Workspace(d, f, r)
    pre = torch.empty(f, device="cuda")
    ei = torch.empty(f, dtype=torch.int32, device="cuda")
    ec = torch.empty(1, dtype=torch.int32, device="cuda")
    y = torch.empty(d, device="cuda")
    sc = torch.empty((1, f), device="cuda")
    pi = torch.empty((1, f), dtype=torch.int32, device="cuda")
    pc = torch.empty(1, dtype=torch.int32, device="cuda")
    rec, prec = [], []
    for x in synth.x_normal(7000, n_tokens, d):
        xt = torch.from_numpy(x[None]).cuda()
        cs.cs_exact_ffn(layer, xt, pre, ei, ec, y, ws)
        cs.cs_predict(pred, xt, sc, ws)
        cs.cs_select(sc, cs.select_params(cs.CS_SEL_TOPK, k), pi, pc, ws=ws)
        torch.cuda.synchronize()
        P = pi.cpu().numpy()[0, :int(pc.item())]
        E = ei.cpu().numpy()[:int(ec.item())]
        hit = np.intersect1d(P, E).size
        rec.append(hit / max(E.size, 1))
        prec.append(hit / max(P.size, 1))
    return float(np.mean(rec)), float(np.mean(prec))


def step_bytes(W, k):
    """Algorithmic bytes of one step (S8(d)-style accounting): predictor weights,
    scores written and read, selected rows (+ index and bias), x and y."""
    d, f, r = W["d"], W["f"], W["r"]
    hot = W.get("hot", 0)   # always-on prefix: not predicted, always gathered
    e = 4 if W["dt"] == 0 else 2
    m = 3 if W["glu"] else 2
    pred = e * (r * d + (f - hot) * r) + 4 * (d + r) * 2
    sel = 4 * (f - hot) + 4 * (hot + k)
    ffn = (hot + k) * (m * d * e + 4 + 4) + 4 * d * 2
    return pred + sel + ffn, ffn


def run_ours(args, W, rank, world):
    import torch
    import contextual_sparsity_sparse_gb300 as cs
    import synth
    import synth.device as synthdev
    from contextual_sparsity_sparse_gb300 import build as cb

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    cb.build()
    synthdev.build()
    d, f, r = W["d"], W["f"], W["r"]
    k = synth.ceil_k(f, W["share"])
    copies = build_copies(W, torch, cs, synthdev)
    quality = None
    if W.get("fit"):
        # setup: fit every copy's up map, then measure the first copy's
        # recall / precision against the exact mask on held-out tokens
        Nc, lam = W["fit"]["N"], W["fit"]["lam_per_token"] * W["fit"]["N"]
        rec0, _ = fitted_quality(cs, torch, copies[0], d, f, r, k)
        for l, (layer, pred, _) in enumerate(copies):
            cs.cs_fit_predictor(layer, pred, torch.from_numpy(synth.x_normal(5000 + l, Nc, d)).cuda(), lam)
        rec, prec = fitted_quality(cs, torch, copies[0], d, f, r, k)
        quality = {"recall": rec, "precision": prec, "k": k, "random_up_map_recall": rec0,
                   "calibration_tokens": Nc, "lambda": lam, "held_out_tokens": 32,
                   "against": "exact mask {g > 0} (cs_exact_ffn) per held-out token"}
    X = torch.from_numpy(synth.x_normal(1000 + rank, NX, d)).cuda()
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, f, r, stream=s)
    hot = W.get("hot", 0)
    scores = torch.empty((1, f - hot), device="cuda")
    idx = torch.empty((1, f), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    Y = torch.empty((NX, d), device="cuda")
    if W["mode"] == "topk":
        params = cs.select_params(cs.CS_SEL_TOPK, k, hot=hot)
    else:
        # threshold at the (1 - share) quantile of calibration scores (seed 1)
        layer0, pred0, _ = copies[0]
        Xc = torch.from_numpy(synth.x_normal(1, 256, d)).cuda()
        sc = torch.empty((256, f), device="cuda")
        cs.cs_predict(pred0, Xc, sc, cs.Workspace(d, f, r, 256))
        torch.cuda.synchronize()
        tau = float(torch.quantile(sc.flatten()[:: 7].float(), 1 - W["share"]))
        params = cs.select_params(cs.CS_SEL_THRESHOLD, 0, tau)

    def one_step(i, with_events=None):
        layer, pred, _ = copies[i % NCOPY]
        x = X[i % NX: i % NX + 1]
        cs.cs_predict(pred, x, scores, ws, stream=s)
        cs.cs_select(scores, params, idx, cnt, ws=ws, stream=s)
        if with_events is not None:
            with_events[0].record(s)
        cs.cs_sparse_ffn(layer, x, idx, cnt, Y[i % NX: i % NX + 1], ws, stream=s)
        if with_events is not None:
            with_events[1].record(s)

    # graph of NB steps (launch overhead out of the timed region)
    NB = 200
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(3):
            one_step(i)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(NB):
                one_step(i)
    K = max(NB, (args.steps // NB) * NB)
    Wm = max(3 * NB, (args.warmup // NB) * NB)
    with torch.cuda.stream(s):
        for _ in range(Wm // NB):
            g.replay()
    s.synchronize()
    if world > 1:
        barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(dev)
    clk.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(K // NB):
            g.replay()
    e1.record(s)
    e1.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    torch.cuda.synchronize()
    ms = max_over_ranks(ms, world)
    barrier(world)
    assert cs.cs_get_device_error(ws, stream=s) == 0

    # roofline pass: the FFN calls of the first NB steps alone, back to back on
    # the same stream (their index lists computed first), timed with CUDA events
    # around graph replays: the average duration of one cs_sparse_ffn launch
    # (gather + reduce) over the same rows the timed steps gather
    idx_all = torch.empty((NB, f), dtype=torch.int32, device="cuda")
    cnt_all = torch.empty(NB, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        for i in range(NB):
            layer, pred, _ = copies[i % NCOPY]
            cs.cs_predict(pred, X[i % NX: i % NX + 1], scores, ws, stream=s)
            cs.cs_select(scores, params, idx_all[i: i + 1], cnt_all[i: i + 1], ws=ws, stream=s)
    s.synchronize()

    def ffn_call(i):
        layer, _, _ = copies[i % NCOPY]
        cs.cs_sparse_ffn(layer, X[i % NX: i % NX + 1], idx_all[i], cnt_all[i: i + 1], Y[i % NX: i % NX + 1],
                         ws, stream=s)

    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        for i in range(3):
            ffn_call(i)
        s.synchronize()
        with torch.cuda.graph(g2, stream=s):
            for i in range(NB):
                ffn_call(i)
        for _ in range(3):
            g2.replay()
    s.synchronize()
    reps = max(3, K // NB // 4)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g2.replay()
    f1.record(s)
    f1.synchronize()
    ffn_avg_s = f0.elapsed_time(f1) / 1e3 / (reps * NB)

    # e2e: one cs_decode_layer call per token with x and y in pinned host
    # memory; the library copies x in and y out on the stream every step
    KE = min(K, 2000)
    xh = torch.from_numpy(synth.x_normal(2000 + rank, 64, d)).pin_memory()
    yh = torch.empty((64, d)).pin_memory()
    xslot, yslot = list(xh.unbind(0)), list(yh.unbind(0))   # the caller's 64 token slots

    def e2e_step(i):
        layer, pred, _ = copies[i % NCOPY]
        cs.cs_decode_layer(layer, pred, xslot[i % 64], yslot[i % 64], params, ws, stream=s)

    with torch.cuda.stream(s):
        for i in range(50):
            e2e_step(i)
    s.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for i in range(KE):
            e2e_step(i)
    s.synchronize()
    e2e_s = time.perf_counter() - t0

    total_b, ffn_b = step_bytes(W, k)
    hbm, src = peaks()
    step_s = ms / 1e3 / K
    ffn_gbs = ffn_b / ffn_avg_s / 1e9
    res = {
        "metric": METRIC, "value": replica_value(K, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "d": d, "f": f, "r": r, "k": k if W["mode"] == "topk" else None,
                   "activation": "silu" if W.get("act", 0) else "relu", "gated": W["glu"],
                   **({"hot": hot, "active": hot + k, "layout": "frequency-sorted (cs_hot_order + cs_permute_rows)"}
                      if hot else {}),
                   "selection": W["mode"], "weights": {0: "f32", 1: "f16", 2: "bf16"}[W["dt"]],
                   "accumulate": "f32", "batch": 1, "global_batch": world, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {NCOPY} layer copies ({NCOPY * (2 * f * d + r * d + (f - hot) * r) * (4 if W['dt'] == 0 else 2) / 1e9:.2f} GB) and {NX} inputs rotate; 7 other steps ({7 * total_b / 1e6:.0f} MB) run between uses of a copy",
                   "step": "cs_predict + cs_select + cs_sparse_ffn, graph of 200 steps"},
        "clocks": clocks,
        **({"quality": quality} if quality else {}),
        "gpu_launches": 5 * K,
        "roofline": {"bound": "hbm", "kernel": "cs_sparse_ffn (gather + fixed-order reduce)",
                     "achieved": ffn_gbs, "peak": hbm, "unit": "GB/s", "frac": ffn_gbs / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                     "bytes_per_launch": ffn_b, "avg_launch_us": ffn_avg_s * 1e6,
                     "traffic": profile_traffic("cs_sparse_ffn", args.workload)},
        "step_roofline": {"bytes_per_step": total_b, "achieved": total_b / step_s / 1e9, "peak": hbm,
                          "frac": total_b / step_s / 1e9 / hbm, "unit": "GB/s"},
        "e2e": {"value": world * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * d,
                "d2h_bytes_per_step": 4 * d, "steps": KE,
                "how": "one cs_decode_layer call per token through the Python binding, x and y in pinned host memory (the call copies x in, replays the layer's graph of predict + select + gathered FFN, copies y out); wall clock"},
    }
    return res, copies


def run_stack(args, W, rank, world):
    """K tokens through the whole L-layer stack (one cs_decode_stack call each,
    replaying the library's cached graph), fresh x per token."""
    import torch
    import contextual_sparsity_sparse_gb300 as cs
    import synth
    import synth.device as synthdev
    from contextual_sparsity_sparse_gb300 import build as cb

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    cb.build()
    synthdev.build()
    d, f, r, L = W["d"], W["f"], W["r"], W["L"]
    k = synth.ceil_k(f, W["share"])
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[W["dt"]]
    sd = 1 / math.sqrt(d)
    layers, preds, keep = [], [], []
    for l in range(L):
        t = {}
        for name, which, rows, cols in (("w_gate", synth.W_GATE, f, d), ("w_down_t", synth.W_DOWN_T, f, d),
                                        ("p_down", synth.P_DOWN, r, d), ("p_up", synth.P_UP, f, r)):
            t[name] = torch.empty((rows, cols), dtype=tdt, device="cuda")
            synthdev.fill_normal(t[name], 0, synth.tensor_id(l, which), sd)
        if W["glu"]:
            t["w_up"] = torch.empty((f, d), dtype=tdt, device="cuda")
            synthdev.fill_normal(t["w_up"], 0, synth.tensor_id(l, synth.W_UP), sd)
        t["bias"] = torch.from_numpy(synth.zipf_bias(0, l, f, W["rho"])).cuda()
        layers.append(cs.FfnLayer(t["w_gate"], t["w_down_t"], w_up=t.get("w_up"), bias=t["bias"]))
        preds.append(cs.Predictor(t["p_down"], t["p_up"]))
        keep.append(t)
    torch.cuda.synchronize()
    NXS = 64
    X = torch.from_numpy(synth.x_normal(5000 + rank, NXS, d)).cuda()
    x = torch.empty(d, device="cuda")
    sm, sp = torch.cuda.Stream(), torch.cuda.Stream()
    ws = cs.Workspace(d, f, r, stream=sm)
    params = cs.select_params(cs.CS_SEL_TOPK, k)
    mode = cs.CS_STACK_LOOKAHEAD if W["stack"] == "lookahead" else cs.CS_STACK_SEQUENTIAL

    def step(i):
        x.copy_(X[i % NXS], non_blocking=True)
        cs.cs_decode_stack(layers, preds, x, 0.1, params, mode, ws, s_main=sm, s_pred=sp)

    torch.cuda.synchronize()
    with torch.cuda.stream(sm):
        for i in range(max(3, args.warmup)):
            step(i)
    sm.synchronize()
    K = max(1, args.steps)
    if world > 1:
        barrier(world)
    clk = Clocks(dev)
    clk.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(sm):
        e0.record(sm)
        for i in range(K):
            step(i)
        e1.record(sm)
    e1.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    assert cs.cs_get_device_error(ws, stream=sm) == 0
    # e2e through the API with host buffers
    KE = min(K, 50)
    xh = torch.from_numpy(synth.x_normal(6000 + rank, NXS, d)).pin_memory()
    yh = torch.empty((NXS, d)).pin_memory()
    with torch.cuda.stream(sm):
        for i in range(3):
            x.copy_(xh[i], non_blocking=True)
            cs.cs_decode_stack(layers, preds, x, 0.1, params, mode, ws, s_main=sm, s_pred=sp)
            yh[i].copy_(x, non_blocking=True)
    sm.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(sm):
        for i in range(KE):
            x.copy_(xh[i % NXS], non_blocking=True)
            cs.cs_decode_stack(layers, preds, x, 0.1, params, mode, ws, s_main=sm, s_pred=sp)
            yh[i % NXS].copy_(x, non_blocking=True)
    sm.synchronize()
    e2e_s = time.perf_counter() - t0
    tot_b, ffn_b = step_bytes(W, k)
    per_token = L * tot_b
    hbm, src = peaks()
    step_s = ms / 1e3 / K
    return {
        "metric": METRIC, "value": replica_value(K, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": max(3, args.warmup), "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "layers": L, "d": d, "f": f, "r": r, "k": k, "selection": "topk",
                   "stack": W["stack"], "weights": {0: "f32", 1: "f16", 2: "bf16"}[W["dt"]],
                   "gated": W["glu"], "accumulate": "f32", "batch": 1, "global_batch": world,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: the stack's weights ({L * (2 + W['glu']) * f * d * (4 if W['dt'] == 0 else 2) / 1e9:.0f} GB) are read once per token",
                   "step": "one token through every layer: cs_decode_stack (graph replay), fresh x per token"},
        "clocks": clocks,
        "gpu_launches": K * L * (5 if W["stack"] else 5),
        "roofline": {"bound": "hbm", "kernel": "whole decode step (predictor, select, gathered FFN of every layer)",
                     "achieved": per_token / step_s / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": per_token / step_s / 1e9 / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)", "bytes_per_launch": per_token,
                     "avg_launch_us": step_s * 1e6, "traffic": None},
        "e2e": {"value": world * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * d,
                "d2h_bytes_per_step": 4 * d, "steps": KE,
                "how": "per token: pinned H2D of x, cs_decode_stack, D2H of x_L; wall clock"},
    }


def oracle_step_inputs(W, layer_index=0):
    import numpy as np
    import oracle
    import synth
    d, f, r, dt = W["d"], W["f"], W["r"], W["dt"]
    sd = 1 / math.sqrt(d)
    mk = lambda which, rows, cols: synth.normal_matrix(0, synth.tensor_id(layer_index, which), rows, cols, sd, dt)
    L = oracle.Layer(d, f, dt, mk(synth.W_GATE, f, d), mk(synth.W_DOWN_T, f, d),
                     w_up=mk(synth.W_UP, f, d) if W["glu"] else None,
                     bias=synth.zipf_bias(0, layer_index, f, W["rho"]), act=W.get("act", 0))
    P = oracle.Predictor(d, r, f, dt, mk(synth.P_DOWN, r, d), mk(synth.P_UP, f, r))
    return L, P


def run_union(args, W, rank, world):
    """B tokens per step: cs_union_mask over their active-set masks, then
    cs_sparse_ffn of all B tokens over the union (tensor-core path from
    B = 4 on), rotating over layer copies and mask sets."""
    import torch
    import contextual_sparsity_sparse_gb300 as cs
    import synth
    import synth.device as synthdev
    from contextual_sparsity_sparse_gb300 import build as cb

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    cb.build()
    synthdev.build()
    d, f, B = W["d"], W["f"], W["union"]
    words = (f + 31) // 32
    tdt = torch.bfloat16 if W["dt"] == 2 else torch.float16
    NCU, NM = 3, 32
    copies = []
    for l in range(NCU):
        t = {}
        for name, which in (("w_gate", synth.W_GATE), ("w_down_t", synth.W_DOWN_T)):
            t[name] = torch.empty((f, d), dtype=tdt, device="cuda")
            synthdev.fill_normal(t[name], 0, synth.tensor_id(l, which), 1 / math.sqrt(d))
        t["bias"] = torch.from_numpy(synth.zipf_bias(0, l, f, W["rho"])).cuda()
        copies.append((cs.FfnLayer(t["w_gate"], t["w_down_t"], bias=t["bias"]), t))
    import numpy as np
    masks = torch.from_numpy(np.stack([synth.union_masks(7000 + 97 * rank + i, B, f, W["rho"])
                                       for i in range(NM)]).view(np.int32)).cuda()      # [NM, B, words]
    X = torch.from_numpy(synth.x_normal(8000 + rank, NM * B, d).reshape(NM, B, d)).cuda()
    Y = torch.empty((B, d), device="cuda")
    umask = torch.empty(words, dtype=torch.int32, device="cuda")
    uidx = torch.empty((NM, f), dtype=torch.int32, device="cuda")
    ucnt = torch.empty(NM, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, f, 1, B, stream=s)

    def step(i, ffn_only=False):
        m = i % NM
        if not ffn_only:
            cs.cs_union_mask(masks[m], f, umask, uidx[m], ucnt[m: m + 1], ws, stream=s)
        cs.cs_sparse_ffn(copies[i % NCU][0], X[m], uidx[m], ucnt[m: m + 1], Y, ws, stream=s)

    NB = 64
    with torch.cuda.stream(s):
        for i in range(NM):
            step(i)
    s.synchronize()
    mean_u = float(ucnt.float().mean().item())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(NB):
                step(i)
    K = max(NB, (args.steps // NB) * NB)
    Wm = max(3 * NB, (args.warmup // NB) * NB)
    with torch.cuda.stream(s):
        for _ in range(Wm // NB):
            g.replay()
    s.synchronize()
    if world > 1:
        barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(dev)
    clk.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(K // NB):
            g.replay()
    e1.record(s)
    e1.synchronize()
    clocks = clk.stop()
    ms = e0.elapsed_time(e1)
    ms = max_over_ranks(ms, world)
    barrier(world)
    assert cs.cs_get_device_error(ws, stream=s) == 0

    # roofline pass: the batched FFN calls alone (unions already computed)
    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g2, stream=s):
            for i in range(NB):
                step(i, ffn_only=True)
        for _ in range(3):
            g2.replay()
    s.synchronize()
    reps = max(3, K // NB // 4)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g2.replay()
    f1.record(s)
    f1.synchronize()
    ffn_s = f0.elapsed_time(f1) / 1e3 / (reps * NB)

    # e2e through the binding: pinned host masks and x in, y out, every step
    KE = min(K, 400)
    mh = masks.cpu().pin_memory()
    xh = X.cpu().pin_memory()
    yh = torch.empty((B, d)).pin_memory()
    md = torch.empty((B, words), dtype=torch.int32, device="cuda")
    xd = torch.empty((B, d), device="cuda")

    def e2e_step(i):
        m = i % NM
        md.copy_(mh[m], non_blocking=True)
        xd.copy_(xh[m], non_blocking=True)
        cs.cs_union_mask(md, f, umask, uidx[0], ucnt[0:1], ws, stream=s)
        cs.cs_sparse_ffn(copies[i % NCU][0], xd, uidx[0], ucnt[0:1], Y, ws, stream=s)
        yh.copy_(Y, non_blocking=True)

    with torch.cuda.stream(s):
        for i in range(10):
            e2e_step(i)
    s.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for i in range(KE):
            e2e_step(i)
    s.synchronize()
    e2e_s = time.perf_counter() - t0

    hbm, src = peaks()
    ffn_b = mean_u * (2 * d * 2 + 4 + 4) + 2 * 4 * B * d
    step_b = ffn_b + 4 * B * words + 4 * words + 4 * mean_u
    tc = 4 <= B and B >= int(os.environ.get("CS_TC_MIN_B", "4")) and B <= 32
    launches = 1 + (4 if tc else 2)
    flops = 2 * mean_u * d * 2 * (2 * B)   # two GEMMs, N = 2B (hi and lo halves)
    res = {
        "metric": METRIC, "value": replica_value(B * K, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "d": d, "f": f, "batch": B, "global_batch": world * B,
                   "weights": "bf16", "accumulate": "f32", "union_mean": mean_u, "union_density": mean_u / f,
                   "path": "tcgen05 gathered GEMM" if tc else "CUDA-core gathered GEMV",
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {NCU} layer copies ({NCU * 2 * f * d * 2 / 1e9:.2f} GB) and {NM} mask sets rotate",
                   "step": "cs_union_mask + cs_sparse_ffn over B tokens, graph of 64 steps"},
        "clocks": clocks,
        "gpu_launches": launches * K,
        "roofline": {"bound": "hbm", "kernel": "cs_sparse_ffn over the union (" + ("split + tcgen05 gate GEMM + tcgen05 down GEMM + reduce" if tc else "gather + reduce") + ")",
                     "achieved": ffn_b / ffn_s / 1e9, "peak": hbm, "unit": "GB/s", "frac": ffn_b / ffn_s / 1e9 / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                     "bytes_per_launch": ffn_b, "avg_launch_us": ffn_s * 1e6,
                     "tensor_tflops": flops / ffn_s / 1e12 if tc else None,
                     "traffic": profile_traffic("cs_sparse_ffn", args.workload)},
        "step_roofline": {"bytes_per_step": step_b, "achieved": step_b / (ms / 1e3 / K) / 1e9, "peak": hbm,
                          "frac": step_b / (ms / 1e3 / K) / 1e9 / hbm, "unit": "GB/s"},
        "e2e": {"value": world * B * KE / e2e_s, "unit": "tokens/s",
                "h2d_bytes_per_step": B * words * 4 + B * d * 4, "d2h_bytes_per_step": B * d * 4, "steps": KE,
                "how": "Python binding per step: pinned H2D of masks and x, cs_union_mask, cs_sparse_ffn, D2H of y; wall clock"},
    }
    return res


def time_oracle_union(W, budget_s, max_steps=None):
    """Time the oracle's union step (mask union, then the sparse FFN of B tokens)."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    B, d, f = W["union"], W["d"], W["f"]
    Ly = oracle.Layer(d, f, W["dt"], synth.normal_matrix(0, synth.tensor_id(0, synth.W_GATE), f, d, 1 / math.sqrt(d), W["dt"]),
                      synth.normal_matrix(0, synth.tensor_id(0, synth.W_DOWN_T), f, d, 1 / math.sqrt(d), W["dt"]),
                      bias=synth.zipf_bias(0, 0, f, W["rho"]))
    X = synth.x_normal(9000, B, d)
    n, tok, t0 = 0, 0, time.perf_counter()
    while True:
        _, wi = oracle.union(synth.union_masks(9100 + n, B, f, W["rho"]), f)
        for b in range(B):
            oracle.ffn(Ly, X[b], wi)
            tok += 1
            el = time.perf_counter() - t0
            if el >= budget_s:
                break
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and n >= max_steps):
            break
    return tok, el, oracle.threads()


def time_oracle(W, budget_s, max_steps=None):
    """Time the oracle's decode step (predict, select, gathered FFN) on the host."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    L, P = oracle_step_inputs(W)
    k = synth.ceil_k(W["f"], W["share"])
    hot = W.get("hot", 0)
    if hot:   # the frequency-sorted layout, built by the oracle's own order
        perm = oracle.hot_order(synth.firing_probs(0, 0, W["f"], W["rho"]))
        pr = lambda a: oracle.permute_rows(a, perm) if a is not None else None
        L = oracle.Layer(L.d, L.f, L.dtype, pr(L.w_gate), pr(L.w_down_t), w_up=pr(L.w_up), bias=pr(L.bias),
                         act=L.act)
        P = oracle.Predictor(P.d, P.r, P.f - hot, P.dtype, P.p_down, oracle.permute_rows(P.p_up, perm[hot:]))
    X = synth.x_normal(3000, 64, W["d"])
    n, t0 = 0, time.perf_counter()
    while True:
        _, s = oracle.predict(P, X[n % 64])
        s32 = s.astype(np.float32)
        if hot:
            sel = oracle.select_hot(s32, hot, oracle.SEL_TOPK, k=k)
        elif W["mode"] == "topk":
            sel = oracle.select_topk(s32, k)
        else:
            if n == 0:  # threshold at the (1 - share) quantile of the oracle's own scores
                tau = np.float32(np.quantile(s32, 1 - W["share"]))
            sel = oracle.select_threshold(s32, tau)
        oracle.ffn(L, X[n % 64], sel)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and n >= max_steps):
            break
    return n, el, oracle.threads()


def attn_bytes(W, k):
    """Algorithmic bytes of one head-sparse attention step: predictor, scores,
    then per selected head its W_q and W_o row blocks and its K and V cache."""
    d, H, dh, S, r = W["d"], W["H"], W["dh"], W["S"], W["r"]
    e = 4 if W["dt"] == 0 else 2
    pred = e * (r * d + H * r) + 4 * (d + r)
    per_head = e * (2 * dh * d + 2 * S * dh)
    attn = k * per_head + 4 * k + 4 * d * 2
    return pred + 8 * H + attn, attn


def run_attn(args, W, rank, world):
    """One token per step: predictor over heads, top-k heads, head-sparse
    attention (cs_sparse_attention), rotating over layer copies."""
    import torch
    import contextual_sparsity_sparse_gb300 as cs
    import synth
    import synth.device as synthdev
    from contextual_sparsity_sparse_gb300 import build as cb

    dev = int(os.environ.get("LOCAL_RANK", "0"))
    torch.cuda.set_device(dev)
    cb.build()
    synthdev.build()
    d, H, dh, S, r = W["d"], W["H"], W["dh"], W["S"], W["r"]
    k = synth.ceil_k(H, W["share"])
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[W["dt"]]
    copies = []
    for l in range(NCOPY):
        t = {}
        for name, which, rows, cols, sd in (("w_q", 0, H * dh, d, 1 / math.sqrt(d)),
                                            ("w_o", 1, H * dh, d, 1 / math.sqrt(dh)),
                                            ("k", 2, H * S, dh, 1.0), ("v", 3, H * S, dh, 1.0),
                                            ("p_down", synth.P_DOWN, r, d, 1 / math.sqrt(d)),
                                            ("p_up", synth.P_UP, H, r, 1 / math.sqrt(r))):
            t[name] = torch.empty((rows, cols), dtype=tdt, device="cuda")
            synthdev.fill_normal(t[name], 0, synth.tensor_id(100 + l, which), sd)
        t["k"], t["v"] = t["k"].view(H, S, dh), t["v"].view(H, S, dh)
        copies.append((cs.AttnLayer(t["w_q"], t["w_o"], H), cs.Predictor(t["p_down"], t["p_up"]), t))
    X = torch.from_numpy(synth.x_normal(1000 + rank, NX, d)).cuda()
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, H, r, stream=s)
    scores = torch.empty((1, H), device="cuda")
    idx_all = torch.empty((NX, H), dtype=torch.int32, device="cuda")
    cnt_all = torch.empty(NX, dtype=torch.int32, device="cuda")
    Y = torch.empty((NX, d), device="cuda")
    params = cs.select_params(cs.CS_SEL_TOPK, k)

    def one_step(i):
        layer, pred, t = copies[i % NCOPY]
        j = i % NX
        cs.cs_predict(pred, X[j:j + 1], scores, ws, stream=s)
        cs.cs_select(scores, params, idx_all[j:j + 1], cnt_all[j:j + 1], ws=ws, stream=s)
        cs.cs_sparse_attention(layer, X[j], idx_all[j], cnt_all[j:j + 1], t["k"], t["v"], Y[j], ws, stream=s)

    NB = 200
    torch.cuda.synchronize()
    with torch.cuda.stream(s):
        for i in range(3):
            one_step(i)
    s.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            for i in range(NB):
                one_step(i)
    K = max(NB, (args.steps // NB) * NB)
    Wm = max(3 * NB, (args.warmup // NB) * NB)
    with torch.cuda.stream(s):
        for _ in range(Wm // NB):
            g.replay()
    s.synchronize()
    if world > 1:
        barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(dev)
    clk.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    with torch.cuda.stream(s):
        for _ in range(K // NB):
            g.replay()
    e1.record(s)
    e1.synchronize()
    clocks = clk.stop()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    assert cs.cs_get_device_error(ws, stream=s) == 0

    # roofline pass: the attention calls of the first NB steps alone (their
    # head lists computed above), back to back on the same stream
    def attn_call(i):
        layer, _, t = copies[i % NCOPY]
        j = i % NX
        cs.cs_sparse_attention(layer, X[j], idx_all[j], cnt_all[j:j + 1], t["k"], t["v"], Y[j], ws, stream=s)

    g2 = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g2, stream=s):
            for i in range(NB):
                attn_call(i)
        for _ in range(3):
            g2.replay()
    s.synchronize()
    reps = max(3, K // NB // 4)
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g2.replay()
    f1.record(s)
    f1.synchronize()
    attn_avg_s = f0.elapsed_time(f1) / 1e3 / (reps * NB)

    # e2e: pinned x in, the three calls, y out, every step
    KE = min(K, 2000)
    xh = torch.from_numpy(synth.x_normal(2000 + rank, 64, d)).pin_memory()
    yh = torch.empty((64, d)).pin_memory()
    xd = torch.empty((1, d), device="cuda")
    yd = torch.empty(d, device="cuda")
    idx1 = torch.empty((1, H), dtype=torch.int32, device="cuda")
    cnt1 = torch.empty(1, dtype=torch.int32, device="cuda")

    def e2e_step(i):
        layer, pred, t = copies[i % NCOPY]
        xd.copy_(xh[i % 64: i % 64 + 1], non_blocking=True)
        cs.cs_predict(pred, xd, scores, ws, stream=s)
        cs.cs_select(scores, params, idx1, cnt1, ws=ws, stream=s)
        cs.cs_sparse_attention(layer, xd[0], idx1[0], cnt1, t["k"], t["v"], yd, ws, stream=s)
        yh[i % 64].copy_(yd, non_blocking=True)

    with torch.cuda.stream(s):
        for i in range(50):
            e2e_step(i)
    s.synchronize()
    t0 = time.perf_counter()
    with torch.cuda.stream(s):
        for i in range(KE):
            e2e_step(i)
    s.synchronize()
    e2e_s = time.perf_counter() - t0

    total_b, attn_b = attn_bytes(W, k)
    hbm, src = peaks()
    step_s = ms / 1e3 / K
    gbs = attn_b / attn_avg_s / 1e9
    return {
        "metric": METRIC, "value": replica_value(K, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": Wm, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "d": d, "heads": H, "d_head": dh, "kv_positions": S, "r": r,
                   "k_heads": k, "weights": {0: "f32", 1: "f16", 2: "bf16"}[W["dt"]], "accumulate": "f32",
                   "batch": 1, "global_batch": world, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {NCOPY} layer copies ({NCOPY * 2 * (H * dh * d + H * S * dh) * (4 if W['dt'] == 0 else 2) / 1e9:.2f} GB) and {NX} inputs rotate",
                   "step": "cs_predict (one score per head) + cs_select (top-k heads) + cs_sparse_attention, graph of 200 steps"},
        "clocks": clocks,
        "gpu_launches": 6 * K,   # predictor (2), select, query, core, reduce
        "roofline": {"bound": "hbm", "kernel": "cs_sparse_attention (per-head attention + fixed-order reduce)",
                     "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                     "bytes_per_launch": attn_b, "avg_launch_us": attn_avg_s * 1e6, "traffic": None},
        "step_roofline": {"bytes_per_step": total_b, "achieved": total_b / step_s / 1e9, "peak": hbm,
                          "frac": total_b / step_s / 1e9 / hbm, "unit": "GB/s"},
        "e2e": {"value": world * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * d,
                "d2h_bytes_per_step": 4 * d, "steps": KE,
                "how": "Python binding per token: pinned H2D of x, cs_predict, cs_select, cs_sparse_attention, D2H of y; wall clock"},
    }


def time_oracle_attn(W, budget_s, max_steps=None):
    """Time the oracle's head-sparse step (predict over heads, top-k, attention)."""
    import numpy as np
    import oracle
    import synth
    oracle.build()
    d, H, dh, S, r, dt = W["d"], W["H"], W["dh"], W["S"], W["r"], W["dt"]
    k = synth.ceil_k(H, W["share"])
    mk = lambda which, rows, cols, sd: synth.normal_matrix(0, synth.tensor_id(100, which), rows, cols, sd, dt)
    A = oracle.AttnLayer(d, H, dh, dt, mk(0, H * dh, d, 1 / math.sqrt(d)), mk(1, H * dh, d, 1 / math.sqrt(dh)))
    kc = mk(2, H * S, dh, 1.0).reshape(H, S, dh)
    vc = mk(3, H * S, dh, 1.0).reshape(H, S, dh)
    P = oracle.Predictor(d, r, H, dt, mk(synth.P_DOWN, r, d, 1 / math.sqrt(d)), mk(synth.P_UP, H, r, 1 / math.sqrt(r)))
    X = synth.x_normal(3000, 64, d)
    n, t0 = 0, time.perf_counter()
    while True:
        _, sc = oracle.predict(P, X[n % 64])
        heads = oracle.select_topk(sc.astype(np.float32), k)
        oracle.attention(A, X[n % 64], heads, kc, vc)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and n >= max_steps):
            break
    return n, el, oracle.threads()


def main():
    args = parse()
    W = WORKLOADS[args.workload]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference" and "union" in W:
        if rank != 0:
            return
        tok, el, cores = time_oracle_union(W, budget_s=20.0, max_steps=max(1, args.steps))
        v = tok / el
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": 1e3 * el / max(1, tok) * W["union"],
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "d": W["d"], "f": W["f"], "batch": W["union"]},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{tok} tokens of union steps, fp64 CPU oracle (at most 20 s)"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    if args.impl == "reference" and W.get("attn"):
        if rank != 0:
            return
        time_oracle_attn(W, budget_s=1e9, max_steps=max(1, args.warmup))
        n, el, cores = time_oracle_attn(W, budget_s=1e9, max_steps=max(1, args.steps))
        v = n / el
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * el / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "d": W["d"], "heads": W["H"], "kv_positions": W["S"]},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} head-sparse attention steps (predict, top-k heads, attention), fp64 CPU oracle"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    if args.impl == "reference":
        if rank != 0:
            return
        n, el, cores = time_oracle(W, budget_s=1e9, max_steps=max(1, args.warmup))
        n, el, cores = time_oracle(W, budget_s=1e9, max_steps=max(1, args.steps))
        v = n / el / W.get("L", 1)
        print(json.dumps({
            "impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": n, "warmup": args.warmup, "ms_per_step": 1e3 * el / n, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "d": W["d"], "f": W["f"], "r": W["r"]},
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": f"{n} single-layer decode steps (predict, select, gathered FFN; layer 0) of the workload, fp64 CPU oracle" + (f", scaled to {W['L']} layers" if "L" in W else "")},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}))
        return
    init_dist(world)
    if W.get("attn"):
        res = run_attn(args, W, rank, world)
    elif "L" in W:
        res = run_stack(args, W, rank, world)
    elif "union" in W:
        res = run_union(args, W, rank, world)
    else:
        res, _ = run_ours(args, W, rank, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline and "union" in W:
        tok, el, cores = time_oracle_union(W, args.cpu_sample_s)
        res["cpu_baseline"] = {"value": tok / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": f"{tok} tokens of union steps (B={W['union']}) in {el:.1f} s, fp64 CPU oracle on {cores} threads"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline and W.get("attn"):
        n, el, cores = time_oracle_attn(W, args.cpu_sample_s)
        res["cpu_baseline"] = {"value": n / el, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": f"{n} head-sparse attention steps in {el:.1f} s, fp64 CPU oracle on {cores} threads"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        n, el, cores = time_oracle(W, args.cpu_sample_s)
        L = W.get("L", 1)
        res["cpu_baseline"] = {"value": n / el / L, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                               "sample": f"{n} single-layer decode steps (layer 0) in {el:.1f} s, fp64 CPU oracle on {cores} threads"
                                         + (f", scaled to {L} layers" if L > 1 else "")}
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
