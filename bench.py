"""Benchmark: sparse-FFN decode tokens/s at batch 1 on one GB300, with the HBM
roofline fraction of the dominant kernel and the CPU oracle as baseline.

Default workload: the LLaMA-70B-shaped ReLUfied SwiGLU stack (80 layers,
d=8192, f=28672, predictor r=1024, bf16 weights, fp32 accumulation, top-k at
15% = 4301 neurons per layer, look-ahead prediction on a second stream),
batch 1: the largest configuration that fits one GPU (113 GB of weights).  A
step is one token through every layer (cs_decode_stack): per layer the
predictor's two GEMVs, top-k selection, the gathered FFN and its fixed-order
reduction with the residual update.

Other workloads (--workload): single layers of the OPT-13B shape (top-k and
threshold at 5/10/20%, the exact mask, a hot prefix, a fitted predictor),
the tiny ReLU layer, the OPT-30B stack, the Falcon-40B batched union at
B = 1..32, head-sparse attention, and one SiLU SwiGLU layer.  Single-layer
steps rotate over NCOPY independent layer copies and distinct inputs, so a
copy's rows are evicted from L2 by the other copies before reuse.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME]

Exactly W untimed warm-up steps and K timed steps run.  Under torchrun
(N > 1) every rank runs the same workload on its own GPU (replicas: the path
has no exchange step); value = all ranks' steps / max time.  --impl reference
times the CPU oracle (the only reference this method has) on rank 0.
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
    "opt13b-thr5": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="threshold", share=0.05),
    "opt13b-thr10": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="threshold", share=0.10),
    "opt13b-thr20": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="threshold", share=0.20),
    # the exact mask {g > 0}: every gate row read (cs_exact_ffn), no predictor
    "opt13b-exact": dict(d=5120, f=20480, r=512, dt=1, glu=False, rho=0.10, mode="exact", share=0.10),
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


DEFAULT_WORKLOAD = "llama70b-stack-lookahead"


def parse():
    p = argparse.ArgumentParser()
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=None,
                   help="timed steps (default: 200 tokens for a stack, 20000 steps for a single layer)")
    p.add_argument("--warmup", type=int, default=None, help="untimed warm-up steps (at least 3; default 5)")
    p.add_argument("--impl", default="ours", choices=["ours", "reference"])
    p.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(WORKLOADS))
    p.add_argument("--cpu-sample-s", type=float, default=8.0,
                   help="seconds of oracle time per CPU-baseline leg (1 thread, then every core)")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--ncopy", type=int, default=None,
                   help="layer copies of a single-layer workload (default 8; fewer only for profiling)")
    p.add_argument("--layers", type=int, default=None,
                   help="layers of a stack workload (default: the workload's; fewer only for profiling)")
    a = p.parse_args()
    W = WORKLOADS[a.workload]
    if a.steps is None:
        a.steps = 200 if "L" in W else 2000 if "union" in W else 5000 if W.get("attn") else 20000
    if a.warmup is None:
        a.warmup = 5
    a.steps = max(1, a.steps)
    a.warmup = max(3, a.warmup)
    return a


class GraphSteps:
    """Runs exactly n steps of step(i) as replays of CUDA graphs of at most nb
    steps (one graph per distinct length, captured on first use; the step
    index restarts at 0 in every replay)."""

    def __init__(self, torch, stream, step, nb):
        self.torch, self.s, self.step, self.nb = torch, stream, step, nb
        self.g = {}

    def _graph(self, n):
        if n not in self.g:
            g = self.torch.cuda.CUDAGraph()
            with self.torch.cuda.stream(self.s):
                with self.torch.cuda.graph(g, stream=self.s):
                    for i in range(n):
                        self.step(i)
            self.g[n] = g
        return self.g[n]

    def prepare(self, n):
        """Capture the graphs that n steps replay (outside any timed region)."""
        q, r = divmod(n, self.nb)
        if q:
            self._graph(self.nb)
        if r:
            self._graph(r)

    def run(self, n):
        q, r = divmod(n, self.nb)
        with self.torch.cuda.stream(self.s):
            for _ in range(q):
                self._graph(self.nb).replay()
            if r:
                self._graph(r).replay()


def warm_and_time(torch, s, gs, args, world, dev, prime):
    """Warm-up of exactly args.warmup steps (the first three eager, through
    prime(i), so every kernel attribute is set before capture; the rest graph
    replays), then exactly args.steps timed steps bracketed by a barrier and a
    synchronize, with CUDA events on the launching stream and the SM clocks
    sampled meanwhile.  Returns (ms over ranks, clocks)."""
    with torch.cuda.stream(s):
        for i in range(3):
            prime(i)
    s.synchronize()
    gs.prepare(args.steps)
    gs.prepare(args.warmup - 3)
    gs.run(args.warmup - 3)
    s.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    clk = Clocks(dev)
    clk.start()
    time.sleep(0.3)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(s)
    gs.run(args.steps)
    e1.record(s)
    e1.synchronize()
    clocks = clk.stop()
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    return ms, clocks


def time_graph(torch, s, g, reps):
    """Average seconds of one replay of graph g (reps replays back to back)."""
    with torch.cuda.stream(s):
        for _ in range(2):
            g.replay()
    s.synchronize()
    f0, f1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    f0.record(s)
    with torch.cuda.stream(s):
        for _ in range(reps):
            g.replay()
    f1.record(s)
    f1.synchronize()
    return f0.elapsed_time(f1) / 1e3 / reps


def capture(torch, s, fn):
    g = torch.cuda.CUDAGraph()
    with torch.cuda.stream(s):
        with torch.cuda.graph(g, stream=s):
            fn()
    return g


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
                 "-lms", "50"], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
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
    """DRAM bytes per launch from a committed ncu summary, if every kernel
    source it was captured on is unchanged since; else None."""
    try:
        with open(os.path.join(ROOT, "profiles", "traffic.json")) as fh:
            t = json.load(fh)
        e = t[kernel][workload]
        for path, sha in e["sources"].items():
            if sha != src_sha(os.path.join(ROOT, path)):
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

def build_copies(W, torch, cs, synthdev, ncopy):
    import synth
    d, f, r, dt = W["d"], W["f"], W["r"], W["dt"]
    tdt = {0: torch.float32, 1: torch.float16, 2: torch.bfloat16}[dt]
    sd = 1 / math.sqrt(d)
    copies = []
    for l in range(ncopy):
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


FIT_KS = (0.05, 0.10, 0.15, 0.20, 0.30)


def fitted_quality(cs, torch, copy, d, f, r, n_tokens=32):
    """Mean recall and precision of a layer copy's predictor against the exact
    mask {g > 0}, both computed on the GPU, over held-out tokens, for top-k at
    each share in FIT_KS."""
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
    ks = [synth.ceil_k(f, q) for q in FIT_KS]
    rec = {k: [] for k in ks}
    prec = {k: [] for k in ks}
    sizes = []
    for x in synth.x_normal(7000, n_tokens, d):
        xt = torch.from_numpy(x[None]).cuda()
        cs.cs_exact_ffn(layer, xt, pre, ei, ec, y, ws)
        cs.cs_predict(pred, xt, sc, ws)
        torch.cuda.synchronize()
        E = ei.cpu().numpy()[:int(ec.item())]
        sizes.append(E.size)
        for k in ks:
            cs.cs_select(sc, cs.select_params(cs.CS_SEL_TOPK, k), pi, pc, ws=ws)
            torch.cuda.synchronize()
            P = pi.cpu().numpy()[0, :int(pc.item())]
            hit = np.intersect1d(P, E).size
            rec[k].append(hit / max(E.size, 1))
            prec[k].append(hit / max(P.size, 1))
    return [{"share": q, "k": k, "recall": float(np.mean(rec[k])), "precision": float(np.mean(prec[k]))}
            for q, k in zip(FIT_KS, ks)], float(np.mean(sizes))


def step_bytes(W, k):
    """Algorithmic bytes of one step (the per-unit accounting of the scope
    table): predictor weights, scores written and read, selected rows (+ index
    and bias), x and y.  Exact mode: every gate row, the pre-activations, then
    the selected rows' other matrices."""
    d, f, r = W["d"], W["f"], W["r"]
    hot = W.get("hot", 0)   # always-on prefix: not predicted, always gathered
    e = 4 if W["dt"] == 0 else 2
    m = 3 if W["glu"] else 2
    if W["mode"] == "exact":
        pre = e * f * d + 4 * (d + f)
        sel = 4 * f + 4 * k
        ffn = k * ((m - 1) * d * e + 4 + 4) + 4 * d * 2
        return pre + sel + ffn, ffn
    pred = e * (r * d + (f - hot) * r) + 4 * (d + r) * 2
    sel = 4 * (f - hot) + 4 * (hot + k)
    ffn = (hot + k) * (m * d * e + 4 + 4) + 4 * d * 2
    return pred + sel + ffn, ffn


NB = 200   # steps per captured graph


def run_ours(args, W, rank, world):
    import numpy as np
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
    ncopy = args.ncopy or NCOPY
    copies = build_copies(W, torch, cs, synthdev, ncopy)
    quality = None
    if W.get("fit"):
        # setup: fit every copy's up map, then measure the first copy's
        # recall / precision against the exact mask on held-out tokens
        Nc, lam = W["fit"]["N"], W["fit"]["lam_per_token"] * W["fit"]["N"]
        curve0, _ = fitted_quality(cs, torch, copies[0], d, f, r)
        for l, (layer, pred, _) in enumerate(copies):
            cs.cs_fit_predictor(layer, pred, torch.from_numpy(synth.x_normal(5000 + l, Nc, d)).cuda(), lam)
        curve, mean_exact = fitted_quality(cs, torch, copies[0], d, f, r)
        at = next(c for c in curve if c["k"] == k)
        quality = {"recall": at["recall"], "precision": at["precision"], "k": k,
                   "curve": curve, "random_up_map_curve": curve0, "exact_mask_mean_size": mean_exact,
                   "calibration_tokens": Nc, "lambda": lam, "held_out_tokens": 32,
                   "against": "exact mask {g > 0} (cs_exact_ffn) per held-out token"}
    X = torch.from_numpy(synth.x_normal(1000 + rank, NX, d)).cuda()
    s = torch.cuda.Stream()
    ws = cs.Workspace(d, f, r, stream=s)
    hot = W.get("hot", 0)
    exact = W["mode"] == "exact"
    scores = torch.empty((1, f - hot), device="cuda")
    pre = torch.empty(f, device="cuda")
    idx = torch.empty((1, f), dtype=torch.int32, device="cuda")
    cnt = torch.empty(1, dtype=torch.int32, device="cuda")
    Y = torch.empty((NX, d), device="cuda")
    tau = None
    if W["mode"] == "topk":
        params = cs.select_params(cs.CS_SEL_TOPK, k, hot=hot)
    elif exact:
        params = cs.select_params(cs.CS_SEL_EXACT, 0, 0.0)
    else:
        # threshold at the (1 - share) quantile of calibration scores (seed 1)
        layer0, pred0, _ = copies[0]
        Xc = torch.from_numpy(synth.x_normal(1, 256, d)).cuda()
        sc = torch.empty((256, f), device="cuda")
        cs.cs_predict(pred0, Xc, sc, cs.Workspace(d, f, r, 256))
        torch.cuda.synchronize()
        tau = float(torch.quantile(sc.flatten()[:: 7].float(), 1 - W["share"]))
        params = cs.select_params(cs.CS_SEL_THRESHOLD, 0, tau)

    def one_step(i):
        layer, pred, _ = copies[i % ncopy]
        x = X[i % NX: i % NX + 1]
        if exact:
            cs.cs_exact_ffn(layer, x, pre, idx[0], cnt, Y[i % NX], ws, stream=s)
            return
        cs.cs_predict(pred, x, scores, ws, stream=s)
        cs.cs_select(scores, params, idx, cnt, ws=ws, stream=s)
        cs.cs_sparse_ffn(layer, x, idx, cnt, Y[i % NX: i % NX + 1], ws, stream=s)

    torch.cuda.synchronize()
    gs = GraphSteps(torch, s, one_step, min(NB, args.steps))
    ms, clocks = warm_and_time(torch, s, gs, args, world, dev, one_step)
    K = args.steps
    assert cs.cs_get_device_error(ws, stream=s) == 0

    # roofline pass: the dominant call of the first NB steps alone, back to
    # back on the same stream over the same rows the timed steps gather
    # (index lists computed first), timed with CUDA events around graph
    # replays: the average duration of one cs_sparse_ffn launch (gather +
    # reduce); in exact mode of one cs_exact_ffn call (pre-activation GEMV,
    # selection, gather, reduce)
    nb = min(NB, 64) if exact else NB
    idx_all = torch.empty((nb, f), dtype=torch.int32, device="cuda")
    cnt_all = torch.empty(nb, dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        for i in range(nb):
            layer, pred, _ = copies[i % ncopy]
            if exact:
                cs.cs_exact_ffn(layer, X[i % NX: i % NX + 1], pre, idx_all[i], cnt_all[i: i + 1], Y[i % NX], ws,
                                stream=s)
                continue
            cs.cs_predict(pred, X[i % NX: i % NX + 1], scores, ws, stream=s)
            cs.cs_select(scores, params, idx_all[i: i + 1], cnt_all[i: i + 1], ws=ws, stream=s)
    s.synchronize()
    mean_count = float(cnt_all.float().mean().item())

    def ffn_calls():
        for i in range(nb):
            layer, _, _ = copies[i % ncopy]
            if exact:
                cs.cs_exact_ffn(layer, X[i % NX: i % NX + 1], pre, idx_all[i], cnt_all[i: i + 1], Y[i % NX], ws,
                                stream=s)
            else:
                cs.cs_sparse_ffn(layer, X[i % NX: i % NX + 1], idx_all[i], cnt_all[i: i + 1],
                                 Y[i % NX: i % NX + 1], ws, stream=s)

    with torch.cuda.stream(s):
        ffn_calls()
    s.synchronize()
    g2 = capture(torch, s, ffn_calls)
    ffn_avg_s = time_graph(torch, s, g2, 5) / nb

    # e2e: one cs_decode_layer call per token with x and y in pinned host
    # memory; the library copies x in and y out on the stream every step
    KE = min(K, 2000)
    xh = torch.from_numpy(synth.x_normal(2000 + rank, 64, d)).pin_memory()
    yh = torch.empty((64, d)).pin_memory()
    xslot, yslot = list(xh.unbind(0)), list(yh.unbind(0))   # the caller's 64 token slots

    def e2e_step(i):
        layer, pred, _ = copies[i % ncopy]
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

    kk = k if W["mode"] == "topk" else int(round(mean_count))
    total_b, ffn_b = step_bytes(W, kk)
    if exact:
        ffn_b = total_b   # the exact call moves the whole step's bytes
    hbm, src = peaks()
    step_s = ms / 1e3 / K
    ffn_gbs = ffn_b / ffn_avg_s / 1e9
    per_copy = (2 + W["glu"]) * f * d + r * d + (f - hot) * r
    res = {
        "metric": METRIC, "value": replica_value(K, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "d": d, "f": f, "r": None if exact else r,
                   "k": k if W["mode"] == "topk" else None,
                   **({"tau": tau, "mean_count": mean_count} if tau is not None else {}),
                   **({"mean_count": mean_count} if exact else {}),
                   "activation": "silu" if W.get("act", 0) else "relu", "gated": W["glu"],
                   **({"hot": hot, "active": hot + k, "layout": "frequency-sorted (cs_hot_order + cs_permute_rows)"}
                      if hot else {}),
                   "selection": W["mode"], "weights": {0: "f32", 1: "f16", 2: "bf16"}[W["dt"]],
                   "accumulate": "f32", "batch": 1, "global_batch": world, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {ncopy} layer copies ({ncopy * per_copy * (4 if W['dt'] == 0 else 2) / 1e9:.2f} GB) and {NX} inputs rotate; {ncopy - 1} other steps ({(ncopy - 1) * total_b / 1e6:.0f} MB) run between uses of a copy",
                   "step": ("cs_exact_ffn (pre-activation GEMV, exact-mask selection, gathered FFN)" if exact else
                            "cs_predict + cs_select + cs_sparse_ffn") + f", graphs of up to {NB} steps"},
        "clocks": clocks,
        **({"quality": quality} if quality else {}),
        "gpu_launches": (4 if exact else 5) * K,
        "roofline": {"bound": "hbm",
                     "kernel": "cs_exact_ffn (pre-activation GEMV + select + gather + reduce)" if exact
                     else "cs_sparse_ffn (gather + fixed-order reduce)",
                     "achieved": ffn_gbs, "peak": hbm, "unit": "GB/s", "frac": ffn_gbs / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                     "bytes_per_launch": ffn_b, "avg_launch_us": ffn_avg_s * 1e6,
                     "traffic": profile_traffic("cs_sparse_ffn", args.workload)},
        "step_roofline": {"bytes_per_step": total_b, "achieved": total_b / step_s / 1e9, "peak": hbm,
                          "frac": total_b / step_s / 1e9 / hbm, "unit": "GB/s"},
        "e2e": {"value": world * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * d,
                "d2h_bytes_per_step": 4 * d, "steps": KE,
                "how": "one cs_decode_layer call per token through the Python binding, x and y in pinned host memory (the call copies x in, replays the layer's graph of " + ("the exact step" if exact else "predict + select + gathered FFN") + ", copies y out); wall clock"},
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
    d, f, r = W["d"], W["f"], W["r"]
    L = args.layers or W["L"]
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
    SA = cs.StackArgs(layers, preds)
    NXS = 64
    X = torch.from_numpy(synth.x_normal(5000 + rank, NXS, d)).cuda()
    x = torch.empty(d, device="cuda")
    sm, sp = torch.cuda.Stream(), torch.cuda.Stream()
    ws = cs.Workspace(d, f, r, stream=sm)
    params = cs.select_params(cs.CS_SEL_TOPK, k)
    mode = cs.CS_STACK_LOOKAHEAD if W["stack"] == "lookahead" else cs.CS_STACK_SEQUENTIAL

    def step(i):
        x.copy_(X[i % NXS], non_blocking=True)
        cs.cs_decode_stack(SA, None, x, 0.1, params, mode, ws, s_main=sm, s_pred=sp)

    torch.cuda.synchronize()
    with torch.cuda.stream(sm):
        for i in range(args.warmup):
            step(i)
    sm.synchronize()
    K = args.steps
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
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1), world)
    barrier(world)
    assert cs.cs_get_device_error(ws, stream=sm) == 0

    # roofline pass: one traced token gives every layer's index list; then the
    # L gathered-FFN calls alone (each layer over its own list), back to back
    # on one stream, and the L predictor + selection calls alone, each timed
    # with CUDA events around graph replays
    tcnt = torch.empty(L, dtype=torch.int32, device="cuda")
    tidx = torch.empty((L, f), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(sm):
        x.copy_(X[0], non_blocking=True)
        cs.cs_decode_stack(SA, None, x, 0.1, params, mode, ws, s_main=sm, s_pred=sp, trace_count=tcnt,
                           trace_idx=tidx)
    sm.synchronize()
    XL = torch.from_numpy(synth.x_normal(5500 + rank, L, d)).cuda()
    YL = torch.empty((L, d), device="cuda")
    scores = torch.empty((1, f), device="cuda")
    i1 = torch.empty((1, f), dtype=torch.int32, device="cuda")
    c1 = torch.empty(1, dtype=torch.int32, device="cuda")

    def ffn_calls():
        for l in range(L):
            cs.cs_sparse_ffn(layers[l], XL[l:l + 1], tidx[l], tcnt[l:l + 1], YL[l:l + 1], ws, stream=sm)

    def pred_calls():
        for l in range(L):
            cs.cs_predict(preds[l], XL[l:l + 1], scores, ws, stream=sm)
            cs.cs_select(scores, params, i1, c1, ws=ws, stream=sm)

    with torch.cuda.stream(sm):
        ffn_calls()
        pred_calls()
    sm.synchronize()
    ffn_avg_s = time_graph(torch, sm, capture(torch, sm, ffn_calls), 3) / L
    pred_avg_s = time_graph(torch, sm, capture(torch, sm, pred_calls), 3) / L

    # e2e through the C ABI with a host buffer: per token the caller's pinned
    # x_0 goes in, cs_decode_stack copies it to the device, runs the stack and
    # copies x_L back into the same pinned buffer, and the caller waits for it
    # (an autoregressive loop reads every token's result before the next)
    KE = min(K, 50)
    xh = torch.from_numpy(synth.x_normal(6000 + rank, NXS, d))
    xio = torch.empty(d).pin_memory()

    def e2e_token(i):
        xio.copy_(xh[i % NXS])
        cs.cs_decode_stack(SA, None, xio, 0.1, params, mode, ws, s_main=sm, s_pred=sp)
        sm.synchronize()

    for i in range(3):
        e2e_token(i)
    t0 = time.perf_counter()
    for i in range(KE):
        e2e_token(i)
    e2e_s = time.perf_counter() - t0

    tot_b, ffn_b = step_bytes(W, k)
    pred_b = tot_b - ffn_b
    per_token = L * tot_b
    hbm, src = peaks()
    step_s = ms / 1e3 / K
    return {
        "metric": METRIC, "value": replica_value(K, world, ms), "unit": "tokens/s", "n_gpus": world,
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "layers": L, "d": d, "f": f, "r": r, "k": k, "selection": "topk",
                   "stack": W["stack"], "weights": {0: "f32", 1: "f16", 2: "bf16"}[W["dt"]],
                   "gated": W["glu"], "activation": "relu", "accumulate": "f32", "batch": 1, "global_batch": world,
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: the stack's weights ({L * ((2 + W['glu']) * f * d + r * d + f * r) * (4 if W['dt'] == 0 else 2) / 1e9:.0f} GB) are read once per token",
                   "step": "one token through every layer: cs_decode_stack (graph replay), fresh x per token"},
        "clocks": clocks,
        "gpu_launches": K * L * 5,
        "roofline": {"bound": "hbm",
                     "kernel": f"cs_sparse_ffn (gather + fixed-order reduce): the {L} layers' calls over their own index lists from one traced token, back to back",
                     "achieved": ffn_b / ffn_avg_s / 1e9, "peak": hbm, "unit": "GB/s",
                     "frac": ffn_b / ffn_avg_s / 1e9 / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                     "bytes_per_launch": ffn_b, "avg_launch_us": ffn_avg_s * 1e6,
                     "traffic": profile_traffic("cs_sparse_ffn", args.workload)},
        "step_roofline": {"bytes_per_step": per_token, "achieved": per_token / step_s / 1e9, "peak": hbm,
                          "frac": per_token / step_s / 1e9 / hbm, "unit": "GB/s"},
        "breakdown": {"per_layer_us_in_stack": step_s * 1e6 / L,
                      "ffn_call_us_alone": ffn_avg_s * 1e6, "ffn_bytes": ffn_b,
                      "predict_select_us_alone": pred_avg_s * 1e6, "predict_select_bytes": pred_b,
                      "serial_sum_us": (ffn_avg_s + pred_avg_s) * 1e6,
                      "note": "per layer: the token's time in the stack against the FFN call and the predictor + selection calls each timed alone (back to back, same stream)"},
        "e2e": {"value": world * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * d,
                "d2h_bytes_per_step": 4 * d, "steps": KE,
                "how": "per token: cs_decode_stack on the caller's pinned host x (the call copies x_0 in and x_L out), then a stream synchronize so the host holds x_L; wall clock"},
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
    NCU, NM = args.ncopy or 3, 32
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

    # the unions of the NM mask sets (setup: their mean size goes into the
    # byte count)
    with torch.cuda.stream(s):
        for m in range(NM):
            cs.cs_union_mask(masks[m], f, umask, uidx[m], ucnt[m: m + 1], ws, stream=s)
    s.synchronize()
    mean_u = float(ucnt.float().mean().item())
    nbu = min(64, args.steps)
    gs = GraphSteps(torch, s, step, nbu)
    ms, clocks = warm_and_time(torch, s, gs, args, world, dev, step)
    K = args.steps
    NB = 64
    assert cs.cs_get_device_error(ws, stream=s) == 0

    # roofline pass: the batched FFN calls alone (unions already computed)
    def ffn_calls():
        for i in range(NB):
            step(i, ffn_only=True)

    ffn_s = time_graph(torch, s, capture(torch, s, ffn_calls), 4) / NB

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
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "d": d, "f": f, "batch": B, "global_batch": world * B,
                   "weights": "bf16", "accumulate": "f32", "union_mean": mean_u, "union_density": mean_u / f,
                   "path": "tcgen05 gathered GEMM" if tc else "CUDA-core gathered GEMV",
                   "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {NCU} layer copies ({NCU * 2 * f * d * 2 / 1e9:.2f} GB) and {NM} mask sets rotate",
                   "step": "cs_union_mask + cs_sparse_ffn over B tokens, graphs of up to 64 steps"},
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


def oracle_inputs(W):
    """Layer 0 of the workload as oracle inputs (built once per process; the
    frequency-sorted layout by the oracle's own order when the workload has a
    hot prefix)."""
    import oracle
    import synth
    oracle.build()
    L, P = oracle_step_inputs(W)
    hot = W.get("hot", 0)
    if hot:
        perm = oracle.hot_order(synth.firing_probs(0, 0, W["f"], W["rho"]))
        pr = lambda a: oracle.permute_rows(a, perm) if a is not None else None
        L = oracle.Layer(L.d, L.f, L.dtype, pr(L.w_gate), pr(L.w_down_t), w_up=pr(L.w_up), bias=pr(L.bias),
                         act=L.act)
        P = oracle.Predictor(P.d, P.r, P.f - hot, P.dtype, P.p_down, oracle.permute_rows(P.p_up, perm[hot:]))
    return L, P


def time_oracle(W, budget_s, max_steps=None, inputs=None):
    """Time the oracle's single-layer decode step (predict, select, gathered
    FFN; in exact mode pre-activations, the exact mask, gathered FFN) on the
    host.  Returns (layer steps, seconds, threads)."""
    import numpy as np
    import oracle
    import synth
    L, P = inputs or oracle_inputs(W)
    k = synth.ceil_k(W["f"], W["share"])
    hot = W.get("hot", 0)
    X = synth.x_normal(3000, 64, W["d"])
    n, t0 = 0, time.perf_counter()
    tau = None
    while True:
        x = X[n % 64]
        if W["mode"] == "exact":
            sel = oracle.select_positive(oracle.preact(L, x).astype(np.float32))
        else:
            _, s = oracle.predict(P, x)
            s32 = s.astype(np.float32)
            if hot:
                sel = oracle.select_hot(s32, hot, oracle.SEL_TOPK, k=k)
            elif W["mode"] == "topk":
                sel = oracle.select_topk(s32, k)
            else:
                if tau is None:  # threshold at the (1 - share) quantile of the oracle's own scores
                    tau = np.float32(np.quantile(s32, 1 - W["share"]))
                sel = oracle.select_threshold(s32, tau)
        oracle.ffn(L, x, sel)
        n += 1
        el = time.perf_counter() - t0
        if el >= budget_s or (max_steps and n >= max_steps):
            break
    return n, el, oracle.threads()


def cpu_baseline(W, budget_s, timer, unit_per, what):
    """The oracle timed on the host at one thread and at every core, each leg
    about budget_s seconds.  timer(budget) -> (units, seconds, threads);
    unit_per converts units to tokens."""
    import oracle
    oracle.build()
    nproc = os.cpu_count() or 1
    oracle.set_threads(1)
    n1, el1, _ = timer(budget_s)
    oracle.set_threads(nproc)
    n, el, cores = timer(budget_s)
    return {"value": n / el / unit_per, "unit": "tokens/s", "cores": cores, "kind": "oracle",
            "sample": f"{n} {what} in {el:.1f} s, fp64 CPU oracle on {cores} threads",
            "single_thread": {"value": n1 / el1 / unit_per, "cores": 1,
                              "sample": f"{n1} {what} in {el1:.1f} s on 1 thread"}}


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

    torch.cuda.synchronize()
    gs = GraphSteps(torch, s, one_step, min(NB, args.steps))
    ms, clocks = warm_and_time(torch, s, gs, args, world, dev, one_step)
    K = args.steps
    assert cs.cs_get_device_error(ws, stream=s) == 0

    # roofline pass: the attention calls of the first NB steps alone (their
    # head lists computed above), back to back on the same stream
    def attn_call(i):
        layer, _, t = copies[i % NCOPY]
        j = i % NX
        cs.cs_sparse_attention(layer, X[j], idx_all[j], cnt_all[j:j + 1], t["k"], t["v"], Y[j], ws, stream=s)

    def attn_calls():
        for i in range(NB):
            attn_call(i)

    attn_avg_s = time_graph(torch, s, capture(torch, s, attn_calls), 5) / NB

    # e2e: one cs_decode_attention call per token on pinned host x and y
    KE = min(K, 2000)
    xh = torch.from_numpy(synth.x_normal(2000 + rank, 64, d)).pin_memory()
    yh = torch.empty((64, d)).pin_memory()

    def e2e_step(i):
        layer, pred, t = copies[i % NCOPY]
        cs.cs_decode_attention(layer, pred, xh[i % 64], yh[i % 64], params, t["k"], t["v"], ws, stream=s)

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
        "steps": K, "warmup": args.warmup, "ms_per_step": ms / K, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": {"workload": args.workload, "d": d, "heads": H, "d_head": dh, "kv_positions": S, "r": r,
                   "k_heads": k, "weights": {0: "f32", 1: "f16", 2: "bf16"}[W["dt"]], "accumulate": "f32",
                   "batch": 1, "global_batch": world, "parallelism": f"replicas x{world}",
                   "l2": f"inputs larger than L2: {NCOPY} layer copies ({NCOPY * 2 * (H * dh * d + H * S * dh) * (4 if W['dt'] == 0 else 2) / 1e9:.2f} GB) and {NX} inputs rotate",
                   "step": "cs_predict (one score per head) + cs_select (top-k heads) + cs_sparse_attention, graphs of up to 200 steps"},
        "clocks": clocks,
        "gpu_launches": 7 * K,   # predictor (2), select, query, attend, output, reduce
        "roofline": {"bound": "hbm", "kernel": "cs_sparse_attention (per-head attention + fixed-order reduce)",
                     "achieved": gbs, "peak": hbm, "unit": "GB/s", "frac": gbs / hbm,
                     "peak_source": f"{src} (MEASURED_PEAKS.json hbm_gbs)" if src == "measured" else "fallback",
                     "bytes_per_launch": attn_b, "avg_launch_us": attn_avg_s * 1e6,
                     "traffic": profile_traffic("cs_sparse_attention", args.workload)},
        "step_roofline": {"bytes_per_step": total_b, "achieved": total_b / step_s / 1e9, "peak": hbm,
                          "frac": total_b / step_s / 1e9 / hbm, "unit": "GB/s"},
        "e2e": {"value": world * KE / e2e_s, "unit": "tokens/s", "h2d_bytes_per_step": 4 * d,
                "d2h_bytes_per_step": 4 * d, "steps": KE,
                "how": "one cs_decode_attention call per token through the Python binding, x and y in pinned host memory (the call's graph reads x, runs predictor + head top-k + attention, writes y); wall clock"},
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
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(reference_arm(args, W)))
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
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        b = args.cpu_sample_s
        if "union" in W:
            res["cpu_baseline"] = cpu_baseline(W, b, lambda t: time_oracle_union(W, t), 1,
                                               f"tokens of union steps (B={W['union']})")
        elif W.get("attn"):
            res["cpu_baseline"] = cpu_baseline(W, b, lambda t: time_oracle_attn(W, t), 1,
                                               "head-sparse attention steps")
        else:
            inp = oracle_inputs(W)
            L = args.layers or W.get("L", 1)
            res["cpu_baseline"] = cpu_baseline(
                W, b, lambda t: time_oracle(W, t, inputs=inp), L,
                "single-layer decode steps (layer 0)" + (f", scaled to {L} layers (layer 0's time stands for "
                                                         "every layer's)" if L > 1 else ""))
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch
        torch.distributed.destroy_process_group()


def reference_arm(args, W):
    """The CPU oracle as it stands on the host's cores: exactly args.warmup
    untimed and then args.steps timed steps of the workload (a stack's step is
    one token: L oracle layer steps on layer 0's weights), stopping early, with
    the count reported, once a leg passes 90 s."""
    import oracle
    oracle.build()
    oracle.set_threads(os.cpu_count() or 1)
    L = args.layers or W.get("L", 1)
    cap = 90.0
    if "union" in W:
        B = W["union"]
        time_oracle_union(W, budget_s=cap, max_steps=args.warmup)
        tok, el, cores = time_oracle_union(W, budget_s=cap, max_steps=args.steps)
        steps, v, what = max(1, tok // B), tok / el, f"{tok} tokens of union steps (B={B})"
        cfg = {"workload": args.workload, "d": W["d"], "f": W["f"], "batch": B}
    elif W.get("attn"):
        time_oracle_attn(W, budget_s=cap, max_steps=args.warmup)
        steps, el, cores = time_oracle_attn(W, budget_s=cap, max_steps=args.steps)
        v, what = steps / el, f"{steps} head-sparse attention steps (predict, top-k heads, attention)"
        cfg = {"workload": args.workload, "d": W["d"], "heads": W["H"], "kv_positions": W["S"]}
    else:
        inp = oracle_inputs(W)
        time_oracle(W, budget_s=cap, max_steps=args.warmup * L, inputs=inp)
        n, el, cores = time_oracle(W, budget_s=cap, max_steps=args.steps * L, inputs=inp)
        steps, v = max(1, n // L), n / el / L
        what = f"{n} single-layer decode steps (predict, select, gathered FFN; layer 0)" + (
            f" = {n / L:.1f} tokens of {L} layers" if L > 1 else "")
        cfg = {"workload": args.workload, "d": W["d"], "f": W["f"], "r": W["r"], **({"layers": L} if L > 1 else {})}
    return {"impl": "reference", "metric": METRIC, "value": v, "unit": "tokens/s", "n_gpus": args.gpus,
            "steps": steps, "warmup": args.warmup, "ms_per_step": 1e3 / v, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": cfg,
            "cpu_baseline": {"value": v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": what + ", fp64 CPU oracle"},
            "e2e": {"value": v, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


if __name__ == "__main__":
    main()
