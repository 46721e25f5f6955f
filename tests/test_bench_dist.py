"""The benchmark's multi-rank (replica) path on CPU: two gloo ranks.

Under torchrun every rank runs the same workload on its own GPU with no
data-path collective; the ranks only agree on the slowest rank's elapsed time,
and the reported value is the units all ranks processed over that time.  These
tests run that agreement with the gloo backend in two spawned processes.
"""
import os
import socket
import subprocess
import sys

import pytest

torch = pytest.importorskip("torch")
import torch.multiprocessing as mp  # noqa: E402

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), CUDA_VISIBLE_DEVICES="")
    sys.path.insert(0, ROOT)
    import bench
    import torch.distributed as dist
    bench.init_dist(world)
    backend = dist.get_backend()
    ms = bench.max_over_ranks(1.5 + rank, world)     # rank 1 is the slower one
    bench.barrier(world)
    q.put((rank, backend, ms, bench.replica_value(100, world, ms)))
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_rank():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(2))
    for p in ps:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert [g[0] for g in got] == [0, 1]
    for rank, backend, ms, v in got:
        assert backend == "gloo"
        assert ms == 2.5
        assert v == pytest.approx(2 * 100 / 2.5e-3)


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench
    bench.init_dist(1)
    bench.barrier(1)
    assert bench.max_over_ranks(3.0, 1) == 3.0
    assert bench.replica_value(10, 1, 2.0) == pytest.approx(5000.0)


def test_reference_arm_on_a_nonzero_rank_prints_nothing():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--gpus", "2"], cwd=ROOT, env=env,
                       capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr
    assert r.stdout.strip() == ""


def test_algorithmic_bytes_match_the_per_unit_accounting():
    """The roofline numerators: predictor bytes e (r d + f r), and per selected
    neuron m d e weight bytes plus its id and bias (4 + 4), for the OPT-13B-
    shaped layer at k = 2048 (26.21 MB of predictor, 41.95 MB of rows)."""
    import bench
    W = bench.WORKLOADS["opt13b-topk10"]
    total, ffn = bench.step_bytes(W, 2048)
    assert ffn == 2048 * (2 * 5120 * 2 + 8) + 8 * 5120 == 42_000_384
    pred = 2 * (512 * 5120 + 20480 * 512)
    assert abs(pred - 26.21e6) < 0.01e6
    assert total == pred + 4 * (5120 + 512) * 2 + 4 * 20480 + 4 * 2048 + ffn
    # the hot layout predicts only the tail; the same 2048 rows are gathered
    th, fh = bench.step_bytes(bench.WORKLOADS["opt13b-hot5-topk5"], 1024)
    assert fh == ffn and total - th == 2 * 1024 * 512 + 4 * 1024
    # head-sparse attention: per head 2 d_head d + 2 S d_head elements
    Wa = bench.WORKLOADS["opt13b-attn-heads25"]
    ta, aa = bench.attn_bytes(Wa, 10)
    assert aa == 10 * 2 * (2 * 128 * 5120 + 2 * 2048 * 128) + 4 * 10 + 8 * 5120


def test_stack_and_exact_bytes_match_the_per_unit_accounting():
    """The LLaMA-70B-shaped stack moves 22.95 GB per token (80 layers of
    75.50 MB of predictor and 4301 gated rows of 3 d e bytes); the exact-mask
    step reads every gate row (f d e = 209.7 MB) plus the chosen down rows."""
    import bench
    import synth
    W = bench.WORKLOADS["llama70b-stack-lookahead"]
    k = synth.ceil_k(W["f"], W["share"])
    assert k == 4301
    total, ffn = bench.step_bytes(W, k)
    assert ffn == k * (3 * 8192 * 2 + 8) + 8 * 8192
    assert abs(2 * (1024 * 8192 + 28672 * 1024) - 75.50e6) < 0.01e6
    assert abs(80 * total - 22.95e9) < 0.03e9
    We = bench.WORKLOADS["opt13b-exact"]
    te, fe = bench.step_bytes(We, 2048)
    assert fe == 2048 * (5120 * 2 + 8) + 8 * 5120
    assert te == 2 * 20480 * 5120 + 4 * (5120 + 20480) + 4 * 20480 + 4 * 2048 + fe
    assert abs(te - 230.7e6) < 0.3e6
