"""The seeded input generator: statistics, row independence and rounding."""
import math

import numpy as np
import torch

import synth


def test_normal_matrix_moments():
    m = synth.normal_matrix(0, 1, 256, 512, 1 / math.sqrt(512), synth.F32).astype(np.float64)
    assert abs(m.mean()) < 3e-3 / math.sqrt(512) * 10
    assert abs(m.std() * math.sqrt(512) - 1.0) < 0.01
    # Irwin-Hall(12) support is +-6 sigma
    assert np.abs(m).max() * math.sqrt(512) <= 6.0


def test_rows_do_not_depend_on_the_subset():
    full = synth.normal_matrix(3, 7, 50, 33, 0.2, synth.F16)
    rows = np.array([49, 0, 17, 17])
    sub = synth.normal_matrix(3, 7, 50, 33, 0.2, synth.F16, row_ids=rows)
    assert np.array_equal(full[rows], sub)


def test_streams_differ():
    a = synth.normal_matrix(0, 0, 4, 64, 1.0, synth.F32)
    b = synth.normal_matrix(0, 1, 4, 64, 1.0, synth.F32)
    c = synth.normal_matrix(1, 0, 4, 64, 1.0, synth.F32)
    assert not np.array_equal(a, b) and not np.array_equal(a, c)


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    v = (rng.standard_normal(100000) * np.exp(rng.uniform(-20, 20, 100000))).astype(np.float32)
    ours = synth.f32_to_bf16_bits(v)
    ref = torch.from_numpy(v).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ours, ref)


def test_zipf_profile():
    for f, rho in ((2048, 0.10), (20480, 0.10), (28672, 0.15), (32768, 0.10)):
        p, s = synth.zipf_probs_by_rank(f, rho)
        assert abs(p.mean() - rho) < 1e-9
        assert p.max() <= 0.9 and np.all(np.diff(p) <= 0)
    p = synth.firing_probs(0, 0, 2048, 0.1)
    assert sorted(p.tolist()) == sorted(synth.zipf_probs_by_rank(2048, 0.1)[0].tolist())


def test_bias_gives_firing_probability():
    b = synth.zipf_bias(0, 0, 1000, 0.1)
    p = synth.firing_probs(0, 0, 1000, 0.1)
    phi = 0.5 * (1 + np.vectorize(math.erf)(b.astype(np.float64) / math.sqrt(2)))
    np.testing.assert_allclose(phi, p, rtol=1e-6, atol=1e-7)


def test_mask_packing_roundtrip():
    rng = np.random.default_rng(1)
    for f in (1, 31, 32, 33, 100):
        act = rng.random(f) < 0.3
        assert np.array_equal(synth.bool_from_bits(synth.bits_from_bool(act), f), act)


def test_ceil_k():
    assert synth.ceil_k(2048, 0.10) == 205
    assert [synth.ceil_k(20480, r) for r in (0.05, 0.10, 0.20)] == [1024, 2048, 4096]
    assert synth.ceil_k(28672, 0.10) == 2868 and synth.ceil_k(28672, 0.15) == 4301


def test_c_twin_matches_numpy_definition():
    rng = np.random.default_rng(7)
    for dt in (synth.F32, synth.F16, synth.BF16):
        for rows, cols in ((1, 1), (37, 53), (8, 512)):
            a = synth.normal_matrix_np(11, 3, rows, cols, 0.7, dt)
            b = synth.normal_matrix(11, 3, rows, cols, 0.7, dt)
            assert np.array_equal(a.view(np.uint8), b.view(np.uint8))
        ids = rng.integers(0, 400, size=17)
        a = synth.normal_matrix_np(2, 9, 400, 72, 0.1, dt, row_ids=ids)
        b = synth.normal_matrix(2, 9, 400, 72, 0.1, dt, row_ids=ids, ld=80)
        assert np.array_equal(a.view(np.uint8), b[:, :72].copy().view(np.uint8))
        assert not b[:, 72:].view(np.uint8).any()
