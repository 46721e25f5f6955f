"""Seeded synthetic inputs for the contextual-sparsity FFN step.

This module is the one place that makes inputs.  It holds none of the
method's arithmetic (no predictor, no selection, no FFN): it only draws
weights, biases, activations and masks from seeds.  Both the CPU oracle and
the CUDA library consume what it makes; neither imports the other.

Generator definition (host here, device twin in ``synth/synth.cu``; the two
must agree bit for bit):

* ``mix64`` is the SplitMix64 output function (Steele, Lea and Flood,
  "Fast splittable pseudorandom number generators", OOPSLA 2014, with the
  13th variant of Stafford's mixer constants, as in Vigna's splitmix64).
* A tensor has a 64-bit key ``K = mix64(seed * G + mix64(tensor_id))`` with
  ``G = 0x9E3779B97F4A7C15``.  Element ``n`` (row-major logical index
  ``row * cols + col``, independent of any row padding) takes three draws
  ``r_i = mix64(K + (3n + i + 1) * G)``, ``i = 0, 1, 2``.
* The twelve 16-bit fields of the three draws are summed: ``S`` in
  ``[0, 12 * 65535]``.  ``t = S - 393210`` is an Irwin-Hall(12) variate with
  mean 0 and standard deviation ~65536, so ``t * 2**-16`` is approximately
  N(0, 1) (support +-6).
* The stored value is ``float32(t) * scale`` in IEEE fp32 (round to nearest
  even), with ``scale = float32(std * 2**-16)``, then rounded to the storage
  type (fp16 or bf16, round to nearest even).  Every step is exact integer
  work or one correctly rounded IEEE operation, so host and device agree.

The activation profile follows the power-law ("hot" and "cold" neurons)
description on the page "Contextual Sparsity and Activation Predictors"
(section "Static locality: hot and cold neurons"): neuron ``j`` fires with
probability ``p_j = min(0.9, 0.5 * (rank_j / s) ** -0.8)``, where ``rank_j``
is a seeded random permutation of ``1..f`` and ``s`` is found by bisection
so that the mean of ``p`` is the target active share ``rho``.  The bias that
makes ``P(w_j . x + b_j > 0) = p_j`` for ``x ~ N(0, I)`` is
``b_j = sigma_j * PhiInv(p_j)`` with ``sigma_j = 1``, the expected norm of a
row drawn N(0, 1/d).
"""
from __future__ import annotations

import math
import statistics

import numpy as np

GAMMA = np.uint64(0x9E3779B97F4A7C15)
_M1 = np.uint64(0xBF58476D1CE4E5B9)
_M2 = np.uint64(0x94D049BB133111EB)
IRWIN_HALL_MEAN = 393210  # 12 * 65535 / 2

# tensor ids: layer l owns ids 8*l .. 8*l+7
W_GATE, W_UP, W_DOWN_T, P_DOWN, P_UP = 0, 1, 2, 3, 4

F32, F16, BF16 = 0, 1, 2
DTYPE_NAMES = {F32: "f32", F16: "f16", BF16: "bf16"}
DTYPE_BYTES = {F32: 4, F16: 2, BF16: 2}


def tensor_id(layer: int, which: int) -> int:
    return 8 * int(layer) + int(which)


def mix64(z: np.ndarray) -> np.ndarray:
    """SplitMix64 output mixer on a uint64 array (wrapping arithmetic)."""
    z = np.asarray(z, dtype=np.uint64)
    with np.errstate(over="ignore"):
        z = (z ^ (z >> np.uint64(30))) * _M1
        z = (z ^ (z >> np.uint64(27))) * _M2
    return z ^ (z >> np.uint64(31))


def stream_key(seed: int, tid: int) -> np.uint64:
    s = np.array([seed], dtype=np.uint64)
    t = mix64(np.array([tid], dtype=np.uint64))
    with np.errstate(over="ignore"):
        return mix64(s * GAMMA + t)[0]


def weight_scale(std: float) -> np.float32:
    """fp32 multiplier applied to the integer Irwin-Hall variate."""
    return np.float32(std * 2.0 ** -16)


def irwin_hall_t(key: np.uint64, n: np.ndarray) -> np.ndarray:
    """Centred Irwin-Hall(12) integer variate for logical element ids n."""
    n = np.asarray(n, dtype=np.uint64)
    s = np.zeros(n.shape, dtype=np.int64)
    mask = np.uint64(0xFFFF)
    with np.errstate(over="ignore"):
        base = n * np.uint64(3)
        for i in range(3):
            r = mix64(key + (base + np.uint64(i + 1)) * GAMMA)
            for q in range(4):
                s += ((r >> np.uint64(16 * q)) & mask).astype(np.int64)
    return (s - IRWIN_HALL_MEAN).astype(np.int32)


def f32_to_bf16_bits(a: np.ndarray) -> np.ndarray:
    """Round fp32 to bf16 (nearest even) and return the raw 16-bit patterns.

    Inputs here are finite; NaN handling is not needed by the generator.
    """
    u = np.ascontiguousarray(a, dtype=np.float32).view(np.uint32).astype(np.uint64)
    bias = np.uint64(0x7FFF) + ((u >> np.uint64(16)) & np.uint64(1))
    return ((u + bias) >> np.uint64(16)).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << np.uint32(16)).view(np.float32)


def to_storage(v32: np.ndarray, dtype: int) -> np.ndarray:
    """fp32 values -> storage array (float32, float16, or uint16 bf16 bits)."""
    if dtype == F32:
        return v32.astype(np.float32)
    if dtype == F16:
        return v32.astype(np.float16)
    if dtype == BF16:
        return f32_to_bf16_bits(v32)
    raise ValueError(f"unknown dtype {dtype}")


def storage_to_f64(a: np.ndarray, dtype: int) -> np.ndarray:
    if dtype == BF16:
        return bf16_bits_to_f32(a).astype(np.float64)
    return np.asarray(a).astype(np.float64)


def normal_matrix_np(seed: int, tid: int, rows: int, cols: int, std: float, dtype: int,
                     row_ids=None, chunk: int = 1 << 22) -> np.ndarray:
    """Rows of a [rows, cols] N(0, std^2) tensor in storage dtype (numpy, the
    readable definition; ``normal_matrix`` is the fast C twin).

    ``row_ids`` selects a subset of rows (default all); the values of a row do
    not depend on which other rows are drawn.
    """
    key = stream_key(seed, tid)
    scale = weight_scale(std)
    if row_ids is None:
        row_ids = np.arange(rows, dtype=np.int64)
    row_ids = np.asarray(row_ids, dtype=np.int64)
    if row_ids.size and (row_ids.min() < 0 or row_ids.max() >= rows):
        raise IndexError("row id out of range")
    out = np.empty((row_ids.size, cols), dtype=np.float32)
    rows_per_chunk = max(1, chunk // max(cols, 1))
    col = np.arange(cols, dtype=np.uint64)
    for r0 in range(0, row_ids.size, rows_per_chunk):
        rr = row_ids[r0:r0 + rows_per_chunk].astype(np.uint64)
        n = (rr[:, None] * np.uint64(cols) + col[None, :]).reshape(-1)
        t = irwin_hall_t(key, n)
        out[r0:r0 + rr.size] = (t.astype(np.float32) * scale).reshape(rr.size, cols)
    return to_storage(out, dtype)


# ----------------------------------------------------------------------------
# activation profile and bias
# ----------------------------------------------------------------------------

def zipf_probs_by_rank(f: int, rho: float, cap: float = 0.9, amp: float = 0.5,
                       alpha: float = 0.8) -> tuple[np.ndarray, float]:
    """p(rank) = min(cap, amp * (rank / s) ** -alpha), rank = 1..f, mean(p) = rho.

    Returns (p indexed by rank-1, s).  s is found by bisection on log s; the
    mean grows monotonically with s.
    """
    rank = np.arange(1, f + 1, dtype=np.float64)

    def mean_p(s):
        return float(np.minimum(cap, amp * (rank / s) ** (-alpha)).mean())

    lo, hi = 1e-6, float(f) * 1e6
    if not (mean_p(lo) < rho < mean_p(hi)):
        raise ValueError("rho out of reach of the profile")
    for _ in range(200):
        mid = math.sqrt(lo * hi)
        if mean_p(mid) < rho:
            lo = mid
        else:
            hi = mid
    s = math.sqrt(lo * hi)
    return np.minimum(cap, amp * (rank / s) ** (-alpha)), s


def neuron_rank(seed: int, layer: int, f: int) -> np.ndarray:
    """rank_j in 1..f for each neuron j (a seeded random permutation)."""
    rng = np.random.default_rng([int(seed), int(layer), 0x5EED])
    return rng.permutation(f).astype(np.int64) + 1


def firing_probs(seed: int, layer: int, f: int, rho: float) -> np.ndarray:
    p_by_rank, _ = zipf_probs_by_rank(f, rho)
    return p_by_rank[neuron_rank(seed, layer, f) - 1]


def zipf_bias(seed: int, layer: int, f: int, rho: float) -> np.ndarray:
    """fp32 bias b_j = PhiInv(p_j) so that P(w_j . x + b_j > 0) = p_j."""
    p_by_rank, _ = zipf_probs_by_rank(f, rho)
    inv = statistics.NormalDist().inv_cdf
    b_by_rank = np.array([inv(float(p)) for p in p_by_rank], dtype=np.float64)
    return b_by_rank[neuron_rank(seed, layer, f) - 1].astype(np.float32)


# ----------------------------------------------------------------------------
# activations, score vectors and masks
# ----------------------------------------------------------------------------

def x_normal(seed: int, B: int, d: int) -> np.ndarray:
    """[B, d] fp32 activations drawn N(0, 1)."""
    rng = np.random.default_rng([int(seed), 0xA11CE])
    return rng.standard_normal((B, d)).astype(np.float32)


def score_vector(seed: int, f: int, ties: int = 0, specials: bool = False,
                 quantize: float | None = None) -> np.ndarray:
    """A fp32 score vector for selection tests.

    ``ties`` copies that many random values onto other positions (equal keys);
    ``quantize`` rounds every score to a multiple of it (many ties);
    ``specials`` plants +-0, +-inf and NaN.
    """
    rng = np.random.default_rng([int(seed), 0x5C0E])
    s = rng.standard_normal(f).astype(np.float32)
    if quantize:
        s = (np.round(s / quantize) * quantize).astype(np.float32)
    if ties and f > 1:
        src = rng.integers(0, f, size=ties)
        dst = rng.integers(0, f, size=ties)
        s[dst] = s[src]
    if specials and f >= 8:
        pos = rng.choice(f, size=min(f, 8), replace=False)
        vals = np.array([0.0, -0.0, np.inf, -np.inf, np.nan, np.nan, 0.0, -0.0],
                        dtype=np.float32)
        s[pos] = vals[: pos.size]
    return s


def union_masks(seed: int, B: int, f: int, rho: float, tail: float = 0.03) -> np.ndarray:
    """Per-token active masks [B, ceil(f/32)] u32: Bernoulli(p_j) on the shared
    power-law profile, united with a uniform random subset of ceil(tail*f)."""
    p = firing_probs(seed, 0, f, rho)
    words = (f + 31) // 32
    out = np.zeros((B, words), dtype=np.uint32)
    for b in range(B):
        rng = np.random.default_rng([int(seed), b, 0x0A5C])
        act = rng.random(f) < p
        extra = rng.permutation(f)[: int(math.ceil(tail * f))]
        act[extra] = True
        out[b] = bits_from_bool(act)
    return out


def bits_from_bool(act: np.ndarray) -> np.ndarray:
    """Pack a bool vector into u32 words, bit j%32 of word j//32."""
    f = act.size
    words = (f + 31) // 32
    padded = np.zeros(words * 32, dtype=np.uint64)
    padded[:f] = act.astype(np.uint64)
    w = padded.reshape(words, 32) << np.arange(32, dtype=np.uint64)[None, :]
    return w.sum(axis=1).astype(np.uint32)


def bool_from_bits(words: np.ndarray, f: int) -> np.ndarray:
    w = np.asarray(words, dtype=np.uint32).astype(np.uint64)
    bits = (w[:, None] >> np.arange(32, dtype=np.uint64)[None, :]) & np.uint64(1)
    return bits.reshape(-1)[:f].astype(bool)


def ceil_k(f: int, frac: float) -> int:
    """k for an active share: ceil(frac * f) (recall-first rounding)."""
    return int(math.ceil(frac * f - 1e-9))


# ----------------------------------------------------------------------------
# fast host twin (synth_host.c, gcc + OpenMP)
# ----------------------------------------------------------------------------
import ctypes as _C
import os as _os
import subprocess as _sp
import threading as _th

_HERE = _os.path.dirname(_os.path.abspath(__file__))
_HOST_SRC = _os.path.join(_HERE, "synth_host.c")
_HOST_LIB = _os.path.join(_HERE, "_build", "libsynthhost.so")
_host_lock = _th.Lock()
_host = None


def build_host(force: bool = False) -> str:
    _os.makedirs(_os.path.dirname(_HOST_LIB), exist_ok=True)
    if (not force and _os.path.exists(_HOST_LIB)
            and _os.path.getmtime(_HOST_LIB) >= _os.path.getmtime(_HOST_SRC)):
        return _HOST_LIB
    tmp = _HOST_LIB + f".tmp{_os.getpid()}"
    _sp.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-ffp-contract=off",
             _HOST_SRC, "-o", tmp], check=True)
    _os.replace(tmp, _HOST_LIB)
    return _HOST_LIB


def _host_lib():
    global _host
    with _host_lock:
        if _host is None:
            L = _C.CDLL(build_host())
            L.synth_host_fill.argtypes = [_C.c_void_p, _C.c_int, _C.c_void_p, _C.c_int64,
                                          _C.c_int64, _C.c_int64, _C.c_uint64, _C.c_float]
            L.synth_host_fill.restype = None
            L.synth_host_key.argtypes = [_C.c_uint64, _C.c_uint64]
            L.synth_host_key.restype = _C.c_uint64
            _host = L
    return _host


_NP_DT = {F32: np.float32, F16: np.float16, BF16: np.uint16}


def normal_matrix(seed: int, tid: int, rows: int, cols: int, std: float, dtype: int,
                  row_ids=None, ld: int | None = None) -> np.ndarray:
    """Same values as ``normal_matrix_np`` (C twin): rows of a [rows, cols]
    N(0, std^2) tensor, optionally padded with zero columns to ``ld``."""
    ld = cols if ld is None else int(ld)
    if row_ids is None:
        ids = None
        n = rows
    else:
        ids = np.ascontiguousarray(row_ids, dtype=np.int64)
        if ids.size and (ids.min() < 0 or ids.max() >= rows):
            raise IndexError("row id out of range")
        n = ids.size
    out = np.empty((n, ld), dtype=_NP_DT[dtype])
    key = int(stream_key(seed, tid))
    _host_lib().synth_host_fill(out.ctypes.data, int(dtype), None if ids is None else ids.ctypes.data,
                                n, int(cols), ld, key, float(weight_scale(std)))
    return out
