"""Seeded synthetic inputs for the GMA forward pass.

This module is shared by the CUDA-path tests, the oracle tests and the
benchmark.  It only draws random numbers and applies the input recipe
(reparametrisation of the variances and priors the caller would do, bf16
rounding of the I/O tensors); it holds none of the method's arithmetic and
imports neither the CUDA binding nor the oracle.

Recipe (per workload): draws are made in the fixed order mu, sigma2-raw,
pi-raw, then Q, K, V (or, for the LM-shaped workload, token embeddings and
three random-init linear projections) from ``numpy.random.PCG64(seed)`` in
float32.  sigma2 = softplus(s * N(0,1)) + 1e-2 (the variance floor the
caller applies), log_pi = log_softmax(N(0,1)); both are kept in float32 and
handed unchanged to both sides.  For bf16 I/O, Q/K/V are rounded to bf16 with
round-to-nearest-even; the float32 arrays then hold exactly the bf16 values the
GPU sees.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass
class Workload:
    name: str
    causal: bool | None  # None: both forms
    dtype: str  # "f32" or "bf16"
    B: int
    H: int
    N: int
    K: int
    d: int = 64
    dv: int = 64
    sigma_raw_std: float = 1.0
    projection: bool = False
    seed: int = 0
    eps: float = 1e-6
    extra: dict = field(default_factory=dict)


def workloads() -> dict[str, Workload]:
    """The five benchmark workloads (the long-context sweep expanded per N)."""
    w = {
        "bidir_f32_B1H1N1024K16": Workload("bidir_f32_B1H1N1024K16", False, "f32", 1, 1, 1024, 16,
                                           sigma_raw_std=1.0, seed=0),
        "bidir_bf16_B4H8N4096K128": Workload("bidir_bf16_B4H8N4096K128", False, "bf16", 4, 8, 4096, 128,
                                             sigma_raw_std=0.5, seed=1),
        "causal_bf16_B4H8N4096K128": Workload("causal_bf16_B4H8N4096K128", True, "bf16", 4, 8, 4096, 128,
                                              sigma_raw_std=1.0, seed=2),
        "causal_lm_bf16_B8H12N2048K256": Workload("causal_lm_bf16_B8H12N2048K256", True, "bf16", 8, 12, 2048, 256,
                                                  sigma_raw_std=0.5, projection=True, seed=3),
    }
    for n in (4096, 16384, 65536, 131072):
        name = "sweep_bf16_B1H8N%dK256" % n
        w[name] = Workload(name, None, "bf16", 1, 8, n, 256, sigma_raw_std=1.0, seed=4)
    return w


def round_bf16(a: np.ndarray) -> np.ndarray:
    """float32 -> nearest bf16 value (ties to even), returned as float32."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    u = a.view(np.uint32).astype(np.uint64)
    u = (u + 0x7FFF + ((u >> 16) & 1)) >> 16
    return (u.astype(np.uint32) << 16).view(np.float32).reshape(a.shape)


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """Bit pattern (uint16) of float32 values that are already bf16-exact."""
    a = np.ascontiguousarray(a, dtype=np.float32)
    return (a.view(np.uint32) >> 16).astype(np.uint16)


def bf16_bits_to_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def _softplus(x: np.ndarray) -> np.ndarray:
    return np.logaddexp(np.float32(0.0), x).astype(np.float32)


def _log_softmax(x: np.ndarray) -> np.ndarray:
    x64 = x.astype(np.float64)
    m = x64.max(axis=-1, keepdims=True)
    return (x64 - m - np.log(np.exp(x64 - m).sum(axis=-1, keepdims=True))).astype(np.float32)


def make_params(rng: np.random.Generator, H: int, K: int, d: int, sigma_raw_std: float = 1.0,
                sigma_floor: float = 1e-2):
    mu = rng.standard_normal((H, K, d), dtype=np.float32)
    s_raw = rng.standard_normal((H, K, d), dtype=np.float32) * np.float32(sigma_raw_std)
    sigma2 = (_softplus(s_raw) + np.float32(sigma_floor)).astype(np.float32)
    pi_raw = rng.standard_normal((H, K), dtype=np.float32)
    log_pi = _log_softmax(pi_raw)
    return mu, sigma2, log_pi


def make_inputs(B: int, H: int, N: int, K: int, d: int = 64, dv: int = 64, dtype: str = "bf16", seed: int = 0,
                sigma_raw_std: float = 1.0, projection: bool = False, x_scale: float = 1.0,
                sigma_floor: float = 1e-2) -> dict:
    """Seeded problem.  Returns float32 arrays (bf16-exact when dtype == 'bf16')."""
    rng = np.random.Generator(np.random.PCG64(seed))
    mu, sigma2, log_pi = make_params(rng, H, K, d, sigma_raw_std, sigma_floor)
    if projection:
        dm = H * d
        E = rng.standard_normal((B, N, dm), dtype=np.float32)
        bound = np.float32(1.0 / np.sqrt(dm))
        outs = []
        for _ in range(3):
            W = rng.uniform(-bound, bound, size=(dm, dm)).astype(np.float32)
            b = rng.uniform(-bound, bound, size=(dm,)).astype(np.float32)
            Y = (E.reshape(B * N, dm) @ W.T + b).astype(np.float32)
            outs.append(np.ascontiguousarray(Y.reshape(B, N, H, d).transpose(0, 2, 1, 3)))
        Q, Kx, V = outs
    else:
        Q = rng.standard_normal((B, H, N, d), dtype=np.float32)
        Kx = rng.standard_normal((B, H, N, d), dtype=np.float32)
        V = rng.standard_normal((B, H, N, dv), dtype=np.float32)
    if x_scale != 1.0:
        Q = Q * np.float32(x_scale)
        Kx = Kx * np.float32(x_scale)
    if dtype == "bf16":
        Q, Kx, V = round_bf16(Q), round_bf16(Kx), round_bf16(V)
    elif dtype != "f32":
        raise ValueError(dtype)
    return dict(Q=Q, K=Kx, V=V, mu=mu, sigma2=sigma2, log_pi=log_pi, dtype=dtype)


def make_projected_inputs(B: int, H: int, N: int, K: int, dm: int | None = None, dtype: str = "bf16", seed: int = 0,
                          sigma_raw_std: float = 0.5) -> dict:
    """Seeded Transformer-block problem: block input X [B,N,dm] ~ N(0,1) and one [dm, 3*H*64] weight
    (column blocks Q | K | V) with a [3*H*64] bias, both U(-1/sqrt(dm), 1/sqrt(dm)) like a default
    linear-layer init, plus the mixture parameters.  X and Wqkv are bf16-exact for dtype 'bf16'."""
    dm = dm or H * 64
    rng = np.random.Generator(np.random.PCG64(seed))
    mu, sigma2, log_pi = make_params(rng, H, K, 64, sigma_raw_std)
    X = rng.standard_normal((B, N, dm), dtype=np.float32)
    bound = np.float32(1.0 / np.sqrt(dm))
    Wqkv = rng.uniform(-bound, bound, size=(dm, 3 * H * 64)).astype(np.float32)
    bqkv = rng.uniform(-bound, bound, size=(3 * H * 64,)).astype(np.float32)
    if dtype == "bf16":
        X, Wqkv = round_bf16(X), round_bf16(Wqkv)
    elif dtype != "f32":
        raise ValueError(dtype)
    return dict(X=X, Wqkv=Wqkv, bqkv=bqkv, mu=mu, sigma2=sigma2, log_pi=log_pi, dtype=dtype)


def make_cross_inputs(B: int, H: int, N: int, Nk: int, K: int, dtype: str = "bf16", seed: int = 0,
                      sigma_raw_std: float = 1.0) -> dict:
    """Seeded cross-attention problem: N queries, Nk keys / values, one shared set of parameters.
    Queries and parameters come from make_inputs(seed); keys and values from a second stream."""
    q = make_inputs(B, H, N, K, dtype=dtype, seed=seed, sigma_raw_std=sigma_raw_std)
    kv = make_inputs(B, H, Nk, K, dtype=dtype, seed=seed + 7919, sigma_raw_std=sigma_raw_std)
    return dict(Q=q["Q"], K=kv["K"], V=kv["V"], mu=q["mu"], sigma2=q["sigma2"], log_pi=q["log_pi"], dtype=dtype)


def make_workload(w: Workload, N: int | None = None) -> dict:
    return make_inputs(w.B, w.H, N or w.N, w.K, w.d, w.dv, w.dtype, w.seed, w.sigma_raw_std, w.projection)
