"""Python face of the float64 CPU oracle (``gma_oracle.c``).

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may call this module; the library path never
does, and this module imports nothing from the CUDA package.

What it computes follows the Gaussian Mixture Attention pages (gist.science
technical summaries, "Core mechanism" items 1-2 and "Variants and training"
item 3; fugumt.com English abstract):

* ``responsibilities``: gamma_ik = p(z=k | x_i) under a K-component diagonal
  GMM with priors pi_k (standard GMM posterior).
* ``forward(causal=False)``: Vt = Gamma_K^T V, Z = Gamma_K^T 1,
  O = Gamma_Q Vt / (Gamma_Q Z + eps).
* ``forward(causal=True)``: the same with inclusive prefix sums over keys.
* ``forward_cross``: the bidirectional form with N queries reading the memory
  written by Nk keys / values (gist.science summary, "Significance and claims",
  closing paragraph: cross-attention applications named as future work).
* ``forward_projected``: the Transformer-block form ("Variants and training":
  GMA as the sequence mixer of a Transformer language model): Q, K, V are the
  biased linear projections of the block input X, split into heads of 64,
  rounded to the I/O precision, then ``forward``.
* ``state``: Vt and Z alone.
* ``backward_bidir`` / ``backward_causal``: gradients of the bidirectional /
  causal forward with respect to Q, K, V, mu, sigma2 and log pi given dL/dO
  ("Variants and training" item 3: the components are learned end to end by
  backpropagation; the causal form through its prefix sums).

All inputs are converted to float64 here; the C code is plain sequential
float64 arithmetic per (batch, head) unit.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gma_oracle.c")
_BUILD_DIR = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD_DIR, "libgma_oracle.so")
_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile the C oracle with gcc (-O2, no fast-math) into ``out``."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + ".tmp%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fno-fast-math", "-ffp-contract=off",
           "-o", tmp, src, "-lm", "-lpthread"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _load(path: str | None = None):
    global _lib
    if path is not None:
        lib = ctypes.CDLL(path)
    else:
        if _lib is not None:
            return _lib
        lib = ctypes.CDLL(build())
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    ci, cl = ctypes.c_int, ctypes.c_int64
    lib.gma_oracle_responsibilities.argtypes = [ci, ci, ci, ci, ci, dp, dp, dp, dp, i64p, cl, dp, ci]
    lib.gma_oracle_responsibilities.restype = ci
    lib.gma_oracle_forward.argtypes = [ci, ci, ci, ci, ci, ci, ci, dp, dp, dp, dp, dp, dp, ctypes.c_double,
                                       i64p, cl, dp, ci]
    lib.gma_oracle_forward.restype = ci
    lib.gma_oracle_forward_cross.argtypes = [ci, ci, ci, ci, ci, ci, ci, dp, dp, dp, dp, dp, dp, ctypes.c_double,
                                             i64p, cl, dp, ci]
    lib.gma_oracle_forward_cross.restype = ci
    lib.gma_oracle_backward_bidir.argtypes = [ci, ci, ci, ci, ci, ci, dp, dp, dp, dp, dp, dp, ctypes.c_double, dp,
                                              dp, dp, dp, dp, dp, dp]
    lib.gma_oracle_backward_bidir.restype = ci
    lib.gma_oracle_backward_causal.argtypes = lib.gma_oracle_backward_bidir.argtypes
    lib.gma_oracle_backward_causal.restype = ci
    lib.gma_oracle_state.argtypes = [ci, ci, ci, ci, ci, ci, dp, dp, dp, dp, dp, dp, dp]
    lib.gma_oracle_state.restype = ci
    if path is None:
        _lib = lib
    return lib


def default_threads() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:  # pragma: no cover
        return os.cpu_count() or 1


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def _rows(rows, N):
    if rows is None:
        return None, 0, None
    r = np.unique(np.asarray(rows, dtype=np.int64))
    if r.size and (r[0] < 0 or r[-1] >= N):
        raise ValueError("row index out of range")
    return r, r.size, r.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def responsibilities(X, mu, sigma2, log_pi, rows=None, nthreads=None, lib=None):
    """Gamma [B,H,N|len(rows),K] for X [B,H,N,d] with per-head mu, sigma2 [H,K,d], log_pi [H,K]."""
    X, mu, sigma2, log_pi = _f64(X), _f64(mu), _f64(sigma2), _f64(log_pi)
    B, H, N, d = X.shape
    K = mu.shape[1]
    assert mu.shape == (H, K, d) and sigma2.shape == (H, K, d) and log_pi.shape == (H, K)
    r, nr, rp = _rows(rows, N)
    out = np.empty((B, H, nr if r is not None else N, K), dtype=np.float64)
    lib = lib or _load()
    lib.gma_oracle_responsibilities(B, H, N, d, K, _ptr(X), _ptr(mu), _ptr(sigma2), _ptr(log_pi), rp, nr,
                                    _ptr(out), nthreads or default_threads())
    return out


def forward(Q, Kx, V, mu, sigma2, log_pi, eps, causal=False, rows=None, nthreads=None, lib=None):
    """O [B,H,N|len(rows),dv].  ``rows`` (sorted unique indices) limits which outputs are formed."""
    Q, Kx, V = _f64(Q), _f64(Kx), _f64(V)
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    K = mu.shape[1]
    assert Kx.shape == Q.shape and V.shape[:3] == (B, H, N)
    assert mu.shape == (H, K, d) and sigma2.shape == (H, K, d) and log_pi.shape == (H, K)
    r, nr, rp = _rows(rows, N)
    out = np.empty((B, H, nr if r is not None else N, dv), dtype=np.float64)
    lib = lib or _load()
    lib.gma_oracle_forward(1 if causal else 0, B, H, N, d, dv, K, _ptr(Q), _ptr(Kx), _ptr(V), _ptr(mu),
                           _ptr(sigma2), _ptr(log_pi), float(eps), rp, nr, _ptr(out), nthreads or default_threads())
    return out


def forward_cross(Q, Kx, V, mu, sigma2, log_pi, eps, rows=None, nthreads=None, lib=None):
    """O [B,H,N|len(rows),dv] for queries Q [B,H,N,d] reading the memory of Kx [B,H,Nk,d], V [B,H,Nk,dv]."""
    Q, Kx, V = _f64(Q), _f64(Kx), _f64(V)
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    B, H, N, d = Q.shape
    Nk = Kx.shape[2]
    dv = V.shape[-1]
    K = mu.shape[1]
    assert Kx.shape == (B, H, Nk, d) and V.shape[:3] == (B, H, Nk)
    assert mu.shape == (H, K, d) and sigma2.shape == (H, K, d) and log_pi.shape == (H, K)
    r, nr, rp = _rows(rows, N)
    out = np.empty((B, H, nr if r is not None else N, dv), dtype=np.float64)
    lib = lib or _load()
    lib.gma_oracle_forward_cross(B, H, N, Nk, d, dv, K, _ptr(Q), _ptr(Kx), _ptr(V), _ptr(mu), _ptr(sigma2),
                                 _ptr(log_pi), float(eps), rp, nr, _ptr(out), nthreads or default_threads())
    return out


def state(Kx, V, mu, sigma2, log_pi, lib=None):
    """(Vt [B,H,K,dv], Z [B,H,K]) summed over all keys."""
    Kx, V = _f64(Kx), _f64(V)
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    B, H, N, d = Kx.shape
    dv = V.shape[-1]
    K = mu.shape[1]
    Vt = np.empty((B, H, K, dv), dtype=np.float64)
    Z = np.empty((B, H, K), dtype=np.float64)
    lib = lib or _load()
    lib.gma_oracle_state(B, H, N, d, dv, K, _ptr(Kx), _ptr(V), _ptr(mu), _ptr(sigma2), _ptr(log_pi), _ptr(Vt), _ptr(Z))
    return Vt, Z


def backward_bidir(Q, Kx, V, mu, sigma2, log_pi, eps, dO, lib=None, causal=False):
    """(dQ, dK, dV, dmu, dsigma2, dlog_pi) of the bidirectional (or causal) forward given dO [B,H,N,dv]."""
    Q, Kx, V, dO = _f64(Q), _f64(Kx), _f64(V), _f64(dO)
    mu, sigma2, log_pi = _f64(mu), _f64(sigma2), _f64(log_pi)
    B, H, N, d = Q.shape
    dv = V.shape[-1]
    K = mu.shape[1]
    assert Kx.shape == Q.shape and V.shape[:3] == (B, H, N) and dO.shape == (B, H, N, dv)
    dQ, dK, dV = np.empty_like(Q), np.empty_like(Kx), np.empty_like(V)
    dmu, dsigma2, dlog_pi = np.empty_like(mu), np.empty_like(sigma2), np.empty_like(log_pi)
    lib = lib or _load()
    fn = lib.gma_oracle_backward_causal if causal else lib.gma_oracle_backward_bidir
    fn(B, H, N, d, dv, K, _ptr(Q), _ptr(Kx), _ptr(V), _ptr(mu), _ptr(sigma2), _ptr(log_pi), float(eps), _ptr(dO),
       _ptr(dQ), _ptr(dK), _ptr(dV), _ptr(dmu), _ptr(dsigma2), _ptr(dlog_pi))
    return dQ, dK, dV, dmu, dsigma2, dlog_pi


def backward_causal(Q, Kx, V, mu, sigma2, log_pi, eps, dO, lib=None):
    """(dQ, dK, dV, dmu, dsigma2, dlog_pi) of the causal forward given dO [B,H,N,dv]."""
    return backward_bidir(Q, Kx, V, mu, sigma2, log_pi, eps, dO, lib=lib, causal=True)


def round_to_bf16(a) -> np.ndarray:
    """Nearest bfloat16 value of each element (ties to even), as float64.  The projection's output is
    rounded to the I/O precision before the forward, as a model in that precision stores it."""
    f = np.ascontiguousarray(np.asarray(a, dtype=np.float64).astype(np.float32))
    u = f.view(np.uint32).astype(np.uint64)
    u = ((u + 0x7FFF + ((u >> 16) & 1)) >> 16) << 16
    return u.astype(np.uint32).view(np.float32).astype(np.float64).reshape(f.shape)


def project_qkv(X, Wqkv, bqkv, H, dtype):
    """Q, K, V [B,H,N,64] from X [B,N,dm]: Y = X Wqkv + bqkv in float64 (Wqkv [dm, 3*H*64], column
    blocks Q | K | V, head h = columns 64h .. 64h+63 of a block), rounded to bf16 for dtype 'bf16'."""
    X = _f64(X)
    B, N, dm = X.shape
    Y = X.reshape(B * N, dm) @ _f64(Wqkv) + _f64(bqkv)[None, :]
    if dtype == "bf16":
        Y = round_to_bf16(Y)
    Y = Y.reshape(B, N, 3, H, 64)
    return tuple(np.ascontiguousarray(Y[:, :, w].transpose(0, 2, 1, 3)) for w in range(3))


def forward_projected(X, Wqkv, bqkv, mu, sigma2, log_pi, eps, causal=False, dtype="bf16", rows=None, nthreads=None,
                      lib=None):
    H = np.asarray(mu).shape[0]
    Q, Kx, V = project_qkv(X, Wqkv, bqkv, H, dtype)
    return forward(Q, Kx, V, mu, sigma2, log_pi, eps, causal=causal, rows=rows, nthreads=nthreads, lib=lib)
