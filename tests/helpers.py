"""Shared helpers for the GPU parity tests (marshalling and the error metric only)."""
import numpy as np

from gaussian_mixture_sequence_gma_gb300.inputs import bf16_bits

# Parity bar: max |O_gpu - O_ref| / max |O_ref| over the compared outputs.
TOL = {"f32": 1e-3, "bf16": 2e-2}


def to_device(inp, dev="cuda"):
    import torch
    out = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev) for k in ("mu", "sigma2", "log_pi")}
    for k in ("Q", "K", "V"):
        if inp["dtype"] == "bf16":
            out[k] = torch.from_numpy(bf16_bits(inp[k]).view(np.int16)).to(dev).view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(inp[k])).to(dev)
    return out


def rel_err(O, ref):
    O = np.asarray(O, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    return float(np.abs(O - ref).max() / np.abs(ref).max())


def sample_rows(N, n_random=192, seed=0):
    """Row indices for sampled parity: the ends, tile boundaries and random rows."""
    r = np.random.Generator(np.random.PCG64(seed))
    fixed = [0, 1, 2, N - 3, N - 2, N - 1]
    for b in (127, 128, 129, 255, 256, 4095, 4096, 16383, 16384, 65535, 65536):
        if b < N:
            fixed.append(b)
    rows = np.concatenate([np.array([x for x in fixed if 0 <= x < N], dtype=np.int64),
                           r.integers(0, N, size=min(n_random, N), dtype=np.int64)])
    return np.unique(rows)
