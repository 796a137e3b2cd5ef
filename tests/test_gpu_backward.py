"""GPU parity of the backward passes (gma_backward_bidir, gma_backward_causal) against the float64
oracle's gradients, which are pinned by finite differences of the forward oracle.

Bar per gradient tensor: max |g_gpu - g_ref| / max |g_ref| <= 1e-3 (float32 I/O) or 2e-2 (bf16 I/O:
inputs and dQ, dK, dV in bf16, float32 arithmetic)."""
import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs, round_bf16
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu

NAMES = ("dQ", "dK", "dV", "dmu", "dsigma2", "dlog_pi")


@pytest.fixture(scope="module")
def gma():
    import torch  # noqa: F401
    from gaussian_mixture_sequence_gma_gb300 import gma as g
    g.lib()
    return g


def _dO(inp, seed):
    G = np.random.Generator(np.random.PCG64(seed)).standard_normal(inp["V"].shape).astype(np.float32)
    return round_bf16(G) if inp["dtype"] == "bf16" else G


def check(gma, inp, eps=1e-6, seed=0, causal=False):
    import torch
    G = _dO(inp, seed)
    t = to_device(inp)
    gd = to_device(dict(Q=G, K=G, V=G, mu=inp["mu"], sigma2=inp["sigma2"], log_pi=inp["log_pi"], dtype=inp["dtype"]))["Q"]
    f = gma.backward_causal if causal else gma.backward_bidir
    got = f(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], gd, eps=eps)
    torch.cuda.synchronize()
    ref = orc.backward_bidir(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], eps, G,
                             causal=causal)
    errs = {}
    for name, a, b in zip(NAMES, got, ref):
        a = a.float().cpu().numpy()
        assert a.shape == b.shape, name
        assert np.isfinite(a).all(), name
        errs[name] = rel_err(a, b)
    bad = {k: v for k, v in errs.items() if v > TOL[inp["dtype"]]}
    assert not bad, "max rel err above the bar: %s" % bad
    return errs


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [3, 17, 64, 100, 128])
def test_backward_small(gma, dtype, K):
    check(gma, make_inputs(2, 3, 150, K, dtype=dtype, seed=200 + K), seed=K)


@pytest.mark.parametrize("N", [1, 31, 33, 300])
def test_backward_lengths_f32(gma, N):
    check(gma, make_inputs(1, 2, N, 16, dtype="f32", seed=300 + N), seed=N)


def test_backward_large_eps(gma):
    check(gma, make_inputs(1, 2, 200, 8, dtype="f32", seed=7), eps=3.0, seed=7)


def test_backward_bf16_B1H2N2048K256(gma):
    check(gma, make_inputs(1, 2, 2048, 256, dtype="bf16", seed=9), seed=9)


def test_backward_zero_length(gma):
    import torch
    inp = make_inputs(1, 2, 0, 16, dtype="f32", seed=1)
    t = to_device(inp)
    gd = torch.empty((1, 2, 0, 64), device="cuda")
    got = gma.backward_bidir(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], gd)
    torch.cuda.synchronize()
    for g in got[3:]:
        assert bool((g == 0).all())


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [3, 17, 64, 100, 128])
def test_causal_backward_small(gma, dtype, K):
    check(gma, make_inputs(2, 3, 150, K, dtype=dtype, seed=400 + K), seed=K, causal=True)


@pytest.mark.parametrize("N", [1, 31, 33, 300, 1000])
def test_causal_backward_lengths_f32(gma, N):
    # N = 1000 spreads over several segments (suffix scan across segments).  With one key, O = v g / (g + eps)
    # and every gradient but dV is proportional to eps: eps = 0.3 keeps it above float32 resolution.
    check(gma, make_inputs(1, 2, N, 16, dtype="f32", seed=500 + N), eps=0.3 if N == 1 else 1e-6, seed=N, causal=True)


def test_causal_backward_bf16_B1H2N2048K256(gma):
    check(gma, make_inputs(1, 2, 2048, 256, dtype="bf16", seed=19), seed=19, causal=True)


@pytest.mark.parametrize("causal", [False, True])
def test_backward_full_size_one_head(gma, causal):
    """The bench's backward workload (B=4 H=8 N=4096 K=128, bf16), launched whole as the bench times it;
    the oracle checks head 3 over every batch entry, so that head's dmu, dsigma2 and dlog_pi are
    complete sums and dQ, dK, dV are checked for all 4 x 4096 of its rows."""
    import torch
    from gaussian_mixture_sequence_gma_gb300.inputs import make_workload, workloads
    w = workloads()["bidir_bf16_B4H8N4096K128"]
    inp = make_workload(w)
    G = _dO(inp, 77)
    t = to_device(inp)
    gd = to_device(dict(Q=G, K=G, V=G, mu=inp["mu"], sigma2=inp["sigma2"], log_pi=inp["log_pi"], dtype="bf16"))["Q"]
    f = gma.backward_causal if causal else gma.backward_bidir
    got = f(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], gd, eps=w.eps)
    torch.cuda.synchronize()
    h = 3
    ref = orc.backward_bidir(inp["Q"][:, h:h + 1], inp["K"][:, h:h + 1], inp["V"][:, h:h + 1], inp["mu"][h:h + 1],
                             inp["sigma2"][h:h + 1], inp["log_pi"][h:h + 1], w.eps, G[:, h:h + 1], causal=causal)
    errs = {}
    for name, a, b in zip(NAMES, got, ref):
        a = a.float().cpu().numpy()
        a = a[:, h:h + 1] if name in ("dQ", "dK", "dV") else a[h:h + 1]
        assert a.shape == b.shape, name
        assert np.isfinite(a).all(), name
        errs[name] = rel_err(a, b)
    bad = {k: v for k, v in errs.items() if v > TOL["bf16"]}
    assert not bad, "max rel err above the bar: %s" % bad
