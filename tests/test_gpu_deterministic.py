"""The deterministic reduction mode (gma_set_deterministic) on the GPU: with it on, repeated calls on
the same inputs give bitwise-equal outputs, and the outputs still meet the oracle bar.

The write of the bidirectional form sums Gamma_K^T [V | 1] over all keys ("Latent memory routing",
linear-time form); by default the CTAs of a long key sequence add their partial states with atomics,
in whatever order they finish.  The shapes below make many write CTAs per head (hundreds of tiles of
keys), so an order-dependent sum would show.  Bars as for the forward and backward parity tests."""
import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import (bf16_bits, make_cross_inputs, make_inputs,
                                                        make_projected_inputs, round_bf16)
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, sample_rows, to_device

pytestmark = pytest.mark.gpu

REPEATS = 3


@pytest.fixture
def gma():
    import torch  # noqa: F401
    from gaussian_mixture_sequence_gma_gb300 import gma as g
    g.lib()
    g.set_deterministic(1)
    try:
        yield g
    finally:
        g.set_deterministic(-1)


def _same(outs):
    import torch
    for o in outs[1:]:
        if isinstance(o, tuple):
            for a, b in zip(outs[0], o):
                assert torch.equal(a, b)
        else:
            assert torch.equal(outs[0], o)


def _n(dtype):
    return 20000 if dtype == "bf16" else 3000  # >= 150 write tiles per head on either path


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_bidir_repeatable(gma, dtype):
    N = _n(dtype)
    inp = make_inputs(1, 2, N, 200, dtype=dtype, seed=71)
    t = to_device(inp)
    outs = [gma.forward_bidir(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]) for _ in range(REPEATS)]
    _same(outs)
    rows = sample_rows(N, n_random=64, seed=1)
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, rows=rows)
    assert rel_err(outs[0].float().cpu().numpy()[:, :, rows], R) <= TOL[dtype]
    gma.set_deterministic(0)
    O = gma.forward_bidir(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]).float().cpu().numpy()
    assert rel_err(O[:, :, rows], R) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_cross_repeatable(gma, dtype):
    inp = make_cross_inputs(2, 2, 300, _n(dtype), 64, dtype=dtype, seed=72)
    t = to_device(inp)
    outs = [gma.forward_cross(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]) for _ in range(REPEATS)]
    _same(outs)
    R = orc.forward_cross(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6)
    assert rel_err(outs[0].float().cpu().numpy(), R) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_state_repeatable(gma, dtype):
    inp = make_inputs(1, 3, _n(dtype), 17, dtype=dtype, seed=73)
    t = to_device(inp)
    outs = [gma.causal_state(t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]) for _ in range(REPEATS)]
    _same(outs)
    Vt, Z = orc.state(inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"])
    S = outs[0].cpu().numpy()
    assert rel_err(S[..., :64], Vt) <= TOL[dtype]
    assert rel_err(S[..., 64], Z) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("causal", [False, True])
def test_projected_repeatable(gma, dtype, causal):
    import torch
    inp = make_projected_inputs(2, 2, 1024, 64, dm=256, dtype=dtype, seed=74)
    t = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda() for k in ("mu", "sigma2", "log_pi", "bqkv")}
    for k in ("X", "Wqkv"):
        if dtype == "bf16":
            t[k] = torch.from_numpy(bf16_bits(inp[k]).view(np.int16)).cuda().view(torch.bfloat16)
        else:
            t[k] = torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
    outs = [gma.forward_projected(t["X"], t["Wqkv"], t["bqkv"], t["mu"], t["sigma2"], t["log_pi"], causal=causal)
            for _ in range(REPEATS)]
    _same(outs)
    rows = sample_rows(1024, n_random=48, seed=2)
    R = orc.forward_projected(inp["X"], inp["Wqkv"], inp["bqkv"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6,
                              causal=causal, dtype=dtype, rows=rows)
    assert rel_err(outs[0].float().cpu().numpy()[:, :, rows], R) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
def test_backward_repeatable(gma, dtype, causal):
    inp = make_inputs(2, 3, 700, 100, dtype=dtype, seed=75)
    G = np.random.Generator(np.random.PCG64(76)).standard_normal(inp["V"].shape).astype(np.float32)
    G = round_bf16(G) if dtype == "bf16" else G
    t = to_device(inp)
    gd = to_device(dict(Q=G, K=G, V=G, mu=inp["mu"], sigma2=inp["sigma2"], log_pi=inp["log_pi"], dtype=dtype))["Q"]
    f = gma.backward_causal if causal else gma.backward_bidir
    outs = [f(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], gd) for _ in range(REPEATS)]
    _same(outs)
    ref = orc.backward_bidir(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, G,
                             causal=causal)
    for name, a, b in zip(("dQ", "dK", "dV", "dmu", "dsigma2", "dlog_pi"), outs[0], ref):
        assert rel_err(a.float().cpu().numpy(), b) <= TOL[dtype], name


def test_workspace_sized_without_the_mode_is_refused(gma):
    """A workspace sized with the mode off is too small for the same call with it on."""
    import torch
    inp = make_inputs(1, 2, 4096, 64, dtype="bf16", seed=77)
    t = to_device(inp)
    gma.set_deterministic(0)
    prob = gma.problem(1, 2, 4096, 64, gma.GMA_BF16, 1e-6)
    ws = torch.empty(gma.workspace_bytes(prob, gma.OP_BIDIR), dtype=torch.uint8, device="cuda")
    gma.set_deterministic(1)
    with pytest.raises(gma.GmaError) as e:
        gma.forward_bidir(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], workspace=ws)
    assert e.value.status == gma.GMA_ERR_WORKSPACE


def test_static_workspace_entry_follows_the_mode(gma):
    """The allocation-free entry sizes its scratch with the mode too: a bf16 problem whose partials fit
    in its 16 MiB runs and repeats bit for bit."""
    inp = make_inputs(1, 2, 20000, 64, dtype="bf16", seed=78)
    t = to_device(inp)
    outs = [gma.forward_bidir_static_ws(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
            for _ in range(REPEATS)]
    _same(outs)
    rows = sample_rows(20000, n_random=48, seed=3)
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, rows=rows)
    assert rel_err(outs[0].float().cpu().numpy()[:, :, rows], R) <= TOL["bf16"]
