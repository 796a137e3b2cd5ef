"""GPU parity of the causal state and decode step (the recurrent form of the prefix sums) against
the float64 oracle, through the C ABI (gma_causal_state, gma_causal_decode).

A decode step's outputs must equal the causal forward outputs of the same positions over the whole
sequence seen so far; the state must equal the latent memory / normaliser of every key seen.
Bar: 1e-3 for float32 I/O, 2e-2 for bf16 I/O (max |x_gpu - x_ref| / max |x_ref|)."""
import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gma():
    import torch  # noqa: F401
    from gaussian_mixture_sequence_gma_gb300 import gma as g
    g.lib()
    return g


def _slice(t, a, b):
    return {k: (v[:, :, a:b].contiguous() if k in ("Q", "K", "V") else v) for k, v in t.items()}


def _ref_state(inp, n):
    Vt, Z = orc.state(inp["K"][:, :, :n], inp["V"][:, :, :n], inp["mu"], inp["sigma2"], inp["log_pi"])
    return np.concatenate([Vt, Z[..., None]], axis=-1)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [17, 256])
def test_state_matches_oracle(gma, dtype, K):
    inp = make_inputs(2, 3, 900, K, dtype=dtype, seed=30 + K)
    t = to_device(inp)
    S = gma.causal_state(t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]).cpu().numpy()
    ref = _ref_state(inp, 900)
    assert S.shape == ref.shape
    assert rel_err(S, ref) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [17, 256])
def test_decode_continues_the_prompt(gma, dtype, K):
    N0, T = 700, 9
    inp = make_inputs(2, 3, N0 + T, K, dtype=dtype, seed=40 + K)
    t = to_device(inp)
    state = gma.causal_state(t["K"][:, :, :N0].contiguous(), t["V"][:, :, :N0].contiguous(), t["mu"], t["sigma2"],
                             t["log_pi"])
    outs = []
    for s in range(T):  # one token per call, state resident between calls
        d = _slice(t, N0 + s, N0 + s + 1)
        outs.append(gma.causal_decode(d["Q"], d["K"], d["V"], t["mu"], t["sigma2"], t["log_pi"], state))
    O = np.concatenate([o.float().cpu().numpy() for o in outs], axis=2)
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, causal=True,
                    rows=np.arange(N0, N0 + T))
    assert np.isfinite(O).all()
    assert rel_err(O, R) <= TOL[dtype]
    # the state now holds every key seen
    assert rel_err(state.cpu().numpy(), _ref_state(inp, N0 + T)) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 5, 64, 200])
def test_decode_from_empty_state_is_causal_forward(gma, dtype, K):
    # K <= 16 runs 64 threads (one per output column) with idle component slots; K = 200 leaves part
    # of the last warps idle
    import torch
    inp = make_inputs(1, 4, 37, K, dtype=dtype, seed=50 + K)
    t = to_device(inp)
    state = torch.zeros((1, 4, K, 65), dtype=torch.float32, device="cuda")
    O = gma.causal_decode(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], state).float().cpu().numpy()
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, causal=True)
    assert rel_err(O, R) <= TOL[dtype]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_one_call_equals_token_by_token(gma, dtype):
    # the same float32 arithmetic in the same order: bit-identical outputs and state
    inp = make_inputs(2, 2, 320, 32, dtype=dtype, seed=60)
    t = to_device(inp)
    p = _slice(t, 0, 300)
    s1 = gma.causal_state(p["K"], p["V"], t["mu"], t["sigma2"], t["log_pi"])
    s2 = s1.clone()
    d = _slice(t, 300, 320)
    O1 = gma.causal_decode(d["Q"], d["K"], d["V"], t["mu"], t["sigma2"], t["log_pi"], s1)
    O2 = [gma.causal_decode(_slice(t, i, i + 1)["Q"], _slice(t, i, i + 1)["K"], _slice(t, i, i + 1)["V"], t["mu"],
                            t["sigma2"], t["log_pi"], s2) for i in range(300, 320)]
    import torch
    assert torch.equal(O1, torch.cat(O2, dim=2))
    assert torch.equal(s1, s2)


def test_empty_prompt_state_is_zero(gma):
    import torch
    inp = make_inputs(1, 2, 0, 16, dtype="bf16", seed=70)
    t = to_device(inp)
    S = gma.causal_state(t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"],
                         state=torch.full((1, 2, 16, 65), float("nan"), device="cuda"))
    assert bool((S == 0).all())


def test_decode_lm_shape_bf16_B8H12K256(gma):
    inp = make_inputs(8, 12, 2048 + 4, 256, dtype="bf16", seed=3, sigma_raw_std=0.5, projection=True)
    t = to_device(inp)
    p = _slice(t, 0, 2048)
    state = gma.causal_state(p["K"], p["V"], t["mu"], t["sigma2"], t["log_pi"])
    d = _slice(t, 2048, 2052)
    O = gma.causal_decode(d["Q"], d["K"], d["V"], t["mu"], t["sigma2"], t["log_pi"], state).float().cpu().numpy()
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, causal=True,
                    rows=np.arange(2048, 2052))
    assert rel_err(O, R) <= TOL["bf16"]


def test_decode_bench_shape(gma):
    """The bench's decode shape (B=8, H=12, K=256, bf16, one token per call, 96 CTAs) after a 300-token
    prompt, three steps: every head's outputs and final state against the oracle."""
    N0, T = 300, 3
    inp = make_inputs(8, 12, N0 + T, 256, dtype="bf16", seed=90, sigma_raw_std=0.5)
    t = to_device(inp)
    state = gma.causal_state(t["K"][:, :, :N0].contiguous(), t["V"][:, :, :N0].contiguous(), t["mu"], t["sigma2"],
                             t["log_pi"])
    outs = []
    for s in range(T):
        d = _slice(t, N0 + s, N0 + s + 1)
        outs.append(gma.causal_decode(d["Q"], d["K"], d["V"], t["mu"], t["sigma2"], t["log_pi"], state))
    O = np.concatenate([o.float().cpu().numpy() for o in outs], axis=2)
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, causal=True,
                    rows=np.arange(N0, N0 + T))
    assert np.isfinite(O).all()
    assert rel_err(O, R) <= TOL["bf16"]
    assert rel_err(state.cpu().numpy(), _ref_state(inp, N0 + T)) <= TOL["bf16"]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [17, 256])
def test_prepared_decode_is_bit_identical(gma, dtype, K):
    """gma_decode_prepare + gma_causal_decode_prepared give the outputs and state of gma_causal_decode
    bit for bit (the same fold, the same decode kernel), step after step with the parameters folded
    once, and a multi-token prepared call equals the single-token ones."""
    import torch
    N0, T = 300, 6
    inp = make_inputs(2, 3, N0 + T, K, dtype=dtype, seed=80 + K)
    t = to_device(inp)
    p = _slice(t, 0, N0)
    s_ref = gma.causal_state(p["K"], p["V"], t["mu"], t["sigma2"], t["log_pi"])
    s_pre, s_multi = s_ref.clone(), s_ref.clone()
    ws = gma.decode_prepare(t["mu"], t["sigma2"], t["log_pi"], dtype=t["Q"].dtype)
    for i in range(N0, N0 + T):
        d = _slice(t, i, i + 1)
        o_ref = gma.causal_decode(d["Q"], d["K"], d["V"], t["mu"], t["sigma2"], t["log_pi"], s_ref)
        o_pre = gma.causal_decode_prepared(d["Q"], d["K"], d["V"], s_pre, ws)
        assert torch.equal(o_ref, o_pre)
        assert torch.equal(s_ref, s_pre)
    d = _slice(t, N0, N0 + T)
    o_multi = gma.causal_decode_prepared(d["Q"], d["K"], d["V"], s_multi, ws)
    assert torch.equal(s_multi, s_ref)
    R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6, causal=True,
                    rows=np.arange(N0, N0 + T))
    assert rel_err(o_multi.float().cpu().numpy(), R) <= TOL[dtype]
