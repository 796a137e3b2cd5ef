"""GPU parity of the cross-attention form (N queries reading the memory of Nk keys / values)
against the float64 oracle, through the C ABI (gma_forward_cross).

Bar: 1e-3 for float32 I/O, 2e-2 for bf16 I/O (max |O_gpu - O_ref| / max |O_ref|)."""
import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import make_cross_inputs
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, sample_rows, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gma():
    import torch  # noqa: F401
    from gaussian_mixture_sequence_gma_gb300 import gma as g
    g.lib()
    return g


def check(gma, inp, eps=1e-6, rows=None):
    t = to_device(inp)
    O = gma.forward_cross(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"], eps=eps).float().cpu().numpy()
    R = orc.forward_cross(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], eps, rows=rows)
    if rows is not None:
        O = O[:, :, rows]
    assert np.isfinite(O).all()
    err = rel_err(O, R)
    assert err <= TOL[inp["dtype"]], "max rel err %.3e" % err
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [3, 17, 256])
@pytest.mark.parametrize("N,Nk", [(300, 1000), (1000, 130), (129, 1), (1, 257)])
def test_cross_small(gma, dtype, K, N, Nk):
    check(gma, make_cross_inputs(2, 3, N, Nk, K, dtype=dtype, seed=N + 3 * Nk + K))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_cross_without_keys_is_zero(gma, dtype):
    import torch
    inp = make_cross_inputs(1, 2, 200, 0, 16, dtype=dtype, seed=4)
    t = to_device(inp)
    O = gma.forward_cross(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
    torch.cuda.synchronize()
    assert O.shape == (1, 2, 200, 64) and bool((O == 0).all())


def test_cross_bf16_B1H8_N8192_Nk65536_K256_sampled(gma):
    inp = make_cross_inputs(1, 8, 8192, 65536, 256, dtype="bf16", seed=11)
    check(gma, inp, rows=sample_rows(8192, seed=5))


def test_cross_equal_lengths_matches_bidir(gma):
    # N = Nk with the same key / value tensors is the bidirectional form
    inp = make_cross_inputs(2, 2, 700, 700, 64, dtype="bf16", seed=12)
    t = to_device(inp)
    Oc = gma.forward_cross(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]).float().cpu().numpy()
    Ob = gma.forward_bidir(t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"]).float().cpu().numpy()
    # the same kernels; only the order of the float32 atomic reduction can differ
    assert rel_err(Oc, Ob) <= 1e-2
