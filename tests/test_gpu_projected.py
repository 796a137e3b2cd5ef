"""GPU parity of the Transformer-block form (Q / K / V projection + GMA forward) against the oracle.

The oracle projects in float64, rounds Q, K, V to the I/O precision and runs its forward; the GPU
projects with float32 accumulation.  Bar as for the forward: max |O_gpu - O_ref| / max |O_ref| <= 1e-3
(float32 I/O) or 2e-2 (bf16 I/O).
"""
import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import bf16_bits, make_projected_inputs
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gma():
    import torch  # noqa: F401
    from gaussian_mixture_sequence_gma_gb300 import gma as g
    g.lib()
    return g


def dev(inp):
    import torch
    out = {k: torch.from_numpy(np.ascontiguousarray(inp[k])).cuda() for k in ("mu", "sigma2", "log_pi", "bqkv")}
    for k in ("X", "Wqkv"):
        if inp["dtype"] == "bf16":
            out[k] = torch.from_numpy(bf16_bits(inp[k]).view(np.int16)).cuda().view(torch.bfloat16)
        else:
            out[k] = torch.from_numpy(np.ascontiguousarray(inp[k])).cuda()
    return out


def check(gma, inp, causal, rows=None, eps=1e-6):
    t = dev(inp)
    O = gma.forward_projected(t["X"], t["Wqkv"], t["bqkv"], t["mu"], t["sigma2"], t["log_pi"], causal=causal,
                              eps=eps).float().cpu().numpy()
    R = orc.forward_projected(inp["X"], inp["Wqkv"], inp["bqkv"], inp["mu"], inp["sigma2"], inp["log_pi"], eps,
                              causal=causal, dtype=inp["dtype"], rows=rows)
    if rows is not None:
        O = O[:, :, rows]
    assert np.isfinite(O).all()
    err = rel_err(O, R)
    assert err <= TOL[inp["dtype"]], "max rel err %.3e" % err
    return err


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dm", [96, 128])
def test_projected_ragged(gma, dtype, causal, dm):
    inp = make_projected_inputs(2, 2, 300, 17, dm=dm, dtype=dtype, seed=11 + dm)
    check(gma, inp, causal)


@pytest.mark.parametrize("causal", [False, True])
def test_projected_lm_block_B8H12N2048K256_sampled(gma, causal):
    # the language-model block shape: d_model 768, 12 heads of 64, K = 256
    inp = make_projected_inputs(8, 12, 2048, 256, dtype="bf16", seed=3)
    check(gma, inp, causal, rows=sample_rows(2048, n_random=48, seed=5))


def test_projected_equals_forward_on_its_projection(gma):
    # the projected call and the plain forward on the same Q, K, V (taken from the projection the
    # library itself produced in its workspace) agree exactly: the two calls share the forward kernels
    import torch
    inp = make_projected_inputs(1, 2, 512, 64, dtype="bf16", seed=21)
    t = dev(inp)
    prob = gma.problem(1, 2, 512, 64, torch.bfloat16)
    ws = gma.alloc_workspace(prob, gma.OP_PROJECTED_CAUSAL, "cuda")
    O1 = gma.forward_projected(t["X"], t["Wqkv"], t["bqkv"], t["mu"], t["sigma2"], t["log_pi"], causal=True,
                               workspace=ws)
    Y = (t["X"].float().reshape(512, -1) @ t["Wqkv"].float() + t["bqkv"]).reshape(1, 512, 3, 2, 64)
    qkv = [Y[:, :, w].permute(0, 2, 1, 3).contiguous().to(torch.bfloat16) for w in range(3)]
    O2 = gma.forward_causal(qkv[0], qkv[1], qkv[2], t["mu"], t["sigma2"], t["log_pi"])
    # torch's GEMM may round a few projected values differently from cuBLASLt's: compare with the bar
    assert rel_err(O1.float().cpu().numpy(), O2.float().cpu().numpy()) <= TOL["bf16"]


@pytest.mark.parametrize("B,H,N,dm", [(1, 1, 5, 8), (3, 1, 129, 1000), (1, 3, 257, 40)])
def test_projected_edge_shapes_bf16(gma, B, H, N, dm):
    """Edges of the bf16 projection GEMM's tiling: dm below one K block (8) and far above it with a tail
    (1000), one head (192 output columns, a partial column tile), row counts that are not multiples of
    the 256-row tile and tiles that cross a batch boundary."""
    inp = make_projected_inputs(B, H, N, 16, dm=dm, dtype="bf16", seed=90 + dm)
    check(gma, inp, True)
