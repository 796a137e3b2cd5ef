"""The allocation-free bidirectional entry point (gma_forward_bidir_static_ws).

Callers that cannot allocate device memory (no allocator on their execute path, or every byte
planned ahead) use this entry point; its scratch is an array held inside the library.  These tests
call it through the C ABI and compare it with the regular workspace entry point, on two calls in a
row with different inputs (the array keeps the previous call's contents, so stale state would show).
This file is collected last on purpose.
"""
import ctypes

import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs
from tests.helpers import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def gma():
    from gaussian_mixture_sequence_gma_gb300 import gma as g
    g.lib()
    return g


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_static_ws_matches_workspace_entry_point_twice(gma, dtype):
    import torch
    for call, (N, K, seed) in enumerate([(1000, 256, 31), (777, 48, 32)]):
        inp = make_inputs(2, 3, N, K, dtype=dtype, seed=seed)
        t = to_device(inp)
        args = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
        ref = gma.forward_bidir(*args, eps=1e-6).float()
        out = torch.full_like(t["Q"], float("nan"))
        prob = gma.problem(2, 3, N, K, t["Q"].dtype, 1e-6)
        s = gma.lib().gma_forward_bidir_static_ws(
            ctypes.byref(prob), t["Q"].data_ptr(), t["K"].data_ptr(), t["V"].data_ptr(), t["mu"].data_ptr(),
            t["sigma2"].data_ptr(), t["log_pi"].data_ptr(), out.data_ptr(), torch.cuda.current_stream().cuda_stream)
        assert s == gma.GMA_OK, "call %d: %s" % (call, gma.status_string(s))
        torch.cuda.synchronize()
        got = out.float()
        assert torch.isfinite(got).all()
        assert rel_err(got.cpu().numpy(), ref.cpu().numpy()) <= TOL[dtype], "call %d" % call


def test_static_ws_rejects_problems_beyond_capacity(gma):
    import torch
    cap = gma.static_ws_capacity()
    assert cap == 16 << 20
    # B*H*K large enough that the write-phase accumulator alone exceeds the array
    prob = gma.problem(64, 16, 128, 256, torch.bfloat16, 1e-6)
    assert gma.workspace_bytes(prob, gma.OP_BIDIR) > cap
    x = torch.zeros(64, 16, 128, 64, dtype=torch.bfloat16, device="cuda")
    mu = torch.zeros(16, 256, 64, device="cuda")
    s2 = torch.ones(16, 256, 64, device="cuda")
    lp = torch.zeros(16, 256, device="cuda")
    out = torch.empty_like(x)
    n0 = gma.launch_count()
    s = gma.lib().gma_forward_bidir_static_ws(ctypes.byref(prob), x.data_ptr(), x.data_ptr(), x.data_ptr(),
                                              mu.data_ptr(), s2.data_ptr(), lp.data_ptr(), out.data_ptr(), None)
    assert s == gma.GMA_ERR_WORKSPACE
    assert gma.launch_count() == n0


def test_static_ws_binding_wrapper(gma):
    inp = make_inputs(1, 2, 300, 17, dtype="bf16", seed=40)
    t = to_device(inp)
    args = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
    a = gma.forward_bidir_static_ws(*args).float().cpu().numpy()
    b = gma.forward_bidir(*args).float().cpu().numpy()
    assert rel_err(a, b) <= TOL["bf16"]


def test_static_ws_timeout_is_readable_without_allocation(gma):
    """A bounded wait that runs out inside the allocation-free call (the first key tile withheld by the
    test hook) leaves GMA_ERR_TIMEOUT in the library-held array's error word; the accessor reads it,
    and the next call clears it and computes normally."""
    import torch
    inp = make_inputs(1, 2, 512, 64, dtype="bf16", seed=41)
    t = to_device(inp)
    args = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
    ref = gma.forward_bidir(*args).float().cpu().numpy()
    gma.forward_bidir_static_ws(*args)
    assert gma.static_ws_check_error() == gma.GMA_OK
    gma.lib().gma_debug_withhold_first_load()
    gma.forward_bidir_static_ws(*args)
    assert gma.static_ws_check_error() == gma.GMA_ERR_TIMEOUT
    got = gma.forward_bidir_static_ws(*args).float().cpu().numpy()
    assert gma.static_ws_check_error() == gma.GMA_OK
    assert rel_err(got, ref) <= TOL["bf16"]
