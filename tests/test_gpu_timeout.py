"""Bounded device waits: a withheld copy makes a wait run out; the kernel reports it and exits.

The test hook (gma_debug_withhold_first_load) stops the producer of the next bidirectional write
kernel from loading its first key tile.  The row warps waiting for that tile give up after the wait
limit (about a second), record GMA_ERR_TIMEOUT in the workspace error word, and every CTA leaves
through the common exit that releases its tensor memory.  Nothing traps or faults, so the context
stays usable: the next call on the same workspace runs normally and passes parity.
"""
import os
import subprocess
import sys
import time

import numpy as np
import pytest

from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, to_device

pytestmark = pytest.mark.gpu


def test_withheld_load_times_out_and_context_recovers():
    import torch
    from gaussian_mixture_sequence_gma_gb300 import gma
    inp = make_inputs(1, 2, 512, 64, dtype="bf16", seed=21)
    t = to_device(inp)
    args = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
    prob = gma.problem(1, 2, 512, 64, torch.bfloat16, 1e-6)
    ws = gma.alloc_workspace(prob, gma.OP_BIDIR, "cuda")
    gma.forward_bidir(*args, workspace=ws)
    assert gma.check_device_error(ws) == gma.GMA_OK
    gma.lib().gma_debug_withhold_first_load()
    t0 = time.time()
    gma.forward_bidir(*args, workspace=ws)
    assert gma.check_device_error(ws) == gma.GMA_ERR_TIMEOUT
    assert time.time() - t0 < 30
    O = gma.forward_bidir(*args, workspace=ws).float().cpu().numpy()
    assert gma.check_device_error(ws) == gma.GMA_OK
    ref = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6)
    assert np.isfinite(O).all()
    assert rel_err(O, ref) <= TOL["bf16"]


def test_short_wait_limit_reports_sooner():
    """With the limit set to 20 ms the withheld load is reported as GMA_ERR_TIMEOUT well within the 1 s
    default (a chain of a few bounded waits, each 20 ms), and restoring the default leaves the next call
    normal."""
    import torch
    from gaussian_mixture_sequence_gma_gb300 import gma
    inp = make_inputs(1, 2, 512, 64, dtype="bf16", seed=22)
    t = to_device(inp)
    args = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
    prob = gma.problem(1, 2, 512, 64, torch.bfloat16, 1e-6)
    ws = gma.alloc_workspace(prob, gma.OP_BIDIR, "cuda")
    gma.forward_bidir(*args, workspace=ws)
    assert gma.check_device_error(ws) == gma.GMA_OK
    gma.set_wait_limit_ns(20_000_000)
    try:
        gma.lib().gma_debug_withhold_first_load()
        torch.cuda.synchronize()
        t0 = time.time()
        gma.forward_bidir(*args, workspace=ws)
        assert gma.check_device_error(ws) == gma.GMA_ERR_TIMEOUT
        assert time.time() - t0 < 0.9
    finally:
        gma.set_wait_limit_ns(0)
    O = gma.forward_bidir(*args, workspace=ws).float().cpu().numpy()
    assert gma.check_device_error(ws) == gma.GMA_OK
    ref = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6)
    assert rel_err(O, ref) <= TOL["bf16"]


def test_fault_inject_environment_variable():
    """GMA_FAULT_INJECT arms the withheld load for the first bf16 bidirectional call of a fresh process:
    that call reports GMA_ERR_TIMEOUT (20 ms wait limit), the next one is normal and passes parity."""
    code = """
import numpy as np, torch
from gaussian_mixture_sequence_gma_gb300 import gma
from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs
from oracle import oracle as orc
from tests.helpers import rel_err, to_device
inp = make_inputs(1, 2, 512, 64, dtype="bf16", seed=23)
t = to_device(inp)
args = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
ws = gma.alloc_workspace(gma.problem(1, 2, 512, 64, torch.bfloat16, 1e-6), gma.OP_BIDIR, "cuda")
gma.forward_bidir(*args, workspace=ws)
first = gma.check_device_error(ws)
O = gma.forward_bidir(*args, workspace=ws).float().cpu().numpy()
second = gma.check_device_error(ws)
ref = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6)
print(first, second, rel_err(O, ref))
"""
    from gaussian_mixture_sequence_gma_gb300 import gma
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ, GMA_FAULT_INJECT="1", GMA_WAIT_LIMIT_MS="20")
    out = subprocess.run([sys.executable, "-c", code], cwd=root, env=env, capture_output=True, text=True, timeout=300)
    assert out.returncode == 0, out.stderr[-2000:]
    first, second, err = out.stdout.strip().splitlines()[-1].split()
    assert int(first) == gma.GMA_ERR_TIMEOUT
    assert int(second) == gma.GMA_OK
    assert float(err) <= TOL["bf16"]
