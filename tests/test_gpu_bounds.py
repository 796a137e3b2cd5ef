"""The bounds-check debug build (libgma_checked.so) on the GPU.

In that build every computed global-memory index of the forward kernels is compared with the extent
the host planned for its buffer (workspace sections, outputs, the float32 path's input rows); a failed
check skips the access and is recorded instead of trapping.  A child process loads the checked build,
first makes one check fail on purpose (a kernel that touches no memory) to show the record works, then
runs every forward entry point over ragged lengths, K classes and both dtypes, with and without the
deterministic reduction mode, and requires an empty record and oracle parity."""
import json
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = r"""
import json, numpy as np, torch
from gaussian_mixture_sequence_gma_gb300 import gma
from gaussian_mixture_sequence_gma_gb300.inputs import make_inputs, make_cross_inputs, make_projected_inputs, bf16_bits
from oracle import oracle as orc
from tests.helpers import TOL, rel_err, sample_rows, to_device

L = gma.lib()
assert gma.lib_path().endswith("libgma_checked.so")
res = {}
L.gma_debug_bounds_clear()
assert L.gma_debug_bounds_selftest(None) == 0
torch.cuda.synchronize()
res["selftest"] = gma.bounds_record()
L.gma_debug_bounds_clear()
worst = 0.0
for det in (0, 1):
    gma.set_deterministic(det)
    for dtype in ("bf16", "f32"):
        for (B, H, N, K) in ((1, 2, 1, 1), (2, 3, 127, 17), (1, 2, 129, 64), (2, 1, 300, 100), (1, 3, 4097, 256),
                             (3, 2, 2000, 129)):
            inp = make_inputs(B, H, N, K, dtype=dtype, seed=N + K)
            t = to_device(inp)
            a = (t["Q"], t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
            rows = sample_rows(N, n_random=16, seed=1)
            for causal in (False, True):
                f = gma.forward_causal if causal else gma.forward_bidir
                O = f(*a).float().cpu().numpy()[:, :, rows]
                R = orc.forward(inp["Q"], inp["K"], inp["V"], inp["mu"], inp["sigma2"], inp["log_pi"], 1e-6,
                                causal=causal, rows=rows)
                worst = max(worst, rel_err(O, R) / TOL[dtype])
            gma.causal_state(t["K"], t["V"], t["mu"], t["sigma2"], t["log_pi"])
            gma.responsibilities(t["Q"], t["mu"], t["sigma2"], t["log_pi"])
        ci = make_cross_inputs(2, 2, 77, 1500, 40, dtype=dtype, seed=5)
        ct = to_device(ci)
        gma.forward_cross(ct["Q"], ct["K"], ct["V"], ct["mu"], ct["sigma2"], ct["log_pi"])
        pi = make_projected_inputs(2, 2, 300, 64, dm=128, dtype=dtype, seed=6)
        pt = {k: torch.from_numpy(np.ascontiguousarray(pi[k])).cuda() for k in ("mu", "sigma2", "log_pi", "bqkv")}
        for k in ("X", "Wqkv"):
            pt[k] = (torch.from_numpy(bf16_bits(pi[k]).view(np.int16)).cuda().view(torch.bfloat16) if dtype == "bf16"
                     else torch.from_numpy(np.ascontiguousarray(pi[k])).cuda())
        for causal in (False, True):
            gma.forward_projected(pt["X"], pt["Wqkv"], pt["bqkv"], pt["mu"], pt["sigma2"], pt["log_pi"], causal=causal)
gma.set_deterministic(-1)
torch.cuda.synchronize()
res["record"] = gma.bounds_record()
res["worst_over_tol"] = worst
print(json.dumps(res))
"""


def test_checked_build_records_nothing_on_every_forward():
    from gaussian_mixture_sequence_gma_gb300 import build as gbuild
    gbuild.build(checked=True)
    env = dict(os.environ, GMA_LIBRARY="checked")
    out = subprocess.run([sys.executable, "-c", CHILD], cwd=ROOT, env=env, capture_output=True, text=True,
                         timeout=900)
    assert out.returncode == 0, out.stderr[-3000:]
    res = json.loads(out.stdout.strip().splitlines()[-1])
    site, index, extent, count = res["selftest"]
    assert (site, index, extent) == (999, 3, 3) and count >= 1
    assert res["record"] == [0, 0, 0, 0], res["record"]
    assert res["worst_over_tol"] <= 1.0
